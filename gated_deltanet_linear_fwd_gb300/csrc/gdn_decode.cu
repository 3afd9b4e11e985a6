// One-token step of the gated delta rule for a batch of sequences (the
// generation-time counterpart of the chunked prefill): per sequence n and
// value head j, with H = S^T the stored state,
//   S <- exp(g) S (I - beta k k^T) + beta v k^T,   o = scale S q
// (Yang, Kautz, Hatamizadeh, "Gated Delta Networks", section "Gated delta
// rule").  The state is read and written once (64 KB each way per (n, j)), so
// the step is bound by HBM bandwidth; it runs on the CUDA cores in fp32.
//
// Two CTAs of 256 threads per (n, j), one per half of d_v (the rows of S are
// independent, so the halves share nothing but k and q): thread (g, part)
// holds columns 64 z + 4g .. 64 z + 4g + 3 of H (rows of S) for d_k = 8 part
// .. 8 part + 7, so half a warp reads and writes the CTA's 256 bytes of one
// row of H per 16-byte instruction.  S k and S q are summed over the sixteen
// parts through shared memory.  Halving the CTAs' size lets the last wave of
// a batch fill the SMs.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;

template <typename T>
__device__ __forceinline__ float load_elem(const T* p);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p) {
  return *p;
}
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void store_elem(T* p, float x);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, float x) {
  *p = x;
}
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(kDecThreads, 4) decode_kernel(const DecodeArgs a) {
  constexpr int kParts = 16, kRowsPerPart = kDim / kParts;  // 8 rows of H (d_k) per part
  __shared__ float sk[kDim], sq[kDim];
  __shared__ float4 red[kParts][16];
  const int n = blockIdx.x, j = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, g = tid & 15, part = tid >> 4;
  const int iq = (int)(((int64_t)j * a.h_qk) / a.h_v);
  if (tid < kDim) {
    sk[tid] = load_elem(reinterpret_cast<const T*>(a.k) + ((size_t)n * a.h_qk + iq) * kDim + tid);
    sq[tid] = load_elem(reinterpret_cast<const T*>(a.q) + ((size_t)n * a.h_qk + iq) * kDim + tid);
  }
  float4* H = reinterpret_cast<float4*>(a.state + ((size_t)n * a.h_v + j) * kDim * kDim +
                                        (size_t)(part * kRowsPerPart) * kDim + 64 * z) +
              g;
  float4 h[kRowsPerPart];
#pragma unroll
  for (int e = 0; e < kRowsPerPart; ++e) h[e] = H[(size_t)e * (kDim / 4)];
  __syncthreads();
  // (S_{t-1} k) for this thread's 4 rows of S over its 8 columns, then over all parts
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int e = 0; e < kRowsPerPart; ++e) {
    const float kc = sk[part * kRowsPerPart + e];
    acc.x = fmaf(h[e].x, kc, acc.x);
    acc.y = fmaf(h[e].y, kc, acc.y);
    acc.z = fmaf(h[e].z, kc, acc.z);
    acc.w = fmaf(h[e].w, kc, acc.w);
  }
  red[part][g] = acc;
  __syncthreads();
  float4 s_k = red[0][g];
#pragma unroll
  for (int q = 1; q < kParts; ++q) {
    const float4 t = red[q][g];
    s_k.x += t.x;
    s_k.y += t.y;
    s_k.z += t.z;
    s_k.w += t.w;
  }
  const float alpha = expf(a.g[(size_t)n * a.h_v + j]), beta = a.beta[(size_t)n * a.h_v + j];
  const T* vrow = reinterpret_cast<const T*>(a.v) + ((size_t)n * a.h_v + j) * kDim + 64 * z + 4 * g;
  const float4 bsk = make_float4(beta * s_k.x, beta * s_k.y, beta * s_k.z, beta * s_k.w);
  const float4 bv = make_float4(beta * load_elem(vrow), beta * load_elem(vrow + 1), beta * load_elem(vrow + 2),
                                beta * load_elem(vrow + 3));
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int e = 0; e < kRowsPerPart; ++e) {
    const float kc = sk[part * kRowsPerPart + e], qc = sq[part * kRowsPerPart + e];
    float4 hn;
    hn.x = fmaf(alpha, fmaf(-bsk.x, kc, h[e].x), bv.x * kc);
    hn.y = fmaf(alpha, fmaf(-bsk.y, kc, h[e].y), bv.y * kc);
    hn.z = fmaf(alpha, fmaf(-bsk.z, kc, h[e].z), bv.z * kc);
    hn.w = fmaf(alpha, fmaf(-bsk.w, kc, h[e].w), bv.w * kc);
    H[(size_t)e * (kDim / 4)] = hn;
    o.x = fmaf(hn.x, qc, o.x);
    o.y = fmaf(hn.y, qc, o.y);
    o.z = fmaf(hn.z, qc, o.z);
    o.w = fmaf(hn.w, qc, o.w);
  }
  __syncthreads();  // everyone has read red
  red[part][g] = o;
  __syncthreads();
  if (part == 0) {
    float4 t = red[0][g];
#pragma unroll
    for (int q = 1; q < kParts; ++q) {
      const float4 u = red[q][g];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    T* orow = reinterpret_cast<T*>(a.out) + ((size_t)n * a.h_v + j) * kDim + 64 * z + 4 * g;
    store_elem(orow, a.scale * t.x);
    store_elem(orow + 1, a.scale * t.y);
    store_elem(orow + 2, a.scale * t.z);
    store_elem(orow + 3, a.scale * t.w);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, bool f32, cudaStream_t st) {
  dim3 grid(a.n_seqs, a.h_v, 2);
  if (f32)
    decode_kernel<float><<<grid, kDecThreads, 0, st>>>(a);
  else
    decode_kernel<__nv_bfloat16><<<grid, kDecThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
