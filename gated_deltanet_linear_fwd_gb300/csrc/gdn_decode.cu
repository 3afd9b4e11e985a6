// One-token step of the gated delta rule for a batch of sequences (the
// generation-time counterpart of the chunked prefill): per sequence n and
// value head j, with H = S^T the stored state,
//   S <- exp(g) S (I - beta k k^T) + beta v k^T,   o = scale S q
// (Yang, Kautz, Hatamizadeh, "Gated Delta Networks", section "Gated delta
// rule").  The state is read and written once (64 KB each way per (n, j)), so
// the step is bound by HBM bandwidth; it runs on the CUDA cores in fp32.
//
// One CTA of 512 threads per (n, j): thread (i, part) holds column i of H
// (row i of S) for d_k = 32 part .. 32 part + 31, so a warp reads and writes
// 128 contiguous bytes of H per instruction.  S k and S q are summed over
// the four parts through shared memory.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecThreads = 512;

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
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeArgs a) {
  __shared__ float sk[kDim], sq[kDim];
  __shared__ float part_sum[4][kDim];
  const int n = blockIdx.x, j = blockIdx.y;
  const int tid = threadIdx.x, i = tid & (kDim - 1), part = tid >> 7;
  const int iq = (int)(((int64_t)j * a.h_qk) / a.h_v);
  const T* q = reinterpret_cast<const T*>(a.q) + ((size_t)n * a.h_qk + iq) * kDim;
  const T* k = reinterpret_cast<const T*>(a.k) + ((size_t)n * a.h_qk + iq) * kDim;
  if (part == 0) {
    sk[i] = load_elem(k + i);
    sq[i] = load_elem(q + i);
  }
  float* H = a.state + ((size_t)n * a.h_v + j) * kDim * kDim + (size_t)(part * 32) * kDim + i;
  float h[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) h[e] = H[(size_t)e * kDim];
  __syncthreads();
  // (S_{t-1} k)_i over this part's 32 columns
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e & 3] = fmaf(h[e], sk[part * 32 + e], acc[e & 3]);
  part_sum[part][i] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  __syncthreads();
  const float s_k = (part_sum[0][i] + part_sum[1][i]) + (part_sum[2][i] + part_sum[3][i]);
  const float alpha = expf(a.g[(size_t)n * a.h_v + j]), beta = a.beta[(size_t)n * a.h_v + j];
  const float vi = load_elem(reinterpret_cast<const T*>(a.v) + ((size_t)n * a.h_v + j) * kDim + i);
  const float bsk = beta * s_k, bv = beta * vi;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float kc = sk[part * 32 + e];
    const float hn = fmaf(alpha, fmaf(-bsk, kc, h[e]), bv * kc);
    H[(size_t)e * kDim] = hn;
    o[e & 3] = fmaf(hn, sq[part * 32 + e], o[e & 3]);
  }
  __syncthreads();  // everyone has read part_sum
  part_sum[part][i] = (o[0] + o[1]) + (o[2] + o[3]);
  __syncthreads();
  if (part == 0) {
    const float oi = (part_sum[0][i] + part_sum[1][i]) + (part_sum[2][i] + part_sum[3][i]);
    store_elem(reinterpret_cast<T*>(a.out) + ((size_t)n * a.h_v + j) * kDim + i, a.scale * oi);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, bool f32, cudaStream_t st) {
  dim3 grid(a.n_seqs, a.h_v);
  if (f32)
    decode_kernel<float><<<grid, kDecThreads, 0, st>>>(a);
  else
    decode_kernel<__nv_bfloat16><<<grid, kDecThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
