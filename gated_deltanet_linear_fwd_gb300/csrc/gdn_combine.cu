// Exact combine of context-parallel segment start states (FlashQLA pages,
// section "AutoCP": each segment's local state and transition are computed
// in preprocessing, then the segment start states are combined exactly).
//
// In the S orientation (rows = d_v) a segment maps its start state to
//     S_end = S_start R + S_loc,     R = M^T (d_k x d_k),
// so the start states follow by a serial scan over the segments of a
// sequence:  S_start(0) = h0^T,  S_start(s+1) = S_start(s) R_s + S_loc,s.
// Rows of S are independent, so each CTA owns 8 rows of one (sequence, head)
// and streams R_s through shared memory (double-buffered cp.async) while it
// does the fp32 vector-matrix products.  The CTA of row block 0 also
// records the mode the (sequence, head) takes and its warmup bound.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRows = 8;  // state rows per CTA
constexpr int kCombineSmem = 2 * kDim * kDim * 4 + kRows * kDim * 4;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(256) combine_kernel(const Problem p) {
  extern __shared__ float4 csm4[];
  float* sR = reinterpret_cast<float*>(csm4);  // [2][128*128]
  float* sX = sR + 2 * kDim * kDim;            // [kRows][128]
  __shared__ SegInfo s_seq;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n = blockIdx.x, j = blockIdx.y, r0 = blockIdx.z * kRows;
  if (warp == 0) {
    SegInfo si;
    locate_sequence(p, n, si);
    if ((tid & 31) == 0) s_seq = si;
  }
  __syncthreads();
  const SegInfo si = s_seq;
  const int mode = head_mode_of(p, si, j);
  if (blockIdx.z == 0 && tid == 0) {
    p.head_mode[n * p.h_v + j] = mode;
    p.head_bound[n * p.h_v + j] =
        p.plan_mode == kModeWarmup ? head_log_bound(p, si, j) : -__int_as_float(0x7f800000);
  }
  if (mode != kModeExact || si.n_seg <= 1) return;

  const int rr = tid >> 5;         // row within the block
  const int c4 = (tid & 31) * 4;   // 4 output columns
  const size_t mat = (size_t)kDim * kDim;
  // S_start(0) rows: S[dv][dk] = h0[dk][dv]
  for (int i = tid; i < kRows * kDim; i += 256) {
    const int r = i / kDim, c = i % kDim;
    sX[i] = p.h0 ? p.h0[(size_t)(n * p.h_v + j) * mat + (size_t)c * kDim + (r0 + r)] : 0.f;
  }
  auto prefetch = [&](int s, int buf) {
    const float* src = p.R + ((size_t)(si.seg_base + s) * p.h_v + j) * mat;
    float* dst = sR + buf * mat;
    for (int i = tid; i < kDim * kDim / 4; i += 256) cp_async16(dst + 4 * i, src + 4 * i);
    cp_async_commit();
  };
  // R_0 is not produced when the start state is zero (no h0): skip its product.
  const bool skip_first = p.h0 == nullptr;
  const int last = si.n_seg - 2;  // produce S_start(1 .. n_seg-1)
  int first_product = skip_first ? 1 : 0;
  if (first_product <= last) prefetch(first_product, first_product & 1);
  __syncthreads();
  for (int s = 0; s <= last; ++s) {
    const bool product = s >= first_product;
    if (product && s + 1 <= last) {
      prefetch(s + 1, (s + 1) & 1);
      cp_async_wait<1>();
    } else if (product) {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float4 l4 = *reinterpret_cast<const float4*>(
        p.Sloc + ((size_t)(si.seg_base + s) * p.h_v + j) * mat + (size_t)(r0 + rr) * kDim + c4);
    float a0 = l4.x, a1 = l4.y, a2 = l4.z, a3 = l4.w;
    if (product) {
      const float* Rb = sR + (s & 1) * mat;
      const float* xr = sX + rr * kDim;
#pragma unroll 8
      for (int k = 0; k < kDim; ++k) {
        const float x = xr[k];
        const float4 r4 = *reinterpret_cast<const float4*>(Rb + k * kDim + c4);
        a0 = fmaf(x, r4.x, a0);
        a1 = fmaf(x, r4.y, a1);
        a2 = fmaf(x, r4.z, a2);
        a3 = fmaf(x, r4.w, a3);
      }
    }
    __syncthreads();
    *reinterpret_cast<float4*>(sX + rr * kDim + c4) = make_float4(a0, a1, a2, a3);
    *reinterpret_cast<float4*>(p.Sstart + ((size_t)(si.seg_base + s + 1) * p.h_v + j) * mat +
                               (size_t)(r0 + rr) * kDim + c4) = make_float4(a0, a1, a2, a3);
  }
}

}  // namespace

cudaError_t combine_kernel_setup() {
  return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCombineSmem);
}

cudaError_t launch_combine(const Problem& p, cudaStream_t st) {
  dim3 grid(p.n_seqs, p.h_v, kDim / kRows);
  combine_kernel<<<grid, 256, kCombineSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
