// K1: chunk-local gate kernel.  For every (segment, value head) it bounds the
// error a warmup restart would make (FlashQLA pages, section "AutoCP": heads
// whose gates decay fast let a segment restart from a few preceding chunks
// and skip the correction term M; the Telegram post on FlashQLA: on 60-80 %
// of heads old tokens fade quickly, so a 6-8 chunk warmup is almost exact).
//
// A restart from zero w chunks before the segment start (tokens t in the
// window W) leaves the start state off by the exact state at the window
// start, propagated through the window.  Each token map X -> alpha X (I -
// beta k k^T) has spectral norm <= alpha * max(1, |1 - beta ||k||^2|), so
// the relative error is at most
//     exp( sum_{t in W} [ g_t + log max(1, |1 - beta_t ||k_t||^2|) ] ).
// The kernel picks, per segment, the smallest depth w (at most the planned
// maximum) whose exponent is <= log(tol), and writes w and that exponent; a
// depth that reaches the sequence start runs exactly from the initial state
// (exponent -inf).  No acceptable depth: w = -1, and the (sequence, head)
// runs in exact mode.  Segment 0 needs no restart (w = 0).
#include <cuda_bf16.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

template <typename KT>
__device__ __forceinline__ float row_sq_norm(const KT* krow);

template <>
__device__ __forceinline__ float row_sq_norm<__nv_bfloat16>(const __nv_bfloat16* krow) {
  float acc = 0.f;
  const uint4* p4 = reinterpret_cast<const uint4*>(krow);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint4 u = p4[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
      acc = fmaf(lo, lo, acc);
      acc = fmaf(hi, hi, acc);
    }
  }
  return acc;
}

template <>
__device__ __forceinline__ float row_sq_norm<float>(const float* krow) {
  float acc = 0.f;
  const float4* p4 = reinterpret_cast<const float4*>(krow);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float4 u = p4[i];
    acc = fmaf(u.x, u.x, fmaf(u.y, u.y, fmaf(u.z, u.z, fmaf(u.w, u.w, acc))));
  }
  return acc;
}

template <typename KT>
__global__ void __launch_bounds__(256) gate_bound_kernel(const Problem p) {
  constexpr int kMaxWin = 64;
  __shared__ SegInfo s_seg;
  __shared__ float s_chunk[kMaxWin];  // exponent contribution of window chunk cb-1-w
  __shared__ int s_ok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.y;
  if (warp == 0) {
    SegInfo si;
    const bool ok = locate_segment(p, blockIdx.x, si);
    if (lane == 0) {
      s_seg = si;
      s_ok = ok;
    }
  }
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return;
  }
  const SegInfo si = s_seg;
  const float neg_inf = -__int_as_float(0x7f800000);
  const size_t slot = (size_t)blockIdx.x * p.h_v + j;
  if (si.s == 0) {
    if (tid == 0) {
      p.seg_bound[slot] = neg_inf;
      p.seg_w[slot] = 0;
    }
    return;
  }
  const int wmax = min(p.warmup_chunks, kMaxWin);
  const int nwin = min(wmax, si.cb);
  const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
  const KT* kbase = reinterpret_cast<const KT*>(p.k);
  for (int w = warp; w < nwin; w += 8) {  // one warp per window chunk, two tokens per lane
    const int64_t t0 = si.bos + (int64_t)(si.cb - 1 - w) * kChunk;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t t = t0 + 2 * lane + e;
      const float gsum = p.g[(size_t)t * p.h_v + j];
      const float b = p.beta[(size_t)t * p.h_v + j];
      const float kk = row_sq_norm<KT>(kbase + ((size_t)t * p.h_qk + iq) * kDim);
      acc += gsum + __logf(fmaxf(1.f, fabsf(1.f - b * kk)));
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
    if (lane == 0) s_chunk[w] = acc;
  }
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f;
    int wsel = -1;
    float bsel = 0.f;
    for (int w = 1; w <= nwin; ++w) {
      acc += s_chunk[w - 1];
      if (si.cb - w == 0) {  // reaches the sequence start: exact from the initial state
        wsel = w;
        bsel = neg_inf;
        break;
      }
      if (acc <= p.log_tol) {
        wsel = w;
        bsel = acc;
        break;
      }
    }
    if (wsel < 0) bsel = acc;
    p.seg_w[slot] = wsel;
    p.seg_bound[slot] = bsel;
  }
}

}  // namespace

cudaError_t launch_gate_bound(const Problem& p, cudaStream_t st) {
  dim3 grid(p.n_seg_total, p.h_v);
  if (p.elem_f32)
    gate_bound_kernel<float><<<grid, 256, 0, st>>>(p);
  else
    gate_bound_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
