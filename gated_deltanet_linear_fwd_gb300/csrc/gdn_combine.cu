// Exact combine of context-parallel segment start states (FlashQLA pages,
// section "AutoCP": each segment's local state and transition are computed
// in preprocessing, then the segment start states are combined exactly).
//
// In the S orientation (rows = d_v) a segment maps its start state to
//     S_end = S_start R + S_loc,     R = M^T (d_k x d_k),
// so the start states follow by a serial scan over the segments of a
// sequence:  S_start(0) = h0^T,  S_start(s+1) = S_start(s) R_s + S_loc,s.
// Rows of S are independent, so each CTA owns 4 or 8 rows of one (sequence,
// head) and streams R_s and its rows of S_loc,s through shared memory (bulk
// copies, one segment ahead) while it does the fp32 products.  Each warp takes a
// 16-row slice of R for all the CTA's rows (so R is read from shared memory once
// per segment), and the 8 partial sums are added in a second pass.  Four rows
// per CTA halve each segment's step when few (sequence, head) pairs exist.
// The CTA of row block 0 also records the mode the (sequence, head) takes and
// its warmup bound.
//
// BWD: the same scan run backwards for the gradient of the state.  With
// D_end(s) the gradient of segment s's end state (rows d_v after transposing)
// and R_s, S_loc,s the transposed transition and local offset of the
// backward chain over segment s,
//     D_end(n_seg-1) = dh_T^T,   D_end(s-1) = D_end(s) R_s + S_loc,s,
// taking h0's place by dh_T and writing D_end(s-1) where the forward writes
// S_start(s+1).
#include "gdn_dev.cuh"

namespace gdn {
namespace {

constexpr int kSlices = 8;  // k slices of 16 (one per warp)
template <int kRows>
constexpr int combine_smem() {
  return 2 * kDim * kDim * 4 + 2 * kRows * kDim * 4 + kRows * kDim * 4 + kSlices * kRows * kDim * 4;
}

// kRows state rows per CTA (4 or 8)
template <int kRows, bool BWD>
__global__ void __launch_bounds__(256) combine_kernel(const Problem p) {
  extern __shared__ float4 csm4[];
  float* sR = reinterpret_cast<float*>(csm4);  // [2][128*128]
  float* sL = sR + 2 * kDim * kDim;            // [2][kRows][128]: this block's rows of S_loc
  float* sX = sL + 2 * kRows * kDim;           // [kRows][128]
  float* sP = sX + kRows * kDim;               // [kSlices][kRows][128] partial sums
  __shared__ SegInfo s_seq;
  __shared__ uint64_t s_bar[2];
  const int tid = threadIdx.x, warp = tid >> 5;
  // x = row block + (kDim / kRows) * sequence: a (sequence, head)'s row blocks
  // are neighbouring blocks, so they come in the same wave
  constexpr int kBlocks = kDim / kRows;
  const int n = (int)(blockIdx.x / kBlocks), j = blockIdx.y, rb = (int)(blockIdx.x % kBlocks), r0 = rb * kRows;
  __shared__ int s_mode, s_skip;
  // the sequence's segments come from the plan's arithmetic and the sequence
  // bounds (an input): located while the kernel before this one finishes
  SegInfo si;
  if (warp == 0) locate_sequence(p, n, si);
  grid_dependency_wait();  // the segment transitions and local states: written by the kernel before
  grid_launch_dependents();
  if (warp == 0) {  // the status word is fetched beside the segments' depths
    const int st = (tid == 0) ? earlier_failure(p.status) : 0;
    float bound;
    const int mode = head_mode_warp(p, si, j, &bound);
    if (tid == 0) {
      s_skip = st;
      s_seq = si;
      s_mode = mode;
      if (!BWD && rb == 0 && !st) {
        p.head_mode[n * p.h_v + j] = mode;
        p.head_bound[n * p.h_v + j] = bound;
      }
    }
  }
  __syncthreads();
  if (s_skip) return;  // an earlier kernel failed: its results are incomplete
  si = s_seq;
  const int mode = s_mode;
  if (mode != kModeExact || si.n_seg <= 1) return;

  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
  }
  const int rr = tid >> 5;         // row within the block
  const int c4 = (tid & 31) * 4;   // 4 output columns
  const size_t mat = (size_t)kDim * kDim;
  // S_start(0) rows: S[dv][dk] = h0[dk][dv]
  for (int i = tid; i < kRows * kDim; i += 256) {
    const int r = i / kDim, c = i % kDim;
    sX[i] = p.h0 ? p.h0[(size_t)(n * p.h_v + j) * mat + (size_t)c * kDim + (r0 + r)] : 0.f;
  }
  // segment s's inputs into buffer s & 1: R_s (when its product is taken) and S_loc,s rows
  const bool skip_first = p.h0 == nullptr;  // R_0 is not produced for a zero start: skip its product
  const int first_product = skip_first ? 1 : 0;
  const int last = si.n_seg - 2;  // produce S_start(1 .. n_seg-1)
  // step i reads segment seg_of(i) and writes the state of out_of(i)
  auto seg_of = [&](int i) { return BWD ? si.n_seg - 1 - i : i; };
  auto prefetch = [&](int i) {     // one thread; buffer i & 1 was last read in step i - 2
    const int buf = i & 1;
    const bool product = i >= first_product;
    const int s = seg_of(i);
    mbar_arrive_expect_tx(&s_bar[buf], (uint32_t)(kRows * kDim * 4) + (product ? (uint32_t)(mat * 4) : 0u));
    if (product)
      bulk_load(sR + buf * mat, p.R + ((size_t)(si.seg_base + s) * p.h_v + j) * mat, (uint32_t)(mat * 4), &s_bar[buf]);
    bulk_load(sL + buf * kRows * kDim, p.Sloc + ((size_t)(si.seg_base + s) * p.h_v + j) * mat + (size_t)r0 * kDim,
              (uint32_t)(kRows * kDim * 4), &s_bar[buf]);
  };
  __syncthreads();  // barriers initialised, S_start(0) rows in place
  if (tid == 0) prefetch(0);
  for (int s = 0; s <= last; ++s) {
    const bool product = s >= first_product;
    if (tid == 0 && s + 1 <= last) prefetch(s + 1);
    const bool ok = mbar_wait(&s_bar[s & 1], (uint32_t)((s >> 1) & 1), kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) report(p.status, kDevTimeout, kDetTmaWait);
      // let copies already in flight land before the memory is released
      const uint64_t t_start = globaltimer_ns();
      while (globaltimer_ns() - t_start < 2000000ull) {
      }
      return;
    }
    const bool own = rr < kRows;  // the threads that finish one output row each
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (own) {
      const float4 l4 = *reinterpret_cast<const float4*>(sL + (s & 1) * kRows * kDim + rr * kDim + c4);
      a0 = l4.x;
      a1 = l4.y;
      a2 = l4.z;
      a3 = l4.w;
    }
    if (product) {
      // partial products over k = 16 ks .. 16 ks + 15 for all rows, columns c4 .. c4 + 3
      const int ks = tid >> 5;
      const float* Rb = sR + (s & 1) * mat + (size_t)(16 * ks) * kDim + c4;
      float acc[kRows][4];
#pragma unroll
      for (int r = 0; r < kRows; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 16; k4 += 4) {
        float4 x4[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) x4[r] = *reinterpret_cast<const float4*>(sX + r * kDim + 16 * ks + k4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 r4 = *reinterpret_cast<const float4*>(Rb + (k4 + e) * kDim);
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const float x = (&x4[r].x)[e];
            acc[r][0] = fmaf(x, r4.x, acc[r][0]);
            acc[r][1] = fmaf(x, r4.y, acc[r][1]);
            acc[r][2] = fmaf(x, r4.z, acc[r][2]);
            acc[r][3] = fmaf(x, r4.w, acc[r][3]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r)
        *reinterpret_cast<float4*>(sP + (ks * kRows + r) * kDim + c4) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      __syncthreads();  // partial sums written; R, S_loc and sX read for this step
      if (own) {
#pragma unroll
        for (int q = 0; q < kSlices; ++q) {
          const float4 t4 = *reinterpret_cast<const float4*>(sP + (q * kRows + rr) * kDim + c4);
          a0 += t4.x;
          a1 += t4.y;
          a2 += t4.z;
          a3 += t4.w;
        }
      }
    } else {
      __syncthreads();  // S_loc read before its buffer is refilled
    }
    // The new rows go to sX once every thread has read it (the barrier above);
    // the next step reads them, and overwrites sP, only after its own barrier.
    if (own) {
      *reinterpret_cast<float4*>(sX + rr * kDim + c4) = make_float4(a0, a1, a2, a3);
      const int out_seg = BWD ? seg_of(s) - 1 : s + 1;
      *reinterpret_cast<float4*>(p.Sstart + ((size_t)(si.seg_base + out_seg) * p.h_v + j) * mat +
                                 (size_t)(r0 + rr) * kDim + c4) = make_float4(a0, a1, a2, a3);
    }
  }
}

}  // namespace

cudaError_t combine_kernel_setup() {
  cudaError_t e =
      cudaFuncSetAttribute(combine_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, combine_smem<4>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_kernel<8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, combine_smem<8>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_kernel<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, combine_smem<4>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_kernel<8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, combine_smem<8>());
  return e;
}

template <bool BWD>
static cudaError_t launch_combine_dir(const Problem& p, int sm_count, cudaStream_t st) {
  // 32 CTAs of 4 rows per exact (sequence, head) if they fit in about two waves when
  // all pairs are launched (the forward: only the exact heads' blocks stay), in one
  // wave for the backward (every head is exact there)
  if ((int64_t)p.n_seqs * p.h_v * 32 <= (BWD ? 1 : 2) * (int64_t)sm_count)
    return launch_kernel(combine_kernel<4, BWD>, dim3(p.n_seqs * (kDim / 4), p.h_v), dim3(256), combine_smem<4>(), st,
                         true, p);
  return launch_kernel(combine_kernel<8, BWD>, dim3(p.n_seqs * (kDim / 8), p.h_v), dim3(256), combine_smem<8>(), st,
                       true, p);
}

cudaError_t launch_combine(const Problem& p, int sm_count, cudaStream_t st) {
  return launch_combine_dir<false>(p, sm_count, st);
}

// The backward's combine: p.h0 = dh_T, p.R / p.Sloc = the backward chain's
// transposed transitions and local offsets, p.Sstart receives D_end.
cudaError_t launch_combine_bwd(const Problem& p, int sm_count, cudaStream_t st) {
  return launch_combine_dir<true>(p, sm_count, st);
}

}  // namespace gdn
