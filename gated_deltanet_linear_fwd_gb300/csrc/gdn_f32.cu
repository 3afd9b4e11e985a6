// fp32 path of the forward (all of q, k, v, o in fp32), for callers that need
// results within 1e-4 of the exact recurrence.  The tensor-core path rounds
// its operands to fp16 and cannot reach that, so this path runs the gated
// delta rule itself in fp32 on the CUDA cores:
//   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//   o_t = scale S_t q_t.
// Each row s of S (one d_v index) evolves on its own given k, g and beta:
//   s <- a s + c k,   a = exp(g_t),  c = beta_t (v_t[row] - a (s . k)),
// so a CTA of 256 threads holds a whole state: eight neighbouring threads of a
// warp hold four rows, each thread 16 columns of them (64 fp32 registers), so
// that every k and q value a thread reads from shared memory serves four rows;
// the group's partial dot products of its four rows are summed in four
// shuffles, each thread ending with one row's total.  The
// state is kept as S = sigma R with one scale for the whole state: the decay
// a multiplies sigma, so a token's update R <- R + (c / sigma) k is one FMA
// per element; sigma is folded back into R whenever it leaves [2^-60, 2^60].
//
// Context parallelism (FlashQLA pages, section "AutoCP": segments whose start
// states are combined exactly through the correction term M) supplies the
// parallelism the token loop lacks: over a segment the map s_start -> s_end
// is affine, s_end = s_start R + s_loc, so
//   transition  (role 0): rows of the identity run with no value input -> R
//   local       (role 1): rows from zero with the value input          -> S_loc
// run for every segment but each sequence's last at once, the fp32 combine
// kernel chains the segments' start states, and
//   output      (role 2): each segment from its start state (h0 for the
//                         first) writes o, and the last segment the final
//                         state.
// Without context parallelism only the output role runs, one CTA per
// (sequence, value head).
//
// Tokens are staged through shared memory in blocks of 16 (k, q, v rows by
// cp.async, the gates by plain loads), double buffered; a thread's columns
// 4 part + 32 m + e (m, e < 4) make each warp-wide k or q read one contiguous
// 128-byte line.
#include "gdn_dev.cuh"

namespace gdn {
namespace {

constexpr int kF32Threads = 256;
constexpr int kRowsT = 4, kColsT = 16;  // rows and columns of S per thread (8 threads per row group)
constexpr int kTokBlock = 16;
constexpr int kBufFloats = 3 * kTokBlock * kDim + 2 * kTokBlock;  // k, q, v rows, then exp(g), beta
constexpr int kF32Smem = 2 * kBufFloats * 4;


__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// OUT: the output role; else blockIdx.z = 0 runs the transition and 1 the
// local state.
template <bool OUT>
__global__ void __launch_bounds__(kF32Threads, 2) recurrence_f32_kernel(const Problem p) {
  extern __shared__ float4 f32_smem4[];
  float* smem = reinterpret_cast<float*>(f32_smem4);
  __shared__ SegInfo s_seg;
  __shared__ int s_skip;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int part = tid & 7, row0 = kRowsT * (tid >> 3);  // rows row0 .. row0 + 3, columns 4 part + 32 m + e
  const int j = blockIdx.y;
  const bool transition = !OUT && blockIdx.z == 0;  // rows of the identity, no value input
  const bool with_v = !transition;
  grid_dependency_wait();  // start states (output role): written by the combine before
  grid_launch_dependents();
  if (warp == 0) {
    SegInfo si;
    const bool ok = locate_segment(p, blockIdx.x, si);
    if (lane == 0) {
      if (!ok) si.n = -1;
      s_seg = si;
      s_skip = earlier_failure(p.status);
    }
  }
  __syncthreads();
  if (s_skip) return;
  const SegInfo si = s_seg;
  if (si.n < 0) {
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return;
  }
  if (!OUT) {
    if (si.s == si.n_seg - 1) return;                    // the last segment's map is not needed
    if (transition && si.s == 0 && p.h0 == nullptr) return;  // nor R_0 for a zero start
  }
  const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
  const int64_t t_begin = si.bos + (int64_t)si.cb * kChunk;
  const int64_t t_end = min(si.bos + (int64_t)si.ce * kChunk, si.eos);
  const size_t mat = (size_t)kDim * kDim;
  const size_t seg_off = ((size_t)(si.seg_base + si.s) * p.h_v + j) * mat;

  float s[kRowsT][kColsT];  // s[r][4 m + e] = R[row0 + r][4 part + 32 m + e], S = sigma R
  if (!OUT) {
#pragma unroll
    for (int r = 0; r < kRowsT; ++r)
#pragma unroll
      for (int i = 0; i < kColsT; ++i)
        s[r][i] = (transition && 4 * part + 32 * (i >> 2) + (i & 3) == row0 + r) ? 1.f : 0.f;
  } else if (si.s > 0) {  // the combined start state, rows = d_v
#pragma unroll
    for (int r = 0; r < kRowsT; ++r)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 v4 = *reinterpret_cast<const float4*>(p.Sstart + seg_off + (size_t)(row0 + r) * kDim + 4 * part +
                                                           32 * m);
        s[r][4 * m] = v4.x;
        s[r][4 * m + 1] = v4.y;
        s[r][4 * m + 2] = v4.z;
        s[r][4 * m + 3] = v4.w;
      }
  } else if (p.h0) {  // H = S^T: S[row][c] = h0[c][row], four rows in one float4
    const float* h0 = p.h0 + (size_t)(si.n * p.h_v + j) * mat;
#pragma unroll
    for (int i = 0; i < kColsT; ++i) {
      const float4 v4 = *reinterpret_cast<const float4*>(h0 + (size_t)(4 * part + 32 * (i >> 2) + (i & 3)) * kDim + row0);
      s[0][i] = v4.x;
      s[1][i] = v4.y;
      s[2][i] = v4.z;
      s[3][i] = v4.w;
    }
  } else {
#pragma unroll
    for (int r = 0; r < kRowsT; ++r)
#pragma unroll
      for (int i = 0; i < kColsT; ++i) s[r][i] = 0.f;
  }

  const float* q = reinterpret_cast<const float*>(p.q);
  const float* k = reinterpret_cast<const float*>(p.k);
  const float* v = reinterpret_cast<const float*>(p.v);
  float* o = reinterpret_cast<float*>(p.out);
  const int n_blocks = (int)((t_end - t_begin + kTokBlock - 1) / kTokBlock);
  const uint32_t sm0 = smem_u32(smem);
  // Block b's rows into buffer b & 1: 16 tokens x 512 bytes for each of k,
  // (q, v where used); thread tid copies 16-byte piece tid % 32 of token
  // 8 r + tid / 32, r = 0..1.  Tokens past the range are filled with zeros.
  auto stage = [&](int b) {
    const uint32_t buf = sm0 + (uint32_t)((b & 1) * kBufFloats) * 4u;
#pragma unroll
    for (int r = 0; r < kTokBlock / 8; ++r) {
      const int tt = 8 * r + warp, piece = lane * 4;
      const int64_t t = t_begin + (int64_t)b * kTokBlock + tt;
      const bool valid = t < t_end;
      const int64_t tc = valid ? t : t_begin;  // a valid address even for the zero fill
      const uint32_t off = (uint32_t)(tt * kDim + piece) * 4u;
      cp_async16(buf + off, k + ((size_t)tc * p.h_qk + iq) * kDim + piece, valid);
      if (OUT)
        cp_async16(buf + (uint32_t)(kTokBlock * kDim) * 4u + off, q + ((size_t)tc * p.h_qk + iq) * kDim + piece, valid);
      if (with_v)
        cp_async16(buf + (uint32_t)(2 * kTokBlock * kDim) * 4u + off, v + ((size_t)tc * p.h_v + j) * kDim + piece, valid);
    }
    cp_async_commit();
  };
  // The gates of block b (threads 0..15, one token each) into registers.
  auto gates = [&](int b, float& a, float& be) {
    const int64_t t = t_begin + (int64_t)b * kTokBlock + tid;
    a = 0.f;
    be = 0.f;
    if (tid < kTokBlock && t < t_end) {
      a = expf(p.g[(size_t)t * p.h_v + j]);
      be = p.beta[(size_t)t * p.h_v + j];
    }
  };
  auto put_gates = [&](int b, float a, float be) {
    if (tid < kTokBlock) {
      smem[(b & 1) * kBufFloats + 3 * kTokBlock * kDim + tid] = a;
      smem[(b & 1) * kBufFloats + 3 * kTokBlock * kDim + kTokBlock + tid] = be;
    }
  };
  // The four rows' partial dot products x[0..3] of the eight threads of a row
  // group, summed so that thread (part) ends with the total of row rsel =
  // 2 (part >> 2 & 1) + (part >> 1 & 1): each level sends the half it does
  // not keep (four shuffles in all instead of twelve).
  const int b2 = (part >> 2) & 1, b1 = (part >> 1) & 1, rsel = 2 * b2 + b1;
  const int group_lane = lane & ~7;
  auto rows_sum = [&](const float (&x)[kRowsT]) {
    const float y0 = (b2 ? x[2] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[2], 4);
    const float y1 = (b2 ? x[3] : x[1]) + __shfl_xor_sync(0xffffffffu, b2 ? x[1] : x[3], 4);
    float z = (b1 ? y1 : y0) + __shfl_xor_sync(0xffffffffu, b1 ? y0 : y1, 2);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
    return z;
  };
  float sigma = 1.f;  // S = sigma R
  if (n_blocks > 0) {
    float a0, b0;
    stage(0);
    gates(0, a0, b0);
    put_gates(0, a0, b0);
  }
  for (int b = 0; b < n_blocks; ++b) {
    float a1 = 0.f, b1 = 0.f;
    if (b + 1 < n_blocks) {  // buffer (b + 1) & 1 was last read in block b - 1
      stage(b + 1);
      gates(b + 1, a1, b1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // block b's rows and gates are in buffer b & 1
    const float* buf = smem + (b & 1) * kBufFloats;
    const int nt = (int)min((int64_t)kTokBlock, t_end - t_begin - (int64_t)b * kTokBlock);
    for (int tt = 0; tt < nt; ++tt) {
      const float a = buf[3 * kTokBlock * kDim + tt], be = buf[3 * kTokBlock * kDim + kTokBlock + tt];
      float kc[kColsT];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 k4 = *reinterpret_cast<const float4*>(buf + tt * kDim + 4 * part + 32 * m);
        kc[4 * m] = k4.x;
        kc[4 * m + 1] = k4.y;
        kc[4 * m + 2] = k4.z;
        kc[4 * m + 3] = k4.w;
      }
      const float vsel = with_v ? buf[2 * kTokBlock * kDim + tt * kDim + row0 + rsel] : 0.f;
      float x[kRowsT];
#pragma unroll
      for (int r = 0; r < kRowsT; ++r) {  // this thread's part of R . k
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int i = 0; i < kColsT; i += 2) {
          x0 = fmaf(s[r][i], kc[i], x0);
          x1 = fmaf(s[r][i + 1], kc[i + 1], x1);
        }
        x[r] = x0 + x1;
      }
      // c = beta (v - a s . k) with s . k = sigma (R . k): for row rsel, then every row's
      const float csel = be * (vsel - a * (sigma * rows_sum(x)));
      float c[kRowsT];
#pragma unroll
      for (int r = 0; r < kRowsT; ++r) c[r] = __shfl_sync(0xffffffffu, csel, group_lane | (4 * (r >> 1) + 2 * (r & 1)));
      // S <- a S + c k: sigma <- a sigma, R <- R + (c / sigma) k
      sigma *= a;
      if (!(sigma >= 0x1p-60f && sigma <= 0x1p60f)) {  // (the same in every thread)
#pragma unroll
        for (int r = 0; r < kRowsT; ++r)
#pragma unroll
          for (int i = 0; i < kColsT; ++i) s[r][i] *= sigma;
        sigma = 1.f;
      }
      const float inv = 1.f / sigma;
#pragma unroll
      for (int r = 0; r < kRowsT; ++r) {
        const float cr = c[r] * inv;
#pragma unroll
        for (int i = 0; i < kColsT; ++i) s[r][i] = fmaf(cr, kc[i], s[r][i]);
      }
      if (OUT) {
        float qc[kColsT];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 q4 = *reinterpret_cast<const float4*>(buf + kTokBlock * kDim + tt * kDim + 4 * part + 32 * m);
          qc[4 * m] = q4.x;
          qc[4 * m + 1] = q4.y;
          qc[4 * m + 2] = q4.z;
          qc[4 * m + 3] = q4.w;
        }
        float xq[kRowsT];
#pragma unroll
        for (int r = 0; r < kRowsT; ++r) {
          float x0 = 0.f, x1 = 0.f;
#pragma unroll
          for (int i = 0; i < kColsT; i += 2) {
            x0 = fmaf(s[r][i], qc[i], x0);
            x1 = fmaf(s[r][i + 1], qc[i + 1], x1);
          }
          xq[r] = x0 + x1;
        }
        const float osel = p.scale * (sigma * rows_sum(xq));
        const int64_t t = t_begin + (int64_t)b * kTokBlock + tt;
        if ((part & 1) == 0) o[((size_t)t * p.h_v + j) * kDim + row0 + rsel] = osel;
      }
    }
    put_gates(b + 1, a1, b1);  // buffer (b + 1) & 1's gates: read from the next block on
    __syncthreads();           // buffer b & 1 is read before block b + 2 is staged into it
  }
#pragma unroll
  for (int r = 0; r < kRowsT; ++r)
#pragma unroll
    for (int i = 0; i < kColsT; ++i) s[r][i] *= sigma;
  if (OUT) {
    if (p.hT && si.s == si.n_seg - 1) {  // H = S^T: four rows of S are one float4 of a row of H
      float* hT = p.hT + (size_t)(si.n * p.h_v + j) * mat;
#pragma unroll
      for (int i = 0; i < kColsT; ++i)
        *reinterpret_cast<float4*>(hT + (size_t)(4 * part + 32 * (i >> 2) + (i & 3)) * kDim + row0) =
            make_float4(s[0][i], s[1][i], s[2][i], s[3][i]);
    }
  } else {
    float* dst = (transition ? p.R : p.Sloc) + seg_off;
#pragma unroll
    for (int r = 0; r < kRowsT; ++r)
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<float4*>(dst + (size_t)(row0 + r) * kDim + 4 * part + 32 * m) =
            make_float4(s[r][4 * m], s[r][4 * m + 1], s[r][4 * m + 2], s[r][4 * m + 3]);
  }
}

}  // namespace

cudaError_t f32_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(recurrence_f32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kF32Smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(recurrence_f32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF32Smem);
}

// The segments' transitions and local states (context-parallel plans only).
cudaError_t launch_f32_prep(const Problem& p, cudaStream_t st) {
  return launch_kernel(recurrence_f32_kernel<false>, dim3(p.n_seg_total, p.h_v, 2), dim3(kF32Threads), kF32Smem, st,
                       true, p);
}

// The output pass: every segment from its start state.
cudaError_t launch_recurrence_f32(const Problem& p, cudaStream_t st, bool dependent) {
  return launch_kernel(recurrence_f32_kernel<true>, dim3(p.n_seg_total, p.h_v), dim3(kF32Threads), kF32Smem, st,
                       dependent, p);
}

}  // namespace gdn
