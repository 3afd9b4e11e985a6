// Internal definitions shared by the kernels and the host entry points.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gdn_plan_rule.cuh"

namespace gdn {

// Status word codes (first int of the workspace), mirrored in gdn_status.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 5;
constexpr int kDevCheck = 7;

// Detail words: which wait or check tripped.
constexpr int kDetTmaWait = 1;
constexpr int kDetMmaWait = 2;
constexpr int kDetSegMismatch = 3;
constexpr int kDetCombineOrder = 4;
constexpr int kDetFp16Range = 5;  // a value outside the fp16 MMA operand range
constexpr int kDetStallTest = 6;  // the test hook's wait ran out (Problem::stall_ns)

// Head mode words (workspace head-mode section).
constexpr int kModeOff = 0;
constexpr int kModeExact = 1;
constexpr int kModeWarmup = 2;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per bounded wait

// Chunk-local records written by the WY kernel and read by the scans: operand
// tiles already in the 128-byte-swizzled shared-memory image the tcgen05 MMAs
// read, so one bulk copy per tile brings them on chip.
//   per (chunk, value head):
constexpr uint32_t kRecWn = 0;        // fp16 -W, MN-major B tile: row d_k, 64 chunk rows (16 KB)
constexpr uint32_t kRecU = 16384;     // fp16 U^T, K-major A tile: row d_v, 64 chunk rows (16 KB)
constexpr uint32_t kRecP = 32768;     // fp16 P, K-major B tile: row r, columns s <= r (8 KB)
constexpr uint32_t kRecGam = 40960;   // fp32 exp(G_r), then exp(G_63 - G_r) (2 x 64)
constexpr uint32_t kRecBytes = 41472;

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;          // [n_seqs, h_v, d_k, d_v] or null
  const int32_t* cu;        // device cu_seqlens or null
  void* out;
  float* hT;                // [n_seqs, h_v, d_k, d_v] or null
  int T_row;                // tokens per batch row (with cu: all tokens, one row)
  int n_seqs, h_qk, h_v;
  float scale;
  int elem_f32;             // q/k/v/out are fp32 (else bf16)
  // plan
  int plan_mode;            // kModeOff / kModeExact / kModeWarmup
  int lambda_q8;
  int warmup_chunks;
  float log_tol;            // log(warmup_tol)
  int tol_noise;            // the tolerance of a segment is at least the noise floor at its start
  int n_seg_total;
  // workspace sections
  int* status;              // [0] code, [1] detail
  int* head_mode;           // [n_seqs * h_v]
  float* head_bound;        // [n_seqs * h_v]
  float* seg_bound;         // [n_seg_total * h_v] log warmup error bound of the chosen depth
  int* seg_w;               // [n_seg_total * h_v] warmup depth in chunks; -1: no depth up to the
                            // planned maximum meets the tolerance (the head runs exactly)
  float* R;                 // [n_seg_total, h_v, 128, 128] row-major (row = d_k in)
  float* Sloc;              // [n_seg_total, h_v, 128, 128] row = d_v
  float* Sstart;            // [n_seg_total, h_v, 128, 128] row = d_v
  // chunk index: chunks are numbered over all sequences in order
  int n_chunks_total;
  int32_t* seq_chunk_base;  // varlen: [n_seqs + 1] global index of each sequence's first chunk
  int4* chunk_info;         // varlen: [n_chunks_total] {sequence, valid tokens, first token (lo, hi)}
  float* chunk_exp;         // [n_chunks_total, h_v] warmup exponent of each chunk:
                            // sum over its tokens of g + log max(1, |1 - beta ||k||^2|)
  uint8_t* wy;              // [n_chunks_total, h_v] records of kRecBytes
  // Written for the backward only (null in a plain forward):
  uint8_t* wyA;             // [n_chunks_total, h_v] fp16 A^T = ((I + L)^{-1})^T, 64 x 64 in the
                            // 128-byte-swizzled image (8 KB each)
  uint8_t* hchunk;          // [n_chunks_total, h_v] fp16 chunk-start state S = H^T (rows d_v), two
                            // 128 x 64 panels (d_k 0-63 | 64-127) in the swizzled image (32 KB each)
  // Test hook (0 in normal use): the WY kernel's CTAs first wait this many
  // nanoseconds on an mbarrier nothing arrives on, so the bounded wait runs
  // out and the call takes its timeout path.
  uint32_t stall_ns;
};

// Backward arguments (gdn_chunk_bwd) beside the forward's Problem.
struct BwdArgs {
  const void* dout;    // [T, h_v, 128] bf16: gradient of o
  const float* dhT;    // [n_seqs, h_v, 128, 128] gradient of the final state, or null (zero)
  void* dq;            // [T, h_qk, 128] bf16
  void* dk;            // [T, h_qk, 128] bf16
  void* dv;            // [T, h_v, 128] bf16
  float* dg;           // [T, h_v]
  float* dbeta;        // [T, h_v]
  float* dh0;          // [n_seqs, h_v, 128, 128] or null (not written)
  // workspace, per (chunk, value head), fp16 in the 128-byte-swizzled image, 32 KB each:
  uint8_t* tmat;       // T' = -W^T Ktil (rows d_k out, panels d_k in)
  uint8_t* emat;       // E = scale (diag(gamma) Q)^T dO - W^T scale P^T dO (rows d_k, panels d_v)
  uint8_t* dstate;     // D = gradient of the chunk's end state (rows d_k, panels d_v)
};

// Arguments of the one-token step (gdn_decode_step).
struct DecodeArgs {
  const void* q;   // [n_seqs, h_qk, 128]
  const void* k;   // [n_seqs, h_qk, 128]
  const void* v;   // [n_seqs, h_v, 128]
  const float* g;  // [n_seqs, h_v]
  const float* beta;
  float* state;    // [n_seqs, h_v, 128, 128] (H = S^T), updated in place
  void* out;       // [n_seqs, h_v, 128]
  int n_seqs, h_qk, h_v;
  float scale;
};

__device__ __forceinline__ void report(int* status, int code, int detail) {
  if (atomicCAS(status, 0, code) == 0) atomicExch(status + 1, detail);
}

// The status word as the kernels before this one left it.  Each kernel of
// the forward after the chunk-local one reads it once (one thread, after
// grid_dependency_wait) and, if an earlier kernel reported a failure, does no
// work: its inputs would be incomplete.
__device__ __forceinline__ int earlier_failure(const int* status) {
  return *reinterpret_cast<const volatile int*>(status);
}

struct SegInfo {
  int n;         // sequence
  int s;         // segment within the sequence
  int n_seg;     // segments of the sequence
  int seg_base;  // global index of segment 0 of this sequence
  int n_chunks;  // chunks of the sequence
  int cb, ce;    // chunk range of this segment
  int64_t bos, eos;
};

// Global index of sequence n's first chunk: arithmetic for fixed-length rows,
// else from the chunk index built by chunk_map_kernel.
__device__ __forceinline__ int seq_first_chunk(const Problem& p, int n) {
  return p.cu ? p.seq_chunk_base[n] : n * chunks_of(p.T_row);
}

// Segments of sequence n (cp_off: one); -1 when its device offsets are not a
// range inside [0, T], or the first sequence does not start at 0 or the last
// end at T (the offsets disagree with the plan: nothing of it is touched).
__device__ __forceinline__ int seq_seg_count(const Problem& p, int n, int64_t& bos, int64_t& eos,
                                             int& n_chunks) {
  if (p.cu) {
    bos = p.cu[n];
    eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > (int64_t)p.T_row || (n == 0 && bos != 0) ||
        (n == p.n_seqs - 1 && eos != (int64_t)p.T_row)) {
      n_chunks = 0;
      return -1;
    }
  } else {
    bos = (int64_t)n * p.T_row;
    eos = bos + p.T_row;
  }
  n_chunks = chunks_of(eos - bos);
  return seg_count(n_chunks, p.lambda_q8, p.plan_mode == kModeOff);
}

// Locates global segment `seg` (warp-cooperative; call with a full warp,
// every lane gets the result).  Returns false if seg is out of range, if a
// sequence up to it has offsets outside [0, T], or if the sequence's segments
// reach past the plan's.
__device__ inline bool locate_segment(const Problem& p, int seg, SegInfo& out) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int n0 = 0; n0 < p.n_seqs; n0 += 32) {
    const int n = n0 + lane;
    int cnt = 0, nch = 0;
    int64_t bos = 0, eos = 0;
    if (n < p.n_seqs) cnt = seq_seg_count(p, n, bos, eos, nch);
    if (__any_sync(0xffffffffu, cnt < 0)) return false;
    int incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const int excl = base + incl - cnt;
    const bool mine = (n < p.n_seqs) && seg >= excl && seg < excl + cnt;
    const unsigned hit = __ballot_sync(0xffffffffu, mine);
    if (hit) {
      const int src = __ffs(hit) - 1;
      out.n = __shfl_sync(0xffffffffu, n, src);
      out.seg_base = __shfl_sync(0xffffffffu, excl, src);
      out.n_seg = __shfl_sync(0xffffffffu, cnt, src);
      out.n_chunks = __shfl_sync(0xffffffffu, nch, src);
      out.bos = __shfl_sync(0xffffffffu, bos, src);
      out.eos = __shfl_sync(0xffffffffu, eos, src);
      out.s = seg - out.seg_base;
      out.cb = seg_first(out.s, out.n_chunks, out.n_seg);
      out.ce = seg_first(out.s + 1, out.n_chunks, out.n_seg);
      return out.seg_base + out.n_seg <= p.n_seg_total;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
}

// Segment range of sequence n (warp-cooperative, every lane gets the result).
// Offsets outside [0, T] up to n, or segments reaching past the plan's, give
// no segments (n_seg = 0).
__device__ inline void locate_sequence(const Problem& p, int n, SegInfo& out) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  bool bad = false;
  for (int n0 = 0; n0 < n; n0 += 32) {
    const int m = n0 + lane;
    int cnt = 0, nch = 0;
    int64_t bos, eos;
    if (m < n) cnt = seq_seg_count(p, m, bos, eos, nch);
    bad |= __any_sync(0xffffffffu, cnt < 0);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
    base += cnt;
  }
  out.n = n;
  out.seg_base = base;
  out.n_seg = seq_seg_count(p, n, out.bos, out.eos, out.n_chunks);
  if (bad || out.n_seg < 0 || base + out.n_seg > p.n_seg_total) {
    out.n_seg = 0;
    out.n_chunks = 0;
  }
  out.s = 0;
  out.cb = 0;
  out.ce = out.n_chunks;
}

// Warmup depth of segment `cb` (its first chunk) of the sequence whose first
// global chunk is chunk0 (FlashQLA pages, section "AutoCP": a fast-decaying
// head restarts each segment from a few preceding chunks, which brings the
// state error below the noise floor).  A restart from zero w chunks early
// errs, relative to the state there, by at most exp(sum of the window's
// chunk exponents), since each token map X -> alpha X (I - beta k k^T) has
// spectral norm <= alpha max(1, |1 - beta ||k||^2|).  The tolerance is
// exp(log_tol), or with tol_noise the larger of that and the noise floor of
// the exact path at the segment start: each chunk rounds the state operand to
// fp16 (relative 2^-11), and that rounding m chunks back reaches the start
// scaled by at most the bound of the last m chunks, so the floor is 2^-11 (1
// + sum over the window's depths of their bounds, each capped at 1) -- a
// lower bound, since chunks before the window also contribute, and at most
// 9 x 2^-11 whatever the gates.  The depth is the smallest w <=
// the planned maximum whose bound is <= the tolerance; a window reaching the
// sequence start is exact (bound -inf); no such w gives -1 (the head runs
// exactly) with the full window's exponent.
__device__ inline void seg_warmup_depth(const Problem& p, int chunk0, int cb, int j, int& w_out, float& b_out) {
  const int nwin = min(p.warmup_chunks, cb);
  constexpr int kPre = 8;  // window exponents loaded together before the scan
  float pre[kPre];
#pragma unroll
  for (int w = 1; w <= kPre; ++w) pre[w - 1] = w <= nwin ? p.chunk_exp[(size_t)(chunk0 + cb - w) * p.h_v + j] : 0.f;
  float log_thr = p.log_tol;
  if (p.tol_noise) {
    float acc = 0.f, floor_sum = 1.f;
#pragma unroll
    for (int w = 1; w <= kPre; ++w)
      if (w <= nwin) {
        acc += pre[w - 1];
        floor_sum += __expf(fminf(acc, 0.f));
      }
    log_thr = fmaxf(log_thr, __logf(floor_sum) - 11.f * 0.69314718f);
  }
  float acc = 0.f;
  // true when depth w ends the search (w_out, b_out set)
  auto accept = [&](int w, float e) {
    acc += e;
    if (cb - w == 0) {
      w_out = w;
      b_out = -__int_as_float(0x7f800000);
      return true;
    }
    if (acc <= log_thr) {
      w_out = w;
      b_out = acc;
      return true;
    }
    return false;
  };
#pragma unroll
  for (int w = 1; w <= kPre; ++w)  // constant indices keep pre[] in registers
    if (w <= nwin && accept(w, pre[w - 1])) return;
  for (int w = kPre + 1; w <= nwin; ++w)
    if (accept(w, p.chunk_exp[(size_t)(chunk0 + cb - w) * p.h_v + j])) return;
  w_out = -1;
  b_out = acc;
}

// Warp-cooperative (call with a full warp; every lane gets the result): the
// mode a (sequence, head) takes under the plan -- warmup when every segment
// found a restart depth -- and the largest of its segments' warmup bounds.
// The segments' words are read in parallel across the lanes.
__device__ inline int head_mode_warp(const Problem& p, const SegInfo& si, int j, float* log_bound) {
  const int lane = threadIdx.x & 31;
  float m = -__int_as_float(0x7f800000);
  bool none = false;
  if (p.plan_mode == kModeWarmup) {
    for (int s = 1 + lane; s < si.n_seg; s += 32) {
      const size_t slot = (size_t)(si.seg_base + s) * p.h_v + j;
      none |= p.seg_w[slot] < 0;
      m = fmaxf(m, p.seg_bound[slot]);
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  none = __any_sync(0xffffffffu, none);
  if (log_bound) *log_bound = m;
  if (p.plan_mode == kModeOff) return kModeOff;
  if (p.plan_mode == kModeExact || none) return kModeExact;
  return kModeWarmup;
}

// Launches kernel<<<grid, block, smem, st>>>(args...); with `dependent`, as a
// programmatic dependent launch: its blocks may start while the previous
// kernel in the stream finishes, and wait for it (grid_dependency_wait)
// before they read anything an earlier kernel wrote.  Each kernel lets its
// dependents launch only after its own wait, so a kernel's blocks start only
// once every kernel before its predecessor has completed.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          bool dependent, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---- kernel launchers (defined in the .cu files) ----
// `dependent`: launched as a programmatic dependent of the kernel before it.
cudaError_t launch_chunk_map(const Problem& p, cudaStream_t st);
cudaError_t launch_wy(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      cudaStream_t st, bool dependent);
cudaError_t launch_scan_prep(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, cudaStream_t st);
cudaError_t launch_combine(const Problem& p, int sm_count, cudaStream_t st);
cudaError_t launch_scan_out(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mo,
                            int grid_x, cudaStream_t st);
cudaError_t launch_recurrence_f32(const Problem& p, cudaStream_t st, bool dependent);
cudaError_t launch_f32_prep(const Problem& p, cudaStream_t st);
cudaError_t f32_kernel_setup();
cudaError_t bwd_kernel_setup();
cudaError_t launch_decode(const DecodeArgs& a, bool f32, cudaStream_t st);
cudaError_t launch_combine_bwd(const Problem& p, int sm_count, cudaStream_t st);
cudaError_t launch_bwd_local_tc(const Problem& p, const BwdArgs& b, cudaStream_t st);
cudaError_t launch_bwd_chain_tc(const Problem& p, const BwdArgs& b, bool prep, cudaStream_t st);
cudaError_t launch_bwd_pre_tc(const Problem& p, const BwdArgs& b, cudaStream_t st);
cudaError_t scan_kernel_setup();
cudaError_t wy_kernel_setup();
cudaError_t combine_kernel_setup();

}  // namespace gdn
