/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated Delta Network chunked-prefill
 * forward.
 *
 * Sources cited below:
 *   [FlashQLA] the FlashQLA blog pages, "FlashQLA: fused linear-attention
 *     kernels for CP/backward (GDN)" (Traditional Chinese and Korean
 *     editions), sections "Optimising GDN chunked prefill", "AutoCP",
 *     "TileLang warp-specialised kernels", "Benchmarks", "Implementation and
 *     requirements"; and the Telegram post on FlashQLA (Russian) on the
 *     fast-decaying heads and the 6-8 chunk warmup.
 *   [GDN] Yang, Kautz, Hatamizadeh, "Gated Delta Networks: Improving Mamba2
 *     with Delta Rule", ICLR 2025, section "Gated delta rule" (the recurrence).
 *
 * The layer (per sequence, per value head j, tokens t in order):
 *   S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t = scale * S_t q_t
 * with S_t a d_v x d_k fp32 matrix, q/k taken from query/key head
 * floor(j * h_qk / h_v) (grouped heads) [GDN; FlashQLA, "Benchmarks" table
 * columns h_qk, h_v].  It is evaluated over 64-token chunks, aligned to each
 * sequence's own start, through the chunk-local WY form [FlashQLA,
 * "Optimising GDN chunked prefill"], optionally split into context-parallel
 * segments on one GPU [FlashQLA, "AutoCP"].
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are ordinary host memory.  The caller owns all memory,
 *     including the workspace; the library allocates nothing and keeps no
 *     per-call state.  The only global state is a per-device cache of the
 *     SM count and of the kernel attribute set-up.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device
 *     work is enqueued asynchronously; nothing synchronises except
 *     gdn_get_device_status.
 *   - Every entry point returns a gdn_status.  No exception crosses the ABI.
 *     Kernels never trap: a kernel that fails its own bounds/consistency
 *     check, or whose bounded wait runs out, records a code in the
 *     workspace's status word (read it with gdn_get_device_status) and
 *     returns.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,    /* null pointer, bad size, inconsistent dims/plan */
  GDN_ERR_UNSUPPORTED = 2,    /* d_k or d_v != 128, unknown dtype or mode */
  GDN_ERR_MISALIGNED = 3,     /* a device pointer not 16-byte (workspace: 256-byte) aligned */
  GDN_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed; see gdn_last_cuda_error() */
  GDN_ERR_DEVICE_TIMEOUT = 5, /* (from gdn_get_device_status) a bounded on-device wait ran out */
  GDN_ERR_WORKSPACE = 6,      /* workspace missing or smaller than plan->workspace_bytes */
  GDN_ERR_DEVICE_CHECK = 7    /* (from gdn_get_device_status) a kernel's own check failed */
} gdn_status;

/* Element types of q, k, v and out.  g, beta, states are always fp32.
 *   GDN_BF16: the chunked tcgen05 path (fp16 MMA operands, fp32 accumulation),
 *             with the plan's context parallelism.
 *   GDN_F32:  fp32 throughout, on the CUDA cores: the recurrence itself,
 *             one state row per thread pair, with the plan's segments always
 *             combined exactly (a WARMUP plan runs as EXACT).  For results
 *             within 1e-4 of exact. */
enum { GDN_BF16 = 0, GDN_F32 = 1 };

/* Intra-card context parallelism [FlashQLA, "AutoCP"]. */
enum {
  GDN_CP_OFF = 0,    /* one CTA-level scan per (sequence, value head) */
  GDN_CP_EXACT = 1,  /* segments; start states combined exactly through M */
  GDN_CP_WARMUP = 2, /* segments; a (sequence, head) whose gate bound is under
                        its tolerance (see tol_rule) restarts each segment
                        from zero up to warmup_chunks chunks early and skips
                        M; the others run exactly */
  GDN_CP_AUTO = 3    /* WARMUP when n_seqs * h_v < sm_count, else OFF */
};

/* How a warmup restart's tolerance is set [FlashQLA, "AutoCP": a restart is
 * good once the state error it leaves is under the noise floor].
 *   GDN_TOL_FIXED: warmup_tol, the same for every head and segment.
 *   GDN_TOL_NOISE: per (sequence, value head) and segment, the larger of
 *     warmup_tol and the noise floor of the exact bf16 path at the segment
 *     start: the fp16 rounding of the state operand in every chunk (relative
 *     2^-11) carried to the start, 2^-11 * (1 + sum over m = 1..w of
 *     min(1, the bound of the last m chunks before the start)), w =
 *     min(warmup_chunks, 8, chunks before the start); so at most 9 * 2^-11.  A head whose gates decay slowly carries more
 *     of that rounding, so its floor, and the depth error it tolerates, is
 *     higher; the warmup error stays below the error the exact path makes
 *     anyway.  The fp32 path always combines exactly. */
enum { GDN_TOL_FIXED = 0, GDN_TOL_NOISE = 1 };

typedef struct gdn_dims {
  int B;      /* batch; must be 1 when cu_seqlens is used */
  int T;      /* tokens per batch row (varlen: total packed tokens) */
  int h_qk;   /* query/key heads */
  int h_v;    /* value heads (one recurrent state each) */
  int d_k;    /* key dim; must be 128 */
  int d_v;    /* value dim; must be 128 */
  int n_seqs; /* varlen: number of sequences (len(cu_seqlens) - 1); fixed length: B */
  float scale; /* output scale; 0 selects 1/sqrt(d_k) */
  int dtype;   /* GDN_BF16 or GDN_F32 */
} gdn_dims;

typedef struct gdn_cp_opts {
  int mode;          /* GDN_CP_* */
  float lambda;      /* segment length L = round(lambda * sqrt(N)) chunks, lambda used in
                        steps of 1/256; <= 0 lets the planner choose it: the lambda (a
                        multiple of 1/8) minimising 2 x (finish of the list schedule of
                        the scan's CTAs in launch order on sm_count SMs, each taking its
                        segment's chunks + 3) + 2 x (most segments of one sequence: a
                        combine step costs about a chunk-time); ties go
                        to fewer segments.  For GDN_F32, whose chains run two CTAs per
                        SM and whose chunks dwarf a combine step, the schedule has 2 x
                        sm_count slots, a CTA takes its chunks alone, and the score is
                        2 x the finish */
  int warmup_chunks; /* warmup restart depth w in chunks; <= 0 selects 8 */
  float warmup_tol;  /* accept warmup for a (sequence, head) when, for every segment,
                        some depth w <= warmup_chunks has its bound exp(sum over the w
                        chunks before the segment of g + log max(1, |1 - beta ||k||^2|))
                        <= the segment's tolerance (see tol_rule); <= 0 selects 1e-4 */
  int sm_count;      /* SMs to plan for; <= 0 queries the current device */
  int tol_rule;      /* GDN_TOL_FIXED or GDN_TOL_NOISE (NULL opts: GDN_TOL_NOISE) */
} gdn_cp_opts;

/* Plain-data plan; fill with gdn_cp_plan, do not edit. */
typedef struct gdn_cp_plan_t {
  int mode;             /* resolved mode: GDN_CP_OFF, GDN_CP_EXACT or GDN_CP_WARMUP */
  int n_seqs;           /* sequences the plan was made for */
  int T_total;          /* B * T */
  int h_v, h_qk, dtype; /* copied from dims, checked by gdn_chunk_fwd */
  int lambda_q8;        /* lambda * 256, rounded */
  int warmup_chunks;
  float warmup_tol;
  int sm_count;
  int tol_rule;         /* GDN_TOL_FIXED or GDN_TOL_NOISE */
  int n_seg_total;      /* segments summed over sequences */
  int max_seg_chunks;   /* longest segment, in chunks */
  int max_chunks;       /* longest sequence, in chunks */
  size_t workspace_bytes;
  size_t off_head;      /* byte offsets of the workspace sections */
  size_t off_seg_bound;
  size_t off_R, off_Sloc, off_Sstart;
  int n_chunks_total;   /* 64-token chunks summed over sequences */
  size_t off_chunk_map; /* chunk index: first chunk of each sequence, sequence of each chunk */
  size_t off_wy;        /* chunk-local records (-W, U, P, gates), 41472 bytes per (chunk, value head) */
} gdn_cp_plan_t;

/*
 * gdn_cp_plan -- host-only planning [FlashQLA, "AutoCP": L = lambda * sqrt(N),
 * N = chunks, L = chunks per segment].  No device work.
 *   dims              : problem sizes (see gdn_dims).
 *   cu_seqlens_host   : n_seqs+1 non-decreasing token offsets starting at 0
 *                       and ending at T, or NULL for B fixed-length rows of T.
 *   opts              : may be NULL (all defaults: mode AUTO, lambda chosen by
 *                       the planner, warmup up to 8 chunks at 1e-4 or the noise
 *                       floor (GDN_TOL_NOISE), SMs of the device).  A tol_rule
 *                       other than GDN_TOL_FIXED or GDN_TOL_NOISE is refused
 *                       with GDN_ERR_UNSUPPORTED.
 *   out_plan          : written on success.
 * Segmentation of a sequence with N = ceil(len/64) chunks: L = max(1,
 * floor((isqrt(lambda_q8^2 * N) + 128) / 256)), n_seg = max(1, ceil(N / L)),
 * segment s = chunks [floor(s N / n_seg), floor((s+1) N / n_seg)).  Mode OFF
 * uses one segment per sequence.  An empty sequence has one empty segment.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA (only when opts->sm_count <= 0 and
 * the device query fails).
 */
gdn_status gdn_cp_plan(const gdn_dims* dims, const int32_t* cu_seqlens_host,
                       const gdn_cp_opts* opts, gdn_cp_plan_t* out_plan);

/*
 * gdn_chunk_fwd -- the chunked-prefill forward [FlashQLA, "Optimising GDN
 * chunked prefill", "AutoCP", "TileLang warp-specialised kernels" (forward
 * pass: V', S and O)].  Asynchronous on `stream`.
 *   q, k          : device, [B*T, h_qk, d_k] (token-major, heads interleaved), dims->dtype.
 *   v             : device, [B*T, h_v, d_v], dims->dtype.
 *   g             : device, [B*T, h_v] fp32, log of the decay gate (alpha = exp(g)).
 *   beta          : device, [B*T, h_v] fp32, write strength.
 *   initial_state : device, [n_seqs, h_v, d_k, d_v] fp32 (H = S^T), or NULL for zeros.
 *   cu_seqlens_dev: device int32 [n_seqs+1], the same offsets given to gdn_cp_plan,
 *                   or NULL for fixed-length rows.  The kernels check them before
 *                   following them: offsets outside [0, T], going back, not ending
 *                   at T, or giving other chunk or segment counts than the plan's
 *                   are reported as GDN_ERR_DEVICE_CHECK with detail 3 in the status
 *                   word, and no access follows them outside the buffers (o and
 *                   final_state are then incomplete).  Other boundaries with the
 *                   same counts go undetected.
 *   out           : device, [B*T, h_v, d_v], dims->dtype (bf16 rounded to nearest even).
 *   final_state   : device, [n_seqs, h_v, d_k, d_v] fp32, or NULL (not written).
 *   dims, plan    : host; plan must come from gdn_cp_plan with these dims.
 *   workspace     : device, 256-byte aligned; its contents on entry do not
 *                   matter.  Must not be shared by calls that may run
 *                   concurrently.
 *   workspace_bytes: size of `workspace`; must be >= plan->workspace_bytes.
 * All device pointers must be 16-byte aligned.  q/k/v/out may not overlap.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA (launch failure).
 */
gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* initial_state,
                         const int32_t* cu_seqlens_dev, void* out, float* final_state,
                         const gdn_dims* dims, const gdn_cp_plan_t* plan, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static storage). */
const char* gdn_status_string(gdn_status status);

/* The cudaError_t of the most recent GDN_ERR_CUDA on this thread (0 if none). */
int gdn_last_cuda_error(void);

/*
 * gdn_get_device_status -- synchronises `stream`, then reads the status word
 * the kernels of the last gdn_chunk_fwd on this workspace wrote.
 *   workspace : device workspace passed to gdn_chunk_fwd.
 *   code      : host; receives GDN_OK, GDN_ERR_DEVICE_TIMEOUT or GDN_ERR_DEVICE_CHECK.
 *   detail    : host, may be NULL; receives a kernel-specific detail word.
 * Returns CUDA on a failed copy/sync, INVALID_ARG on null pointers.
 */
gdn_status gdn_get_device_status(const void* workspace, void* stream, int* code, int* detail);

/*
 * gdn_cp_head_modes -- diagnostics: synchronises `stream` and copies, per
 * (sequence, value head), the mode the last gdn_chunk_fwd on this workspace
 * took (GDN_CP_EXACT or GDN_CP_WARMUP; GDN_CP_OFF for plans without CP; always
 * GDN_CP_EXACT on the fp32 path with CP; the plan's mode when every sequence
 * is a single segment, where nothing is combined or restarted) and
 * the natural log of its warmup error bound (-inf when no segment needs one).
 *   modes_host    : host int32 [n_seqs * h_v], or NULL.
 *   log_bound_host: host fp32 [n_seqs * h_v], or NULL.
 */
gdn_status gdn_cp_head_modes(const void* workspace, const gdn_cp_plan_t* plan, int32_t* modes_host,
                             float* log_bound_host, void* stream);

/*
 * gdn_chunk_fwd_static -- gdn_chunk_fwd for callers that cannot allocate
 * device memory.  The FlashQLA pages have no counterpart: this is a library
 * convenience.  Some callers can't call cudaMalloc or hand out scratch: code
 * running under a runtime that owns all device memory (an inference
 * server's arena, a plugin interface that passes only its inputs and
 * outputs), or code that must not allocate after start-up.  This entry point
 * takes the same arguments as gdn_chunk_fwd minus the workspace and uses a
 * fixed 8 MiB device array built into the library instead; every GPU that
 * loads the library holds that array until the process exits.
 *   - Fits plans whose plan->workspace_bytes is at most 8 MiB: the chunk
 *     records take 41472 bytes per (chunk, value head), so about 200
 *     chunk-heads (e.g. 1000 tokens with 12 value heads, context parallelism
 *     off; with it, each segment adds 192 KB per value head of segment
 *     states); larger plans are rejected with GDN_ERR_WORKSPACE before any
 *     device work.
 *   - Allocates nothing.  Its first call on a device looks up the array's
 *     device address (cudaGetSymbolAddress) with that device current; make
 *     that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     every part the forward reads is written or cleared within the call.
 *     Calls that may overlap on the GPU (other streams, other host threads)
 *     race on the array: serialise them.
 *   - The device status word of these calls lives in the shared array;
 *     read it with gdn_get_static_device_status.
 * Errors: as gdn_chunk_fwd, plus WORKSPACE for plans above the limit.
 */
gdn_status gdn_chunk_fwd_static(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* initial_state,
                                const int32_t* cu_seqlens_dev, void* out, float* final_state,
                                const gdn_dims* dims, const gdn_cp_plan_t* plan, void* stream);

/*
 * gdn_get_static_device_status -- gdn_get_device_status for the calls of
 * gdn_chunk_fwd_static on the current device: synchronises `stream`, then
 * reads the status word the kernels of the last such call wrote into the
 * library's built-in array (no counterpart on the FlashQLA pages).  The
 * first use on a device looks up the array's address like
 * gdn_chunk_fwd_static does.
 *   code   : host; receives GDN_OK, GDN_ERR_DEVICE_TIMEOUT or GDN_ERR_DEVICE_CHECK.
 *   detail : host, may be NULL; receives the kernel-specific detail word.
 * Errors: INVALID_ARG (code NULL), CUDA (address lookup, copy or sync failed).
 */
gdn_status gdn_get_static_device_status(void* stream, int* code, int* detail);

/*
 * gdn_decode_step -- one new token for each of a batch of sequences: the
 * recurrence step itself [GDN, "Gated delta rule"], the generation-time
 * counterpart of gdn_chunk_fwd.  Per sequence n and value head j (q/k head
 * floor(j * h_qk / h_v)):
 *   S <- exp(g) S (I - beta k k^T) + beta v k^T,   o = scale * S q,
 * with the state stored as H = S^T like initial_state/final_state, so the
 * final_state of a prefill continues here directly.  fp32 arithmetic on the
 * CUDA cores; asynchronous on `stream`.
 *   q, k  : device, [B, h_qk, d_k], dims->dtype.
 *   v     : device, [B, h_v, d_v], dims->dtype.
 *   g, beta: device, [B, h_v] fp32.
 *   state : device, [B, h_v, d_k, d_v] fp32; read, then overwritten with the
 *           new state.
 *   out   : device, [B, h_v, d_v], dims->dtype (bf16 rounded to nearest even).
 *   dims  : B sequences, T must be 1, n_seqs must equal B; d_k = d_v = 128.
 * No workspace.  out may not overlap the inputs or the state.
 * Errors: INVALID_ARG (null pointer, T != 1, n_seqs != B), UNSUPPORTED,
 * MISALIGNED (16 bytes), CUDA (launch failure).
 */
gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                           float* state, void* out, const gdn_dims* dims, void* stream);

/*
 * gdn_bwd_workspace_bytes -- device workspace gdn_chunk_bwd needs for `plan`:
 * the forward's plan->workspace_bytes, then, per (chunk, value head), 136 KB
 * (A^T, the chunk-start state and three 32 KB backward tiles), then a bf16
 * copy of o.  Host only.  Errors: INVALID_ARG (NULL), UNSUPPORTED (fp32 plan).
 */
gdn_status gdn_bwd_workspace_bytes(const gdn_cp_plan_t* plan, size_t* bytes);

/*
 * gdn_chunk_bwd -- gradients of the chunked-prefill forward [FlashQLA,
 * "TileLang warp-specialised kernels" (backward pass: the dv, state-gradient,
 * dq/dk/dw/dg and WY gradient steps); the pages give no formulas: these are
 * the exact gradients of gdn_chunk_fwd's function].  For the scalar
 *   sum(o * d_out) + sum(final_state * d_final_state),
 * writes its gradient with respect to q, k, v, g, beta and initial_state.
 * Asynchronous on `stream`.  The forward is recomputed inside the call unless
 * reuse_forward = 1, in which case `workspace` must hold the state a
 * gdn_chunk_fwd_train with the same inputs and plan left there.  The chunk
 * states the gradients use are the forward's in the plan's mode (with
 * GDN_CP_AUTO, a warmup restart where the forward's acceptance rule allows
 * one, so they agree with the exact states within its tolerance; GDN_CP_EXACT
 * gives the exact forward's gradients); the state gradient's own chain is
 * always combined exactly.  bf16 only.
 *   q, k, v, g, beta, initial_state, cu_seqlens_dev, dims, plan: as gdn_chunk_fwd.
 *   d_out         : device, [B*T, h_v, d_v] bf16.
 *   d_final_state : device, [n_seqs, h_v, d_k, d_v] fp32, or NULL (zero).
 *   dq, dk        : device, [B*T, h_qk, d_k] bf16 (summed over each q/k head's value heads).
 *   dv            : device, [B*T, h_v, d_v] bf16.
 *   dg, dbeta     : device, [B*T, h_v] fp32.
 *   d_initial_state: device, [n_seqs, h_v, d_k, d_v] fp32, or NULL (not written);
 *                   written also when initial_state is NULL (the gradient at zero).
 *   workspace     : device, 256-byte aligned, at least gdn_bwd_workspace_bytes(plan).
 * All device pointers 16-byte aligned; outputs may not overlap inputs.
 * Kernels report through the workspace status word like the forward's
 * (gdn_get_device_status), including GDN_ERR_DEVICE_CHECK when an fp16
 * operand of the backward left the fp16 range.
 * Errors: INVALID_ARG, UNSUPPORTED (fp32 dtype), MISALIGNED, WORKSPACE, CUDA.
 */
gdn_status gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* initial_state, const int32_t* cu_seqlens_dev, const void* d_out,
                         const float* d_final_state, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                         float* d_initial_state, const gdn_dims* dims, const gdn_cp_plan_t* plan,
                         void* workspace, size_t workspace_bytes, int reuse_forward, void* stream);

/*
 * gdn_chunk_fwd_train -- gdn_chunk_fwd that also keeps, in `workspace`, what
 * gdn_chunk_bwd needs (no counterpart on the FlashQLA pages: the training
 * pattern of forward then backward).  Same arguments and outputs as
 * gdn_chunk_fwd; the workspace must hold gdn_bwd_workspace_bytes(plan).  It
 * runs in the plan's mode like gdn_chunk_fwd (o and final_state are the same);
 * besides them the call writes A^T and every chunk's start state into the
 * workspace.  A later
 * gdn_chunk_bwd with the same inputs, plan and workspace and reuse_forward = 1
 * then skips its own recompute; nothing checks that the inputs are the same.
 * bf16 only.  Errors: as gdn_chunk_fwd, UNSUPPORTED for fp32.
 */
gdn_status gdn_chunk_fwd_train(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens_dev, void* out,
                               float* final_state, const gdn_dims* dims, const gdn_cp_plan_t* plan,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_debug_stall_ns -- test hook of the failure path (no counterpart on the
 * FlashQLA pages).  While ns > 0, each later gdn_chunk_fwd of this process on
 * the bf16 path makes the blocks of its chunk-local kernel first wait ns
 * nanoseconds on an mbarrier that nothing arrives on.  That bounded wait
 * runs out: the blocks record GDN_ERR_DEVICE_TIMEOUT with detail 6 in the
 * workspace's status word, free their tensor memory and return, and every
 * kernel after them sees the recorded failure and does no work, so o and
 * final_state are left unwritten.  ns = 0 (the default) turns it off.  A
 * process-wide setting for tests; not for production calls.
 * Errors: none.
 */
gdn_status gdn_debug_stall_ns(uint32_t ns);

/*
 * gdn_set_trace_events -- optional per-kernel timing (tracing).  Registers,
 * for the calling host thread, up to 32 caller-created cudaEvent_t handles.
 * While registered, each gdn_chunk_fwd (gdn_chunk_bwd, gdn_decode_step) on this thread
 * brackets its i-th kernel launch with events[2i] (recorded right before the
 * launch) and events[2i + 1] (right after it), both on the stream the kernel
 * is launched on, so cudaEventElapsedTime(events[2i], events[2i + 1]) is the
 * device time of kernel i.  n_events = 0 (or events = NULL) turns tracing
 * off.  The caller keeps ownership of the events.
 * Errors: INVALID_ARG for n_events outside 0..32 or a NULL event.
 */
gdn_status gdn_set_trace_events(void* const* events, int n_events);

/*
 * gdn_trace_last -- names of the kernels the last gdn_chunk_fwd (gdn_chunk_bwd,
 * gdn_decode_step) on this thread launched, in launch order (static
 * strings), and their count (at most 16).
 *   names : host array of at least max_names pointers, or NULL.
 * Returns the number of kernels launched (0 before any call).
 */
int gdn_trace_last(const char** names, int max_names);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
