// Host side of the C ABI declared in include/gdn.h: planning, argument
// checks, TMA tensor maps, and the launch sequence of the forward.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <climits>
#include <cstring>
#include <mutex>
#include <vector>

#include "gdn.h"
#include "gdn_internal.cuh"

using namespace gdn;

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint32_t> g_debug_stall_ns{0};  // test hook of the timeout path (gdn_debug_stall_ns)

// ---- tracing: caller-provided events recorded around each launch ----
// Kernel i of a call is bracketed by events 2i and 2i + 1, recorded on the
// stream it is launched on.
constexpr int kMaxTrace = 32;
thread_local cudaEvent_t g_trace_ev[kMaxTrace];
thread_local int g_trace_n = 0;
thread_local const char* g_last_names[kMaxTrace / 2];
thread_local int g_last_count = 0;

struct LaunchLog {
  // keep: continue the list of the call's kernels (the backward after its forward)
  explicit LaunchLog(bool keep = false) {
    if (!keep) g_last_count = 0;
  }
  // Records the start event of the next kernel on st.
  cudaError_t before(cudaStream_t st) {
    const int k = 2 * g_last_count;
    return k < g_trace_n ? cudaEventRecord(g_trace_ev[k], st) : cudaSuccess;
  }
  // Names the kernel just launched on st and records its end event.
  cudaError_t after(const char* name, cudaStream_t st) {
    const int k = 2 * g_last_count + 1;
    if (g_last_count < kMaxTrace / 2) g_last_names[g_last_count++] = name;
    return k < g_trace_n ? cudaEventRecord(g_trace_ev[k], st) : cudaSuccess;
  }
};

gdn_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return GDN_ERR_CUDA;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- one-time, per-device set-up ----
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
bool g_setup_done[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

gdn_status device_setup(int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  *dev_out = dev;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_setup_done[dev]) return GDN_OK;
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(e == cudaSuccess ? cudaErrorUnknown : e);
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if ((e = scan_kernel_setup()) != cudaSuccess) return cuda_fail(e);
  if ((e = wy_kernel_setup()) != cudaSuccess) return cuda_fail(e);
  if ((e = combine_kernel_setup()) != cudaSuccess) return cuda_fail(e);
  if ((e = f32_kernel_setup()) != cudaSuccess) return cuda_fail(e);
  if ((e = bwd_kernel_setup()) != cudaSuccess) return cuda_fail(e);
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
  g_sm_count[dev] = sms;
  g_setup_done[dev] = true;
  return GDN_OK;
}

// AutoCP's choice of lambda (FlashQLA pages, section "AutoCP": the degree
// of parallelism follows L = lambda sqrt(N)).  The scan kernel runs one CTA
// per (segment, value head), one CTA per SM; a CTA takes about (segment
// chunks + 3) chunk-times (start-up, pipeline fill and warmup chunks).  The
// block scheduler hands CTAs out in launch order (the segments of sequence
// 0, 1, ..., then the next value head) to whichever SM frees first, so the
// planner replays that list schedule.  The combine then walks each
// sequence's segments in order, about a chunk-time per segment.  Among
// lambda = k/8 the planner takes the smallest (schedule finish + the largest
// segment count of a sequence); ties go to fewer segments.
namespace {

constexpr int kCtaOverheadChunks = 3;

// The model's constants per path.  The bf16 scan: a CTA costs its chunks + 3
// (start-up, pipeline fill, warmup) and a combine step about a chunk.
// The fp32 path: a chunk is ~40x a combine step and the start-up is small
// against a chunk, so both count zero; its chains run two CTAs per SM.
struct PlanModel {
  int overhead;     // chunk-times a CTA costs beyond its chunks
  bool combine;     // count the combine's serial steps
};

struct SegStats {
  int64_t segs = 0;
  int longest = 0, most_segs = 0;
  int64_t work = 0;  // sum of (chunks + overhead) over one head's segments
};

SegStats seg_stats(const gdn_dims* d, const int32_t* cu, int q8, const PlanModel& m) {
  SegStats r;
  for (int n = 0; n < d->n_seqs; ++n) {
    const int64_t len = cu ? (int64_t)cu[n + 1] - cu[n] : d->T;
    const int N = chunks_of(len);
    const int ns = seg_count(N, q8, false);
    r.segs += ns;
    r.work += N + (int64_t)ns * m.overhead;
    r.longest = std::max(r.longest, (N + ns - 1) / ns);  // balanced split: ceil(N / ns) at most
    r.most_segs = std::max(r.most_segs, ns);
  }
  return r;
}

// Finish time of the list schedule of the scan's CTAs on sm_count SMs.  The
// earliest free time never decreases along the schedule, so SM free times
// are kept as counts per time step and the earliest is found by a forward
// scan; the finish is at most total / sm_count + the longest CTA (the list
// scheduling bound), which sizes the count array.
int64_t list_schedule(const gdn_dims* d, const int32_t* cu, int q8, int sm_count, const SegStats& st,
                      const PlanModel& m, std::vector<int32_t>& free_at) {
  const int64_t horizon = st.work * d->h_v / sm_count + st.longest + m.overhead + 2;
  free_at.assign((size_t)horizon, 0);
  free_at[0] = sm_count;
  int64_t t = 0, finish = 0;
  for (int j = 0; j < d->h_v; ++j)
    for (int n = 0; n < d->n_seqs; ++n) {
      const int64_t len = cu ? (int64_t)cu[n + 1] - cu[n] : d->T;
      const int N = chunks_of(len);
      const int ns = seg_count(N, q8, false);
      for (int s = 0; s < ns; ++s) {
        while (free_at[(size_t)t] == 0) ++t;
        --free_at[(size_t)t];
        const int64_t end = t + seg_first(s + 1, N, ns) - seg_first(s, N, ns) + m.overhead;
        ++free_at[(size_t)end];
        finish = std::max(finish, end);
      }
    }
  return finish;
}

}  // namespace

int pick_lambda_q8_uncached(const gdn_dims* d, const int32_t* cu, int slots, const PlanModel& m) {
  int best_q8 = 256;
  int64_t best_cost = INT64_MAX, best_segs = INT64_MAX;
  std::vector<int32_t> free_at;
  for (int q8 = 32; q8 <= 4096; q8 += 32) {
    const SegStats st = seg_stats(d, cu, q8, m);
    const int64_t comb = m.combine ? 2 * st.most_segs : 0;
    // in half chunk-times; no schedule ends before its longest CTA or the average slot load
    const int64_t total = st.work * d->h_v;
    const int64_t lower = 2 * std::max<int64_t>(st.longest + m.overhead, (total + slots - 1) / slots) + comb;
    if (lower > best_cost || (lower == best_cost && st.segs >= best_segs)) continue;
    const int64_t cost = 2 * list_schedule(d, cu, q8, slots, st, m, free_at) + comb;
    if (cost < best_cost || (cost == best_cost && st.segs < best_segs)) {
      best_cost = cost;
      best_segs = st.segs;
      best_q8 = q8;
    }
  }
  return best_q8;
}

// The choice depends only on the sequence lengths, h_v, the SM count and the
// path; a model plans the same lengths once per layer, so recent choices are
// kept.
int pick_lambda_q8(const gdn_dims* d, const int32_t* cu, int sm_count) {
  struct Entry {
    int h_v, sm_count, dtype;
    std::vector<int64_t> lens;
    int q8;
  };
  static std::mutex mu;
  static std::vector<Entry> recent;  // most recent last
  std::vector<int64_t> lens((size_t)d->n_seqs);
  for (int n = 0; n < d->n_seqs; ++n) lens[(size_t)n] = cu ? (int64_t)cu[n + 1] - cu[n] : d->T;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : recent)
      if (e.h_v == d->h_v && e.sm_count == sm_count && e.dtype == d->dtype && e.lens == lens) return e.q8;
  }
  const bool f32 = d->dtype == GDN_F32;
  const PlanModel m = f32 ? PlanModel{0, false} : PlanModel{kCtaOverheadChunks, true};
  const int q8 = pick_lambda_q8_uncached(d, cu, f32 ? 2 * sm_count : sm_count, m);
  std::lock_guard<std::mutex> lk(mu);
  if (recent.size() >= 8) recent.erase(recent.begin());
  recent.push_back(Entry{d->h_v, sm_count, d->dtype, std::move(lens), q8});
  return q8;
}

gdn_status check_dims(const gdn_dims* d) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->d_k != kDim || d->d_v != kDim) return GDN_ERR_UNSUPPORTED;
  if (d->dtype != GDN_BF16 && d->dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
  if (d->B < 1 || d->T < 0 || d->h_qk < 1 || d->h_v < 1 || d->n_seqs < 1) return GDN_ERR_INVALID_ARG;
  if ((int64_t)d->B * d->T > (int64_t)0x7fffffff - kChunk) return GDN_ERR_INVALID_ARG;
  if (d->h_qk > 65535 || d->h_v > 65535) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

// ---- tensor maps: [tokens, heads, 128] -> 3-D (d, head, token), 64x1x64 boxes, 128B swizzle ----
gdn_status encode_map(CUtensorMap* m, const void* base, int heads, int64_t tokens, bool f32) {
  const cuuint64_t esz = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * esz, (cuuint64_t)heads * kDim * esz};
  cuuint32_t box[3] = {(cuuint32_t)(f32 ? 32 : 64), 1, (cuuint32_t)kChunk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = (int)r;
    return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

// o: [tokens, h_v, 128] bf16 -> 3-D (d, head, token), whole 128 x 1 x 64 boxes, no swizzle
// (the scan stores each chunk's o from a plain [64][128] shared-memory tile).
gdn_status encode_out_map(CUtensorMap* m, void* base, int heads, int64_t tokens) {
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)heads * kDim * 2};
  cuuint32_t box[3] = {(cuuint32_t)kDim, 1, (cuuint32_t)kChunk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = (int)r;
    return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

// ---- fixed device workspace for callers that cannot allocate ----
// 8 MiB: small problems only (the chunk records take 41472 bytes per
// (chunk, value head); context parallelism adds three 64 KB states per
// (segment, value head)).
constexpr size_t kStaticWorkspaceBytes = size_t(8) << 20;
static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];
void* g_static_ws_dev[kMaxDevices] = {};

// Device address of g_static_workspace on the current device, looked up once
// per device (the host-side name is not a device address).
gdn_status static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_static_ws_dev[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess || !ptr) return cuda_fail(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
    g_static_ws_dev[dev] = ptr;
  }
  *out = g_static_ws_dev[dev];
  return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported (d_k/d_v must be 128; dtype bf16 or f32)";
    case GDN_ERR_MISALIGNED: return "misaligned pointer (16 bytes; workspace 256 bytes)";
    case GDN_ERR_CUDA: return "CUDA call failed";
    case GDN_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait timed out";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    case GDN_ERR_DEVICE_CHECK: return "a kernel's consistency check failed";
  }
  return "unknown status";
}

int gdn_last_cuda_error(void) { return g_last_cuda_error; }

gdn_status gdn_cp_plan(const gdn_dims* dims, const int32_t* cu, const gdn_cp_opts* opts, gdn_cp_plan_t* out) {
  if (!out) return GDN_ERR_INVALID_ARG;
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  const int64_t T_total = (int64_t)dims->B * dims->T;
  if (cu) {
    if (dims->B != 1) return GDN_ERR_INVALID_ARG;
    if (cu[0] != 0 || cu[dims->n_seqs] != dims->T) return GDN_ERR_INVALID_ARG;
    for (int n = 0; n < dims->n_seqs; ++n)
      if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARG;
  } else if (dims->n_seqs != dims->B) {
    return GDN_ERR_INVALID_ARG;
  }
  gdn_cp_opts o = {GDN_CP_AUTO, 0.0f, 8, 1e-4f, 0, GDN_TOL_NOISE};  // NULL opts: the planner picks lambda
  if (opts) o = *opts;
  if (o.mode < GDN_CP_OFF || o.mode > GDN_CP_AUTO) return GDN_ERR_UNSUPPORTED;
  if (o.tol_rule != GDN_TOL_FIXED && o.tol_rule != GDN_TOL_NOISE) return GDN_ERR_UNSUPPORTED;
  const bool auto_lambda = !(o.lambda > 0.f);
  if (o.lambda > 1000.f) return GDN_ERR_INVALID_ARG;
  if (o.warmup_chunks <= 0) o.warmup_chunks = 8;
  if (!(o.warmup_tol > 0.f)) o.warmup_tol = 1e-4f;
  if (o.sm_count <= 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    o.sm_count = sms;
  }
  int mode = o.mode;
  if (mode == GDN_CP_AUTO) mode = ((int64_t)dims->n_seqs * dims->h_v < o.sm_count) ? GDN_CP_WARMUP : GDN_CP_OFF;

  gdn_cp_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.mode = mode;
  p.n_seqs = dims->n_seqs;
  p.T_total = (int)T_total;
  p.h_v = dims->h_v;
  p.h_qk = dims->h_qk;
  p.dtype = dims->dtype;
  if (auto_lambda) {
    p.lambda_q8 = mode == GDN_CP_OFF ? 256 : pick_lambda_q8(dims, cu, o.sm_count);
  } else {
    p.lambda_q8 = (int)std::lround(o.lambda * 256.0);
    if (p.lambda_q8 < 1) p.lambda_q8 = 1;
  }
  p.warmup_chunks = o.warmup_chunks;
  p.warmup_tol = o.warmup_tol;
  p.sm_count = o.sm_count;
  p.tol_rule = o.tol_rule;
  int64_t n_seg_total = 0, n_chunks_total = 0;
  for (int n = 0; n < dims->n_seqs; ++n) {
    const int64_t len = cu ? (int64_t)cu[n + 1] - cu[n] : dims->T;
    const int N = chunks_of(len);
    n_chunks_total += N;
    const int ns = seg_count(N, p.lambda_q8, mode == GDN_CP_OFF);
    n_seg_total += ns;
    if (N > p.max_chunks) p.max_chunks = N;
    for (int s = 0; s < ns; ++s) {
      const int w = seg_first(s + 1, N, ns) - seg_first(s, N, ns);
      if (w > p.max_seg_chunks) p.max_seg_chunks = w;
    }
  }
  if (n_seg_total > 0x7fffffff) return GDN_ERR_INVALID_ARG;
  if (n_chunks_total * std::max(dims->h_v, dims->h_qk) > 0x7fffffff) return GDN_ERR_INVALID_ARG;
  p.n_seg_total = (int)n_seg_total;
  p.n_chunks_total = (int)n_chunks_total;
  // workspace: status | head modes + bounds | segment bounds | R | S_loc | S_start |
  //            chunk index | chunk records (the last two: bf16 path only)
  const size_t heads = (size_t)dims->n_seqs * dims->h_v;
  const size_t segheads = (size_t)n_seg_total * dims->h_v;
  size_t off = 256;
  p.off_head = off;
  off = align_up(off + heads * 8, 256);
  p.off_seg_bound = off;  // seg_bound (fp32) then seg_w (int32)
  off = align_up(off + segheads * 8, 256);
  if (mode != GDN_CP_OFF) {
    const size_t mat = (size_t)kDim * kDim * 4;
    p.off_R = off;
    off += segheads * mat;
    p.off_Sloc = off;
    off += segheads * mat;
    p.off_Sstart = off;
    off += segheads * mat;
  }
  if (dims->dtype == GDN_BF16) {
    p.off_chunk_map = off;  // chunk index (sequence bases, then 16-byte chunk records), then the chunk
                            // warmup exponents
    off = align_up(off + ((size_t)dims->n_seqs + 1) * 4, 16) + (size_t)n_chunks_total * 16;
    off = align_up(off, 256);
    off = align_up(off + (size_t)n_chunks_total * dims->h_v * 4, 1024);
    p.off_wy = off;
    off += (size_t)n_chunks_total * dims->h_v * kRecBytes;
  }
  p.workspace_bytes = off;
  *out = p;
  return GDN_OK;
}

// The forward.  For the backward (hchunk != null) the WY and output-scan
// kernels also write A^T (wyA) and every output chunk's start state (hchunk),
// in the plan's own mode; *p_out receives the
// problem the kernels run with.  launch = false: only that problem (the
// backward of a forward that already ran with the same arguments).
static gdn_status forward_impl(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               const float* initial_state, const int32_t* cu_dev, void* out, float* final_state,
                               const gdn_dims* dims, const gdn_cp_plan_t* plan, void* workspace,
                               size_t workspace_bytes, void* stream, uint8_t* wyA, uint8_t* hchunk,
                               Problem* p_out, bool launch = true) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (!plan) return GDN_ERR_INVALID_ARG;
  const int64_t T_total = (int64_t)dims->B * dims->T;
  if (plan->n_seqs != dims->n_seqs || plan->T_total != T_total || plan->h_v != dims->h_v ||
      plan->h_qk != dims->h_qk || plan->dtype != dims->dtype)
    return GDN_ERR_INVALID_ARG;
  if (cu_dev && dims->B != 1) return GDN_ERR_INVALID_ARG;
  if (!cu_dev && dims->n_seqs != dims->B) return GDN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < plan->workspace_bytes) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_MISALIGNED;
  if (T_total > 0) {
    if (!q || !k || !v || !g || !beta || !out) return GDN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(g) || !aligned16(beta))
      return GDN_ERR_MISALIGNED;
  }
  if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)) ||
      (cu_dev && (reinterpret_cast<uintptr_t>(cu_dev) & 3u)))
    return GDN_ERR_MISALIGNED;

  int dev = 0;
  st = device_setup(&dev);
  if (st != GDN_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);

  Problem p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.h0 = initial_state;
  p.cu = cu_dev;
  p.out = out;
  p.hT = final_state;
  p.T_row = dims->T;
  p.n_seqs = dims->n_seqs;
  p.h_qk = dims->h_qk;
  p.h_v = dims->h_v;
  p.scale = dims->scale != 0.f ? dims->scale : 1.0f / std::sqrt((float)dims->d_k);
  p.elem_f32 = dims->dtype == GDN_F32;
  p.plan_mode = plan->mode == GDN_CP_OFF ? kModeOff : (plan->mode == GDN_CP_EXACT ? kModeExact : kModeWarmup);
  // a plan in which every sequence is one segment has nothing to combine: it
  // runs without the preprocessing and the combine
  const bool cp = plan->mode != GDN_CP_OFF && plan->n_seg_total > plan->n_seqs;
  if (!cp) p.plan_mode = kModeOff;
  p.wyA = wyA;
  p.hchunk = hchunk;
  p.lambda_q8 = plan->lambda_q8;
  p.warmup_chunks = plan->warmup_chunks;
  p.log_tol = std::log(plan->warmup_tol);
  p.tol_noise = plan->tol_rule == GDN_TOL_NOISE;
  p.n_seg_total = plan->n_seg_total;
  p.status = reinterpret_cast<int*>(ws);
  p.head_mode = reinterpret_cast<int*>(ws + plan->off_head);
  p.head_bound = reinterpret_cast<float*>(ws + plan->off_head + (size_t)dims->n_seqs * dims->h_v * 4);
  p.seg_bound = reinterpret_cast<float*>(ws + plan->off_seg_bound);
  p.seg_w = reinterpret_cast<int*>(ws + plan->off_seg_bound + (size_t)plan->n_seg_total * dims->h_v * 4);
  if (plan->mode != GDN_CP_OFF) {
    p.R = reinterpret_cast<float*>(ws + plan->off_R);
    p.Sloc = reinterpret_cast<float*>(ws + plan->off_Sloc);
    p.Sstart = reinterpret_cast<float*>(ws + plan->off_Sstart);
  }
  p.n_chunks_total = plan->n_chunks_total;
  if (dims->dtype == GDN_BF16) {
    const size_t info_off = align_up(plan->off_chunk_map + ((size_t)dims->n_seqs + 1) * 4, 16);
    p.seq_chunk_base = reinterpret_cast<int32_t*>(ws + plan->off_chunk_map);
    p.chunk_info = reinterpret_cast<int4*>(ws + info_off);
    p.chunk_exp = reinterpret_cast<float*>(ws + align_up(info_off + (size_t)plan->n_chunks_total * 16, 256));
    p.wy = ws + plan->off_wy;
  }
  p.stall_ns = g_debug_stall_ns.load(std::memory_order_relaxed);
  if (!launch) {
    if (p_out) *p_out = p;
    return GDN_OK;
  }

  cudaError_t e = cudaMemsetAsync(ws, 0, 256, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  if (T_total == 0) {
    // No tokens: the final state is the initial state.
    if (final_state) {
      const size_t bytes = (size_t)dims->n_seqs * dims->h_v * kDim * kDim * 4;
      e = initial_state ? cudaMemcpyAsync(final_state, initial_state, bytes, cudaMemcpyDeviceToDevice, cs)
                        : cudaMemsetAsync(final_state, 0, bytes, cs);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return GDN_OK;
  }
  if (dims->dtype == GDN_F32) {
    // fp32 inputs: the recurrence on the CUDA cores, in fp32; a context-parallel
    // plan always combines its segments exactly (no warmup restarts)
    LaunchLog log;
    if (cp) {
      p.plan_mode = kModeExact;
      if ((e = log.before(cs)) != cudaSuccess || (e = launch_f32_prep(p, cs)) != cudaSuccess ||
          (e = log.after("recurrence_f32_prep", cs)) != cudaSuccess)
        return cuda_fail(e);
      if ((e = log.before(cs)) != cudaSuccess || (e = launch_combine(p, g_sm_count[dev], cs)) != cudaSuccess ||
          (e = log.after("combine", cs)) != cudaSuccess)
        return cuda_fail(e);
    }
    if ((e = log.before(cs)) != cudaSuccess ||
        (e = launch_recurrence_f32(p, cs, cp)) != cudaSuccess ||
        (e = log.after("recurrence_f32", cs)) != cudaSuccess)
      return cuda_fail(e);
    return GDN_OK;
  }
  CUtensorMap mq, mk, mv, mo;
  const bool f32 = false;
  if ((st = encode_map(&mq, q, dims->h_qk, T_total, f32)) != GDN_OK) return st;
  if ((st = encode_map(&mk, k, dims->h_qk, T_total, f32)) != GDN_OK) return st;
  if ((st = encode_map(&mv, v, dims->h_v, T_total, f32)) != GDN_OK) return st;
  if ((st = encode_out_map(&mo, out, dims->h_v, T_total)) != GDN_OK) return st;

  // chunk index (varlen) -> WY -> [context parallel: preprocessing -> combine]
  // -> output scan
  LaunchLog log;
  if (cu_dev) {  // varlen chunk index (fixed-length rows compute it)
    if ((e = log.before(cs)) != cudaSuccess || (e = launch_chunk_map(p, cs)) != cudaSuccess ||
        (e = log.after("chunk_map", cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  if ((e = log.before(cs)) != cudaSuccess || (e = launch_wy(p, mq, mk, mv, cs, cu_dev != nullptr)) != cudaSuccess ||
      (e = log.after("wy", cs)) != cudaSuccess)
    return cuda_fail(e);
  if (cp) {
    if ((e = log.before(cs)) != cudaSuccess || (e = launch_scan_prep(p, mq, mk, cs)) != cudaSuccess ||
        (e = log.after("scan_prep", cs)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = log.before(cs)) != cudaSuccess || (e = launch_combine(p, g_sm_count[dev], cs)) != cudaSuccess ||
        (e = log.after("combine", cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  if ((e = log.before(cs)) != cudaSuccess || (e = launch_scan_out(p, mq, mk, mo, plan->n_seg_total, cs)) != cudaSuccess ||
      (e = log.after("scan_out", cs)) != cudaSuccess)
    return cuda_fail(e);
  if (p_out) *p_out = p;
  return GDN_OK;
}

gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* initial_state, const int32_t* cu_dev, void* out, float* final_state,
                         const gdn_dims* dims, const gdn_cp_plan_t* plan, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return forward_impl(q, k, v, g, beta, initial_state, cu_dev, out, final_state, dims, plan, workspace,
                      workspace_bytes, stream, nullptr, nullptr, nullptr);
}

// ---- backward ----
// Sections after the forward's workspace, per (chunk, value head): A^T (8 KB),
// the chunk-start state, T', E and D (32 KB each); then a bf16 o the recompute
// writes and nobody reads.
struct BwdLayout {
  size_t wyA, hchunk, tmat, emat, dstate, out, end;
};
static BwdLayout bwd_layout(const gdn_cp_plan_t* plan) {
  BwdLayout L;
  const size_t ch = (size_t)plan->n_chunks_total * plan->h_v;
  size_t off = align_up(plan->workspace_bytes, 1024);
  L.wyA = off;
  off += ch * 8192;
  L.hchunk = off;
  off += ch * 32768;
  L.tmat = off;
  off += ch * 32768;
  L.emat = off;
  off += ch * 32768;
  L.dstate = off;
  off += ch * 32768;
  L.out = off;
  off = align_up(off + (size_t)plan->T_total * plan->h_v * kDim * 2, 256);
  L.end = off;
  return L;
}

gdn_status gdn_chunk_fwd_train(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               const float* initial_state, const int32_t* cu_dev, void* out, float* final_state,
                               const gdn_dims* dims, const gdn_cp_plan_t* plan, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!plan || !dims) return GDN_ERR_INVALID_ARG;
  if (dims->dtype != GDN_BF16 || plan->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  const BwdLayout L = bwd_layout(plan);
  if (!workspace || workspace_bytes < L.end) return GDN_ERR_WORKSPACE;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  return forward_impl(q, k, v, g, beta, initial_state, cu_dev, out, final_state, dims, plan, workspace,
                      workspace_bytes, stream, ws + L.wyA, ws + L.hchunk, nullptr);
}

gdn_status gdn_bwd_workspace_bytes(const gdn_cp_plan_t* plan, size_t* bytes) {
  if (!plan || !bytes) return GDN_ERR_INVALID_ARG;
  if (plan->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  *bytes = bwd_layout(plan).end;
  return GDN_OK;
}

gdn_status gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* initial_state, const int32_t* cu_dev, const void* d_out,
                         const float* d_final_state, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                         float* d_initial_state, const gdn_dims* dims, const gdn_cp_plan_t* plan, void* workspace,
                         size_t workspace_bytes, int reuse_forward, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (!plan) return GDN_ERR_INVALID_ARG;
  if (dims->dtype != GDN_BF16 || plan->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  const BwdLayout L = bwd_layout(plan);
  if (!workspace || workspace_bytes < L.end) return GDN_ERR_WORKSPACE;
  const int64_t T_total = (int64_t)dims->B * dims->T;
  if (T_total > 0) {
    if (!d_out || !dq || !dk || !dv || !dg || !dbeta) return GDN_ERR_INVALID_ARG;
    if (!aligned16(d_out) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg) ||
        !aligned16(dbeta))
      return GDN_ERR_MISALIGNED;
  }
  if ((d_final_state && !aligned16(d_final_state)) || (d_initial_state && !aligned16(d_initial_state)))
    return GDN_ERR_MISALIGNED;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (T_total == 0) {
    // no tokens: h_T = h0, so the gradient of h0 is that of h_T
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_MISALIGNED;
    int dev = 0;
    if ((st = device_setup(&dev)) != GDN_OK) return st;
    cudaError_t e = cudaMemsetAsync(ws, 0, 256, cs);
    if (e == cudaSuccess && d_initial_state) {
      const size_t bytes = (size_t)dims->n_seqs * dims->h_v * kDim * kDim * 4;
      e = d_final_state ? cudaMemcpyAsync(d_initial_state, d_final_state, bytes, cudaMemcpyDeviceToDevice, cs)
                        : cudaMemsetAsync(d_initial_state, 0, bytes, cs);
    }
    return e == cudaSuccess ? GDN_OK : cuda_fail(e);
  }
  Problem p;
  st = forward_impl(q, k, v, g, beta, initial_state, cu_dev, ws + L.out, nullptr, dims, plan, workspace,
                    workspace_bytes, stream, ws + L.wyA, ws + L.hchunk, &p, reuse_forward == 0);
  if (st != GDN_OK) return st;
  int dev = 0;
  if ((st = device_setup(&dev)) != GDN_OK) return st;
  // The forward above kept the chunk states of the plan's own mode (a warmup
  // restart only where its acceptance rule allows one); the state gradient's
  // chain is always combined exactly.
  if (p.plan_mode != kModeOff) p.plan_mode = kModeExact;
  BwdArgs b;
  b.dout = d_out;
  b.dhT = d_final_state;
  b.dq = dq;
  b.dk = dk;
  b.dv = dv;
  b.dg = dg;
  b.dbeta = dbeta;
  b.dh0 = d_initial_state;
  b.tmat = ws + L.tmat;
  b.emat = ws + L.emat;
  b.dstate = ws + L.dstate;
  LaunchLog log(true);
  cudaError_t e;
  if ((e = log.before(cs)) != cudaSuccess || (e = launch_bwd_pre_tc(p, b, cs)) != cudaSuccess ||
      (e = log.after("bwd_pre", cs)) != cudaSuccess)
    return cuda_fail(e);
  if (p.plan_mode != kModeOff) {
    // context parallel: per segment the transition and the local offset, then
    // the segments' end-state gradients by the combine run backwards
    if ((e = log.before(cs)) != cudaSuccess || (e = launch_bwd_chain_tc(p, b, true, cs)) != cudaSuccess ||
        (e = log.after("bwd_chain_prep", cs)) != cudaSuccess)
      return cuda_fail(e);
    Problem pc = p;
    pc.h0 = d_final_state;
    if ((e = log.before(cs)) != cudaSuccess || (e = launch_combine_bwd(pc, g_sm_count[dev], cs)) != cudaSuccess ||
        (e = log.after("bwd_combine", cs)) != cudaSuccess)
      return cuda_fail(e);
  }
  if ((e = log.before(cs)) != cudaSuccess || (e = launch_bwd_chain_tc(p, b, false, cs)) != cudaSuccess ||
      (e = log.after("bwd_chain", cs)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = log.before(cs)) != cudaSuccess || (e = launch_bwd_local_tc(p, b, cs)) != cudaSuccess ||
      (e = log.after("bwd_local", cs)) != cudaSuccess)
    return cuda_fail(e);
  return GDN_OK;
}

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                           float* state, void* out, const gdn_dims* dims, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (dims->T != 1 || dims->n_seqs != dims->B) return GDN_ERR_INVALID_ARG;
  if (!q || !k || !v || !g || !beta || !state || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(state) ||
      !aligned16(out))
    return GDN_ERR_MISALIGNED;
  if (dims->B > 65535 * 32768) return GDN_ERR_INVALID_ARG;
  DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.state = state;
  a.out = out;
  a.n_seqs = dims->B;
  a.h_qk = dims->h_qk;
  a.h_v = dims->h_v;
  a.scale = dims->scale != 0.f ? dims->scale : 1.0f / std::sqrt((float)dims->d_k);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  LaunchLog log;
  cudaError_t e = log.before(cs);
  if (e == cudaSuccess) e = launch_decode(a, dims->dtype == GDN_F32, cs);
  if (e == cudaSuccess) e = log.after("decode", cs);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e);
}

gdn_status gdn_debug_stall_ns(uint32_t ns) {
  g_debug_stall_ns.store(ns, std::memory_order_relaxed);
  return GDN_OK;
}

gdn_status gdn_set_trace_events(void* const* events, int n_events) {
  if (n_events < 0 || n_events > kMaxTrace) return GDN_ERR_INVALID_ARG;
  if (!events) n_events = 0;
  for (int i = 0; i < n_events; ++i) {
    if (!events[i]) return GDN_ERR_INVALID_ARG;
    g_trace_ev[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  }
  g_trace_n = n_events;
  return GDN_OK;
}

int gdn_trace_last(const char** names, int max_names) {
  if (names)
    for (int i = 0; i < g_last_count && i < max_names; ++i) names[i] = g_last_names[i];
  return g_last_count;
}

gdn_status gdn_get_device_status(const void* workspace, void* stream, int* code, int* detail) {
  if (!workspace || !code) return GDN_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int h[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(h, workspace, sizeof(h), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e);
  *code = h[0];
  if (detail) *detail = h[1];
  return GDN_OK;
}

gdn_status gdn_cp_head_modes(const void* workspace, const gdn_cp_plan_t* plan, int32_t* modes, float* bounds,
                             void* stream) {
  if (!workspace || !plan) return GDN_ERR_INVALID_ARG;
  const size_t heads = (size_t)plan->n_seqs * plan->h_v;
  if (plan->mode == GDN_CP_OFF || plan->dtype == GDN_F32 || plan->n_seg_total <= plan->n_seqs) {
    // no warmup decision taken: no context parallelism, the fp32 path (always
    // exact), or one segment per sequence (nothing to combine or restart)
    for (size_t i = 0; i < heads; ++i) {
      if (modes) modes[i] = plan->mode == GDN_CP_OFF ? GDN_CP_OFF : plan->dtype == GDN_F32 ? GDN_CP_EXACT : plan->mode;
      if (bounds) bounds[i] = -INFINITY;
    }
    return GDN_OK;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* ws = reinterpret_cast<const uint8_t*>(workspace);
  cudaError_t e = cudaSuccess;
  if (modes) e = cudaMemcpyAsync(modes, ws + plan->off_head, heads * 4, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess && bounds)
    e = cudaMemcpyAsync(bounds, ws + plan->off_head + heads * 4, heads * 4, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e);
  return GDN_OK;
}

}  // extern "C"

extern "C" gdn_status gdn_chunk_fwd_static(const void* q, const void* k, const void* v, const float* g,
                                          const float* beta, const float* initial_state,
                                          const int32_t* cu_seqlens_dev, void* out, float* final_state,
                                          const gdn_dims* dims, const gdn_cp_plan_t* plan, void* stream) {
  if (!plan) return GDN_ERR_INVALID_ARG;
  if (plan->workspace_bytes > kStaticWorkspaceBytes) return GDN_ERR_WORKSPACE;
  void* ws = nullptr;
  gdn_status st = static_workspace(&ws);
  if (st != GDN_OK) return st;
  return gdn_chunk_fwd(q, k, v, g, beta, initial_state, cu_seqlens_dev, out, final_state, dims, plan, ws,
                       kStaticWorkspaceBytes, stream);
}

extern "C" gdn_status gdn_get_static_device_status(void* stream, int* code, int* detail) {
  if (!code) return GDN_ERR_INVALID_ARG;
  void* ws = nullptr;
  gdn_status st = static_workspace(&ws);
  if (st != GDN_OK) return st;
  return gdn_get_device_status(ws, stream, code, detail);
}
