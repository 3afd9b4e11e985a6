// The chunk scan on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA runs one chain: a run of 64-token chunks of one (sequence, value
// head), carrying the 128x128 state from chunk to chunk on chip.  The same
// kernel template serves two roles:
//
//   scan_kernel<false>  (fused state scan + output, FlashQLA pages section
//     "TileLang warp-specialised kernels", forward pass: V', S and O per
//     chunk): starts from h0, from the exactly combined segment start state,
//     or from zero a few chunks early (warmup restart, section "AutoCP"),
//     writes o and, for a sequence's last segment, the final state.
//   scan_kernel<true>   (context-parallel preprocessing, section "AutoCP",
//     the correction term M): for an exact-mode (sequence, head) segment,
//     blockIdx.z = 0 runs the segment's transition (the state started at the
//     identity with no value input, giving M^T) and blockIdx.z = 1 its local
//     state (started at zero).
//
// Everything is held in the S orientation (rows = d_v, columns = d_k), so
// that every contraction is an M = 128 tcgen05 MMA with the state rows on
// the TMEM lanes.  Per chunk (C = 64 rows, G = inclusive gate cumsum):
//   D_kq = [K;Q] K^T                       -> L (strict, beta, decay), P (inclusive decay)
//   A    = (I + L)^{-1}                    (fp32, blocked 16x16 forward substitution)
//   W^T  = K^T (A diag(beta gamma))^T,  U^T = V^T (A diag(beta))^T
//   V'^T = U^T - S W^T,  Y = S Q^T
//   O^T  = scale (Y diag(gamma) + V'^T P^T)
//   S    = gamma_C S + V'^T diag(exp(G_last - G)) K
//
// Precision: the MMAs run in fp16 with fp32 accumulation.  q, k and v are
// converted from bf16 to fp16 in shared memory (exact for |x| < 65504); the
// state (kept fp32 in registers), A, W, P and V' are rounded once to fp16
// as operands, which keeps the result within about 4e-3 * RMS of the exact
// recurrence where single bf16 operands reach 3e-2.  A value outside the
// fp16 range is reported through the status word.
//
// Warp roles (448 threads): warps 0-7 hold the state (row = d_v lane, 64
// columns each), do the V' and state/output epilogues, and convert the next
// chunk's tiles to fp16 while they would otherwise wait; warps 8-11 do the
// chunk-local work one chunk ahead (gate cumsum, L and P, the triangular
// solve, the W operand); warp 12 loads tiles and gates (TMA); lane 0 of
// warp 13 issues every MMA as soon as its inputs are ready.
// They hand over through mbarriers whose waits are all bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 448;
constexpr int kChainThreads = 256;
constexpr int kPrepThreads = 128;
constexpr int kProducerWarp = 12;

// ---- shared memory map (bytes from a 1024-byte aligned base) ----
constexpr uint32_t kStageBytes = 49152;  // per stage: K,Q halves (32 KB) + V halves (16 KB)
constexpr uint32_t kStKQ = 0;            // [K d0-63 | Q d0-63 | K d64-127 | Q d64-127], 8 KB each
constexpr uint32_t kStV = 32768;         // [V d0-63 | V d64-127]
constexpr uint32_t kSmS = 98304;         // fp16 state, K-major A: two 64-column halves of 16 KB
constexpr uint32_t kSmVp = 131072;       // fp16 V'^T, K-major A; also the bf16 output tile [64][128]
constexpr uint32_t kSmVd = 147456;       // fp16 V'^T diag(decay to chunk end), K-major A
constexpr uint32_t kSmWn = 163840;       // fp16 -W, MN-major B: rows d_k, 64 chunk rows each
constexpr uint32_t kSmP = 180224;        // fp16 P, K-major B: rows r
constexpr uint32_t kSmA = 188416;        // fp16 A diag(beta gamma) | A diag(beta), MN-major B; solve scratch
constexpr uint32_t kSmF = 204800;        // fp32 [64][68]: L below the diagonal, A^T on and above it
constexpr uint32_t kFStride = 68;
constexpr uint32_t kSmGates = 222208;    // 2 x {G, exp(G), decay, beta, exp(-G)}[64] fp32
constexpr uint32_t kGateFloats = 320;    // floats per gates buffer
constexpr uint32_t kSmRaw = 224768;      // 2 x {g, beta}[64] fp32, as loaded
constexpr uint32_t kSmCtl = 225792;      // barriers, TMEM base, flags
constexpr uint32_t kSmemUse = 226048;
constexpr uint32_t kSmemAlloc = kSmemUse + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory over the per-block limit");

// ---- TMEM columns (512 allocated) ----
constexpr uint32_t kTKQ = 0;    // [K K^T ; Q K^T]         128 x 64
constexpr uint32_t kTW = 64;    // W^T                     128 x 64
constexpr uint32_t kTV = 128;   // U^T then V'^T, 2 bufs   128 x 64 each
constexpr uint32_t kTY = 256;   // S Q^T                   128 x 64
constexpr uint32_t kTO2 = 320;  // V'^T P^T                128 x 64
constexpr uint32_t kTD3 = 384;  // V'^T diag(dec) K        128 x 128

enum InitKind { kInitZero = 0, kInitIdentity = 1, kInitH0 = 2, kInitStart = 3 };

// mbarrier indices
enum Bar {
  kFull0 = 0, kFull1, kEmpty0, kEmpty1, kConv0, kConv1,  // TMA stages; converted stages
  kKqFree, kKqDone, kAReady, kWuDone, kWReady,           // chunk-local pipeline
  kSReady, kVaDone, kVReady, kD3Done, kO2Done, kChainDone0, kChainDone1,  // state pipeline
  kNumBars
};

struct Ctl {
  uint64_t bar[kNumBars];
  uint32_t tmem;
  int abort;
  int range_bad;
  float warp_total[2];
  SegInfo seg;
};
static_assert(sizeof(Ctl) <= kSmemUse - kSmCtl, "control block too large");

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %3, 0;\n bar.red.or.pred po, %1, %2, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}"
      : "=r"(r)
      : "r"(id), "r"(count), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 consecutive floats -> one 16-byte fp16 chunk; flags values outside the fp16 range.
__device__ __forceinline__ void store_f16x8(uint32_t addr, const float* f, bool& bad) {
#pragma unroll
  for (int e = 0; e < 8; ++e) bad |= !(fabsf(f[e]) < 65504.f);
  st_shared_v4(addr, pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
               pack_f16x2(f[6], f[7]));
}

// Instruction descriptor for kind::f16 with fp16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(Ctl* ctl, int b, uint32_t parity) {
  if (mbar_try_wait(&ctl->bar[b], parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(&ctl->bar[b], parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&ctl->abort, 0, 100 + b);
      return false;
    }
  }
}

struct Chain {
  int run_begin, run_end, out_begin;
  int init;
  bool has_u, need_q, write_final;
  int iq;
};

template <bool PREP>
__device__ __forceinline__ bool want_out(const Chain& ch, int i) {
  return !PREP && ch.run_begin + i >= ch.out_begin;
}

// ----------------------------------------------------------------- producer
// Loads each chunk's tiles (TMA) and gates (plain loads) into its stage.
template <bool PREP>
__device__ __noinline__ void producer_role(uint8_t* sm, Ctl* ctl, const Problem& p, const SegInfo& si, const Chain& ch,
                              const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv, int j) {
  const int lane = threadIdx.x & 31;
  const int n = ch.run_end - ch.run_begin;
  float* raw = reinterpret_cast<float*>(sm + kSmRaw);
  auto issue = [&](int i) -> bool {
    const int st = i & 1;
    if (i >= 2 && !wait_bar(ctl, kEmpty0 + st, (uint32_t)(((i - 2) >> 1) & 1))) return false;
    const int64_t t0 = si.bos + (int64_t)(ch.run_begin + i) * kChunk;
    if (lane == 0) {
      uint8_t* stg = sm + st * kStageBytes;
      const uint32_t bytes = 16384u + (ch.need_q ? 16384u : 0u) + (ch.has_u ? 16384u : 0u);
      mbar_arrive_expect_tx(&ctl->bar[kFull0 + st], bytes);
      tma_load_3d(stg + kStKQ, mk, &ctl->bar[kFull0 + st], 0, ch.iq, (int)t0);
      tma_load_3d(stg + kStKQ + 16384, mk, &ctl->bar[kFull0 + st], 64, ch.iq, (int)t0);
      if (ch.need_q) {
        tma_load_3d(stg + kStKQ + 8192, mq, &ctl->bar[kFull0 + st], 0, ch.iq, (int)t0);
        tma_load_3d(stg + kStKQ + 24576, mq, &ctl->bar[kFull0 + st], 64, ch.iq, (int)t0);
      }
      if (ch.has_u) {
        tma_load_3d(stg + kStV, mv, &ctl->bar[kFull0 + st], 0, j, (int)t0);
        tma_load_3d(stg + kStV + 8192, mv, &ctl->bar[kFull0 + st], 64, j, (int)t0);
      }
    }
    // gates of rows 2*lane, 2*lane + 1 (rows past the sequence end act as g = beta = 0)
    float* rg = raw + st * 128;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 2 * lane + e;
      const bool ok = t0 + r < si.eos;
      rg[r] = ok ? p.g[(size_t)(t0 + r) * p.h_v + j] : 0.f;
      rg[64 + r] = ok ? p.beta[(size_t)(t0 + r) * p.h_v + j] : 0.f;
    }
    mbar_arrive(&ctl->bar[kFull0 + st]);
    return true;
  };
  for (int i = 0; i < n; ++i)
    if (!issue(i)) break;
}

// ----------------------------------------------------------------- MMA issuer
template <bool PREP>
__device__ __noinline__ void mma_role(uint8_t* sm, Ctl* ctl, const Chain& ch, uint32_t tmem) {
  const int n = ch.run_end - ch.run_begin;
  const uint32_t sS = smem_u32(sm + kSmS), sVp = smem_u32(sm + kSmVp), sVd = smem_u32(sm + kSmVd);
  const uint32_t sWn = smem_u32(sm + kSmWn), sP = smem_u32(sm + kSmP), sA = smem_u32(sm + kSmA);
  const uint32_t id_kq = idesc_f16(128, 64, false, false);
  const uint32_t id_mn = idesc_f16(128, 64, true, true);
  const uint32_t id_sw = idesc_f16(128, 64, false, true);
  const uint32_t id_y = idesc_f16(128, 64, false, false);
  const uint32_t id_d3 = idesc_f16(128, 128, false, true);

  auto issue_kq = [&](int i) {  // D_kq = [K;Q] K^T
    const uint32_t st = smem_u32(sm + (i & 1) * kStageBytes + kStKQ);
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t off = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
      mma_bf16(tmem + kTKQ, sdesc_sw128(st + off, 16, 1024), sdesc_sw128(st + off, 16, 1024), id_kq, ks > 0);
    }
    mma_commit(&ctl->bar[kKqDone]);
  };
  auto issue_wu = [&](int i) {  // W^T, U^T (into V buffer i & 1)
    const uint32_t st = smem_u32(sm + (i & 1) * kStageBytes);
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem + kTW, sdesc_sw128(st + kStKQ + ks * 2048, 16384, 1024), sdesc_sw128(sA + ks * 2048, 8192, 1024),
               id_mn, ks > 0);
    if (ch.has_u) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kTV + (i & 1) * 64, sdesc_sw128(st + kStV + ks * 2048, 8192, 1024),
                 sdesc_sw128(sA + 8192 + ks * 2048, 8192, 1024), id_mn, ks > 0);
    }
    mma_commit(&ctl->bar[kWuDone]);
  };

  // Four groups per chunk i, issued as soon as their inputs are ready (the
  // readiness probes never block, so one late input holds up nothing else):
  //   KQ(i)   after stage i is converted and the prep has read D_kq(i-1)
  //   WU(i)   after a_ready(i), KQ(i) issued, and V buffer i & 1 released (C(i-2) issued)
  //   A(i)    S W^T and S Q^T, after w_ready(i) and s_ready(i)
  //   C(i)    D3 and O2, after v_ready(i); then the stage of chunk i is released
  if (n <= 0) return;
  int nk = 0, nw = 0, na = 0, nc = 0;
  uint64_t t_last = globaltimer_ns();
  while (nc < n) {
    bool progress = false;
    if (na < n && na <= nc && na < nw && mbar_test_wait(&ctl->bar[kWReady], (uint32_t)(na & 1)) &&
        mbar_test_wait(&ctl->bar[kSReady], (uint32_t)(na & 1))) {
      const int i = na;
      const uint32_t stKQ = smem_u32(sm + (i & 1) * kStageBytes + kStKQ);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // V'^T = U^T - S W^T
        const uint64_t a = sdesc_sw128(sS + (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u, 16, 1024);
        mma_bf16(tmem + kTV + (i & 1) * 64, a, sdesc_sw128(sWn + ks * 2048, 8192, 1024), id_sw,
                 (ch.has_u || ks > 0) ? 1u : 0u);
      }
      mma_commit(&ctl->bar[kVaDone]);
      if (want_out<PREP>(ch, i)) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // Y = S Q^T
          const uint32_t off = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
          mma_bf16(tmem + kTY, sdesc_sw128(sS + off, 16, 1024), sdesc_sw128(stKQ + 8192 + off, 16, 1024), id_y,
                   ks > 0);
        }
      }
      ++na;
      progress = true;
    }
    if (nc < na && mbar_test_wait(&ctl->bar[kVReady], (uint32_t)(nc & 1))) {
      const int i = nc;
      const uint32_t stKQ = smem_u32(sm + (i & 1) * kStageBytes + kStKQ);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)  // D3 = V'^T diag(dec) K
        mma_bf16(tmem + kTD3, sdesc_sw128(sVd + ks * 32, 16, 1024), sdesc_sw128(stKQ + ks * 2048, 16384, 1024),
                 id_d3, ks > 0);
      mma_commit(&ctl->bar[kD3Done]);
      if (want_out<PREP>(ch, i)) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // O2 = V'^T P^T
          mma_bf16(tmem + kTO2, sdesc_sw128(sVp + ks * 32, 16, 1024), sdesc_sw128(sP + ks * 32, 16, 1024), id_y,
                   ks > 0);
      }
      mma_commit(&ctl->bar[kO2Done]);
      mma_commit(&ctl->bar[kEmpty0 + (i & 1)]);
      ++nc;
      progress = true;
    }
    if (nk < n && mbar_test_wait(&ctl->bar[kConv0 + (nk & 1)], (uint32_t)((nk >> 1) & 1)) &&
        (nk == 0 || mbar_test_wait(&ctl->bar[kKqFree], (uint32_t)((nk - 1) & 1)))) {
      issue_kq(nk);
      ++nk;
      progress = true;
    }
    if (nw < nk && nw <= nc + 1 && mbar_test_wait(&ctl->bar[kAReady], (uint32_t)(nw & 1))) {
      issue_wu(nw);
      ++nw;
      progress = true;
    }
    if (progress) {
      t_last = globaltimer_ns();
    } else {
      if (*reinterpret_cast<volatile int*>(&ctl->abort)) return;
      if (globaltimer_ns() - t_last > kWaitLimitNs) {
        atomicCAS(&ctl->abort, 0, 200);
        return;
      }
    }
  }
}

// ----------------------------------------------------------------- chunk-local (prep) warps
// Blocked inverse of the unit lower-triangular (I + L), L strictly lower in F.
// A^T is written on and above the diagonal of F (block (j, i) holds A_ij^T);
// the strict lower part of each diagonal block is cleared after phase 1, so
// the products of phase 2 need no masks.  Threads 64-127, idle in phase 1,
// run side() meanwhile; it returns false on a failed wait.  Returns false,
// in every thread alike, if any thread's side() failed.
template <class Side>
__device__ __forceinline__ bool solve_unit_lower(float* F, float* T, int p, Side&& side) {
  // phase 1: diagonal 16x16 blocks, one column per thread; L rows are
  // broadcast float4 loads, four partial sums per row
  float x[16];
  const int b = p >> 4, c = p & 15;
  if (p < 64) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float* Lr = F + (16 * b + r) * kFStride + 16 * b;
      float a[4] = {(r == c) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s4 = 0; s4 < r; s4 += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(Lr + s4);
        const float* lv = &l4.x;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (s4 + e < r) a[e] = fmaf(-lv[e], x[s4 + e], a[e]);
      }
      x[r] = (a[0] + a[1]) + (a[2] + a[3]);
    }
  }
  const bool side_ok = p < 64 ? true : side();
  if (named_bar_or(2, kPrepThreads, !side_ok)) return false;
  if (p < 64) {  // row c of D_bb^T, zero below the block diagonal
    float* Dt = F + (16 * b + c) * kFStride + 16 * b;
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4)
      *reinterpret_cast<float4*>(Dt + r4) =
          make_float4(r4 + 0 >= c ? x[r4] : 0.f, r4 + 1 >= c ? x[r4 + 1] : 0.f, r4 + 2 >= c ? x[r4 + 2] : 0.f,
                      r4 + 3 >= c ? x[r4 + 3] : 0.f);
  }
  named_bar_sync(2, kPrepThreads);
  // phase 2: off-diagonal blocks A_ij = -D_ii sum_{k=j}^{i-1} L_ik A_kj, by distance i - j
  const int r = p >> 3, c0 = (p & 7) * 2;
#pragma unroll 1
  for (int dist = 1; dist <= 3; ++dist) {
#pragma unroll 1
    for (int bb = 0; bb < 4 - dist; ++bb) {
      const int i = bb + dist, jj = bb;
      float t0[2] = {0.f, 0.f}, t1[2] = {0.f, 0.f};
#pragma unroll 1
      for (int k = jj; k < i; ++k) {
        const float* Lr = F + (16 * i + r) * kFStride + 16 * k;    // L_ik row r
        const float* A0 = F + (16 * jj + c0) * kFStride + 16 * k;  // A_kj column c0 (as A^T row)
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(Lr + m);
          const float4 a0 = *reinterpret_cast<const float4*>(A0 + m);
          const float4 a1 = *reinterpret_cast<const float4*>(A0 + kFStride + m);
          const int h = (m >> 2) & 1;
          t0[h] = fmaf(l4.x, a0.x, fmaf(l4.y, a0.y, fmaf(l4.z, a0.z, fmaf(l4.w, a0.w, t0[h]))));
          t1[h] = fmaf(l4.x, a1.x, fmaf(l4.y, a1.y, fmaf(l4.z, a1.z, fmaf(l4.w, a1.w, t1[h]))));
        }
      }
      *reinterpret_cast<float2*>(T + (bb * 16 + r) * 16 + c0) = make_float2(t0[0] + t0[1], t1[0] + t1[1]);
    }
    named_bar_sync(2, kPrepThreads);
#pragma unroll 1
    for (int bb = 0; bb < 4 - dist; ++bb) {
      const int i = bb + dist, jj = bb;
      // A_ij[r][c] = -sum_m D_ii[r][m] T[m][c],  D_ii[r][m] = F[16i + m][16i + r] (zero for m > r)
      float a0[2] = {0.f, 0.f}, a1[2] = {0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float d = F[(16 * i + m) * kFStride + 16 * i + r];
        const float2 t = *reinterpret_cast<const float2*>(T + (bb * 16 + m) * 16 + c0);
        a0[m & 1] = fmaf(d, t.x, a0[m & 1]);
        a1[m & 1] = fmaf(d, t.y, a1[m & 1]);
      }
      F[(16 * jj + c0) * kFStride + 16 * i + r] = -(a0[0] + a0[1]);  // A_ij^T[c0][r]
      F[(16 * jj + c0 + 1) * kFStride + 16 * i + r] = -(a1[0] + a1[1]);
    }
    named_bar_sync(2, kPrepThreads);
  }
  return true;
}

template <bool PREP>
__device__ __noinline__ void prep_role(uint8_t* sm, Ctl* ctl, const Chain& ch, uint32_t tmem) {
  const int p = threadIdx.x - kChainThreads;  // 0..127 = TMEM lane
  const int pw = p >> 5, lane = p & 31;
  const int n = ch.run_end - ch.run_begin;
  const uint32_t lane_base = (uint32_t)(pw * 32) << 16;
  float* F = reinterpret_cast<float*>(sm + kSmF);
  float* T = reinterpret_cast<float*>(sm + kSmA);
  const uint32_t sA = smem_u32(sm + kSmA), sWn = smem_u32(sm + kSmWn), sP = smem_u32(sm + kSmP);
  bool bad = false;
  for (int i = 0; i < n; ++i) {
    const uint32_t par = (uint32_t)(i & 1);
    const int st = i & 1;
    const bool out = want_out<PREP>(ch, i);
    // (a) the producer has loaded the gates and converted the tiles of chunk i
    if (!wait_bar(ctl, kConv0 + st, (uint32_t)((i >> 1) & 1))) break;
    // (b) gate cumsum into gates[i & 1]; chain(i - 2) must be done with that buffer
    if (i >= 2 && !wait_bar(ctl, kChainDone0 + (i & 1), (uint32_t)(((i - 2) >> 1) & 1))) break;
    float* gts = reinterpret_cast<float*>(sm + kSmGates) + (i & 1) * kGateFloats;
    float* sG = gts;
    float* sGam = gts + 64;
    float* sDec = gts + 128;
    float* sBeta = gts + 192;
    float* sEp = sGam;      // exp(G)
    float* sEm = gts + 256;  // exp(-G)
    const float* rg = reinterpret_cast<const float*>(sm + kSmRaw) + st * 128;
    if (p < 64) {
      float x = rg[p];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
      }
      if (lane == 31) ctl->warp_total[pw] = x;
      named_bar_sync(3, 64);
      if (pw == 1) x += ctl->warp_total[0];
      sG[p] = x;
      sBeta[p] = rg[64 + p];
      named_bar_sync(3, 64);
      sGam[p] = __expf(x);
      sDec[p] = __expf(sG[63] - x);
      sEm[p] = __expf(-x);
    }
    named_bar_sync(2, kPrepThreads);
    // exp(G_r - G_s) = exp(G_r) exp(-G_s) when no factor can overflow
    const bool factored = fabsf(sG[0]) < 80.f && fabsf(sG[63]) < 80.f;
    // (c) L (rows 0-63 of D_kq) into F
    if (!wait_bar(ctl, kKqDone, par)) break;
    tc_fence_after();
    if (p < 64) {
      uint32_t rk[4][16];  // this lane's row of D_kq, loaded in one batch
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) tmem_ld16(tmem + lane_base + kTKQ + g4 * 16, rk[g4]);
      tmem_ld_wait(rk[0], rk[1]);
      tmem_ld_wait(rk[2], rk[3]);
      const int r = p;
      const float br = sBeta[r], Gr = sG[r], brE = sBeta[r] * sEp[r];
      float* Lr = F + r * kFStride;
      if (factored) {
#pragma unroll
        for (int s4 = 0; s4 < 64; s4 += 4) {
          const float4 em = *reinterpret_cast<const float4*>(sEm + s4);
          const float* emv = &em.x;
          float4 o4;
          float* o = &o4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = s4 + e;
            o[e] = (s < r) ? brE * __uint_as_float(rk[s >> 4][s & 15]) * emv[e] : 0.f;
          }
          *reinterpret_cast<float4*>(Lr + s4) = o4;
        }
      } else {
#pragma unroll
        for (int s4 = 0; s4 < 64; s4 += 4) {
          float4 o4;
          float* o = &o4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = s4 + e;
            o[e] = (s < r) ? br * __uint_as_float(rk[s >> 4][s & 15]) * __expf(Gr - sG[s]) : 0.f;
          }
          *reinterpret_cast<float4*>(Lr + s4) = o4;
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[kKqFree]);  // rows 0-63 of D_kq have been read
    }
    named_bar_sync(2, kPrepThreads);
    // (d) A = (I + L)^{-1}.  Meanwhile threads 64-127 build P (rows 64-127 of
    //     D_kq) into its operand, once the O2 of the previous chunk has
    //     consumed the old one.
    auto build_p = [&]() -> bool {
      if (out) {
        if (i >= 1 && !wait_bar(ctl, kO2Done, par ^ 1u)) return false;
        uint32_t rk[4][16];
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) tmem_ld16(tmem + lane_base + kTKQ + g4 * 16, rk[g4]);
        tmem_ld_wait(rk[0], rk[1]);
        tmem_ld_wait(rk[2], rk[3]);
        const int r = p - 64;
        const float Gr = sG[r], Er = sEp[r];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float f[8];
          if (factored) {
            const float4 e0 = *reinterpret_cast<const float4*>(sEm + 8 * q);
            const float4 e1 = *reinterpret_cast<const float4*>(sEm + 8 * q + 4);
            const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int s = 8 * q + e;
              f[e] = s <= r ? __uint_as_float(rk[s >> 4][s & 15]) * Er * ev[e] : 0.f;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int s = 8 * q + e;
              f[e] = s <= r ? __uint_as_float(rk[s >> 4][s & 15]) * __expf(Gr - sG[s]) : 0.f;
            }
          }
          store_f16x8(sP + sw128_offset(r, q), f, bad);
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[kKqFree]);  // rows 64-127 of D_kq have been read
      return true;
    };
    if (!solve_unit_lower(F, T, p, build_p)) break;
    {
      const int s = p & 63, mat = p >> 6;
      const float sc = mat == 0 ? sBeta[s] * sGam[s] : sBeta[s];
      const float* At = F + s * kFStride;
      if (mat == 0 || ch.has_u) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 lo4 = *reinterpret_cast<const float4*>(At + 8 * q);
          const float4 hi4 = *reinterpret_cast<const float4*>(At + 8 * q + 4);
          const float v[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = (8 * q + e >= s) ? v[e] * sc : 0.f;
          store_f16x8(sA + mat * 8192 + sw128_offset(s, q), f, bad);
        }
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[kAReady]);
    // (e) -W operand (its proxy fence also covers the P stores).  Waiting
    //     for the chain's V' hand-over of the previous chunk both frees the
    //     old operand (its S W^T is complete) and keeps this w_ready arrival
    //     from running two phases ahead of the chain.
    if (!wait_bar(ctl, kWuDone, par)) break;
    if (i >= 1 && !wait_bar(ctl, kVReady, par ^ 1u)) break;
    tc_fence_after();
#pragma unroll
    for (int g8 = 0; g8 < 2; ++g8) {
      uint32_t ra[16], rb[16];
      tmem_ld16(tmem + lane_base + kTW + g8 * 32, ra);
      tmem_ld16(tmem + lane_base + kTW + g8 * 32 + 16, rb);
      tmem_ld_wait(ra, rb);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = -__uint_as_float(q < 2 ? ra[8 * q + e] : rb[8 * (q - 2) + e]);
        store_f16x8(sWn + sw128_offset(p, 4 * g8 + q), f, bad);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&ctl->bar[kWReady]);
  }
  if (bad) atomicExch(&ctl->range_bad, 1);
}

// ----------------------------------------------------------------- state (chain) warps
template <bool PREP>
__device__ __noinline__ void chain_role(uint8_t* sm, Ctl* ctl, const Problem& p, const SegInfo& si, const Chain& ch,
                           uint32_t tmem, int j, int chain) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127, half = tid >> 7;
  // The state lives only in these warps' registers (loading it outside this
  // role would keep 64 registers busy in every other role too).
  float S[64];
  {
    const size_t head_off = (size_t)(si.n * p.h_v + j) * kDim * kDim;
    if (ch.init == kInitH0) {
#pragma unroll
      for (int e = 0; e < 64; ++e) S[e] = p.h0[head_off + (size_t)(half * 64 + e) * kDim + row];
    } else if (ch.init == kInitStart) {
      const float4* src = reinterpret_cast<const float4*>(
          p.Sstart + ((size_t)(si.seg_base + si.s) * p.h_v + j) * kDim * kDim + (size_t)row * kDim + half * 64);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float4 v4 = src[e];
        S[4 * e] = v4.x;
        S[4 * e + 1] = v4.y;
        S[4 * e + 2] = v4.z;
        S[4 * e + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 64; ++e) S[e] = (ch.init == kInitIdentity && half * 64 + e == row) ? 1.f : 0.f;
    }
  }
  int n = ch.run_end - ch.run_begin;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t sS = smem_u32(sm + kSmS), sVp = smem_u32(sm + kSmVp), sVd = smem_u32(sm + kSmVd);
  uint16_t* sO = reinterpret_cast<uint16_t*>(sm + kSmVp);
  bool bad = false;
  auto store_state = [&]() {
#pragma unroll
    for (int q = 0; q < 8; ++q) store_f16x8(sS + half * 16384 + sw128_offset(row, q), &S[8 * q], bad);
  };
  // bf16 -> fp16 in place, for every tile the MMAs of chunk c read
  auto convert_stage = [&](int c) -> bool {
    const int st = c & 1;
    if (!wait_bar(ctl, kFull0 + st, (uint32_t)((c >> 1) & 1))) return false;
    uint4* base = reinterpret_cast<uint4*>(sm + st * kStageBytes);
    auto conv_range = [&](uint4* b4, int nvec) {  // nvec: a multiple of kChainThreads
#pragma unroll 1
      for (int v0 = tid; v0 < nvec; v0 += 2 * kChainThreads) {
        const bool two = v0 + kChainThreads < nvec;
        uint4 u0 = b4[v0], u1 = two ? b4[v0 + kChainThreads] : u0;
        uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
          bad |= !(fabsf(lo) < 65504.f) || !(fabsf(hi) < 65504.f);
          w[e] = pack_f16x2(lo, hi);
        }
        b4[v0] = make_uint4(w[0], w[1], w[2], w[3]);
        if (two) b4[v0 + kChainThreads] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    };
    if (ch.need_q) {
      conv_range(base, 2048);  // K|Q|K|Q
    } else {
      conv_range(base, 512);         // K d0-63
      conv_range(base + 1024, 512);  // K d64-127
    }
    if (ch.has_u) conv_range(base + 2048, 1024);  // V
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[kConv0 + st]);
    return true;
  };
  store_state();
  fence_proxy_async_smem();
  mbar_arrive(&ctl->bar[kSReady]);
  int done = 0;
  if (n > 0 && !convert_stage(0)) n = -1;
  for (int i = 0; i < n; ++i) {
    if (i + 1 < n && !convert_stage(i + 1)) break;
    const uint32_t par = (uint32_t)(i & 1);
    const bool out = want_out<PREP>(ch, i);
    const int64_t t0 = si.bos + (int64_t)(ch.run_begin + i) * kChunk;
    const int cv = (int)min((int64_t)kChunk, si.eos - t0);
    const float* gts = reinterpret_cast<const float*>(sm + kSmGates) + (i & 1) * kGateFloats;
    // the prep warps' generic writes (gates) are published by their w_ready arrival
    if (!wait_bar(ctl, kWReady, par) || !wait_bar(ctl, kVaDone, par)) break;
    tc_fence_after();
    // V' operands: plain (for O) and decayed to the chunk end (for S)
    {
      uint32_t va[16], vb[16];
      tmem_ld16(tmem + lane_base + kTV + (i & 1) * 64 + half * 32, va);
      tmem_ld16(tmem + lane_base + kTV + (i & 1) * 64 + half * 32 + 16, vb);
      tmem_ld_wait(va, vb);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int g2 = q4 >> 1, q = q4 & 1;
        const float* f = reinterpret_cast<const float*>(g2 == 0 ? &va[q * 8] : &vb[q * 8]);
        const float* d = gts + 128 + half * 32 + g2 * 16 + q * 8;
        const uint32_t off = sw128_offset(row, half * 4 + g2 * 2 + q);
        if (out) store_f16x8(sVp + off, f, bad);
        float fd[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) fd[e] = f[e] * d[e];
        store_f16x8(sVd + off, fd, bad);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&ctl->bar[kVReady]);
    // S = gamma_C S + D3
    if (!wait_bar(ctl, kD3Done, par)) break;
    tc_fence_after();
    {
      const float gC = __expf(gts[63]);
#pragma unroll
      for (int g8 = 0; g8 < 2; ++g8) {
        uint32_t ra[16], rb[16];
        tmem_ld16(tmem + lane_base + kTD3 + half * 64 + g8 * 32, ra);
        tmem_ld16(tmem + lane_base + kTD3 + half * 64 + g8 * 32 + 16, rb);
        tmem_ld_wait(ra, rb);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          S[g8 * 32 + e] = fmaf(gC, S[g8 * 32 + e], __uint_as_float(ra[e]));
          S[g8 * 32 + 16 + e] = fmaf(gC, S[g8 * 32 + 16 + e], __uint_as_float(rb[e]));
        }
      }
    }
    store_state();
    if (!wait_bar(ctl, kO2Done, par)) break;
    tc_fence_after();
    if (out) {  // stage this thread's 32 outputs (sO aliases V', which O2 has consumed)
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        uint32_t yq[16], o2[16];
        tmem_ld16(tmem + lane_base + kTY + half * 32 + g2 * 16, yq);
        tmem_ld16(tmem + lane_base + kTO2 + half * 32 + g2 * 16, o2);
        tmem_ld_wait(yq, o2);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = half * 32 + g2 * 16 + e;
          const float o = p.scale * fmaf(gts[64 + c], __uint_as_float(yq[e]), __uint_as_float(o2[e]));
          sO[c * kDim + row] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&ctl->bar[kSReady]);
    if (out) {
      named_bar_sync(4, kChainThreads);
      __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = tid + q * kChainThreads;
        const int r = idx >> 4, c16 = idx & 15;
        if (r < cv) {
          const uint4 val = *reinterpret_cast<const uint4*>(sO + r * kDim + c16 * 8);
          *reinterpret_cast<uint4*>(outp + ((size_t)(t0 + r) * p.h_v + j) * kDim + c16 * 8) = val;
        }
      }
      named_bar_sync(4, kChainThreads);
    }
    mbar_arrive(&ctl->bar[kChainDone0 + (i & 1)]);
    done = i + 1;
  }
  if (bad) atomicExch(&ctl->range_bad, 1);
  if (done < n || *reinterpret_cast<volatile int*>(&ctl->abort)) return;  // no results from an aborted chain
  if (PREP) {
    float* dst = (chain == 0 ? p.R : p.Sloc) + ((size_t)(si.seg_base + si.s) * p.h_v + j) * kDim * kDim +
                 (size_t)row * kDim + half * 64;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      reinterpret_cast<float4*>(dst)[e] = make_float4(S[4 * e], S[4 * e + 1], S[4 * e + 2], S[4 * e + 3]);
  } else if (ch.write_final) {
    float* dst = p.hT + (size_t)(si.n * p.h_v + j) * kDim * kDim;
#pragma unroll
    for (int e = 0; e < 64; ++e) dst[(size_t)(half * 64 + e) * kDim + row] = S[e];
  }
}

template <bool PREP>
__global__ void __launch_bounds__(kThreads, 1)
    scan_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + kSmCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.y;
  const int chain = PREP ? (int)blockIdx.z : 0;

  // ---- which chain this CTA runs ----
  if (warp == 0) {
    SegInfo si;
    const bool ok = locate_segment(p, blockIdx.x, si);
    if (lane == 0) {
      if (!ok) si.n = -1;
      ctl->seg = si;
    }
  }
  __syncthreads();
  const SegInfo si = ctl->seg;
  if (si.n < 0) {
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return;
  }
  if (blockIdx.x == gridDim.x - 1 && !(si.n == p.n_seqs - 1 && si.s == si.n_seg - 1)) {
    if (tid == 0 && blockIdx.y == 0 && blockIdx.z == 0) report(p.status, kDevCheck, kDetSegMismatch);
  }
  Chain ch;
  ch.run_begin = si.cb;
  ch.run_end = si.ce;
  ch.out_begin = si.cb;
  ch.init = kInitZero;
  ch.has_u = true;
  ch.write_final = false;
  if (PREP) {
    if (head_mode_of(p, si, j) != kModeExact || si.s == si.n_seg - 1) return;
    if (chain == 0 && si.s == 0 && p.h0 == nullptr) return;  // M of segment 0 unused for a zero start
    ch.init = chain == 0 ? kInitIdentity : kInitZero;
    ch.has_u = chain == 1;
  } else {
    const int mode = p.plan_mode == kModeOff ? kModeOff : p.head_mode[si.n * p.h_v + j];
    if (si.s == 0) {
      ch.init = kInitH0;
    } else if (mode == kModeWarmup) {
      const int w = p.seg_w[(size_t)(si.seg_base + si.s) * p.h_v + j];
      const int ws = si.cb - w;
      if (ws <= 0) {
        ch.run_begin = 0;
        ch.init = kInitH0;
      } else {
        ch.run_begin = ws;
        ch.init = kInitZero;
      }
    } else {
      ch.init = kInitStart;
    }
    ch.write_final = (p.hT != nullptr) && si.s == si.n_seg - 1;
  }
  if (ch.init == kInitH0 && p.h0 == nullptr) ch.init = kInitZero;
  ch.need_q = !PREP;
  ch.iq = (int)(((int64_t)j * p.h_qk) / p.h_v);

  // ---- set-up ----
  if (tid == 0) {
    const int counts[kNumBars] = {33, 33, 1, 1, kChainThreads, kChainThreads, kPrepThreads, 1, kPrepThreads, 1,
                                  kPrepThreads,
                                  kChainThreads, 1, kChainThreads, 1, 1, kChainThreads, kChainThreads};
    for (int b = 0; b < kNumBars; ++b) mbar_init(&ctl->bar[b], counts[b]);
    ctl->abort = 0;
    ctl->range_bad = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&mk);
    if (ch.need_q) tma_prefetch_desc(&mq);
    if (ch.has_u) tma_prefetch_desc(&mv);
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  if (warp < 8) {
    chain_role<PREP>(sm, ctl, p, si, ch, tmem, j, chain);
  } else if (warp < 12) {
    prep_role<PREP>(sm, ctl, ch, tmem);
  } else if (warp == kProducerWarp) {
    producer_role<PREP>(sm, ctl, p, si, ch, &mq, &mk, &mv, j);
  } else if (lane == 0) {
    mma_role<PREP>(sm, ctl, ch, tmem);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  const int abort_code = ctl->abort;
  if (abort_code) {
    if (tid == 0) report(p.status, kDevTimeout, abort_code);
    // let copies and MMAs already in flight land before the memory is released
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  } else if (tid == 0 && ctl->range_bad) {
    report(p.status, kDevCheck, kDetFp16Range);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t scan_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
}

cudaError_t launch_scan_prep(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                             cudaStream_t st) {
  dim3 grid(p.n_seg_total, p.h_v, 2);
  scan_kernel<true><<<grid, kThreads, kSmemAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

cudaError_t launch_scan_out(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            int grid_x, cudaStream_t st) {
  dim3 grid(grid_x, p.h_v, 1);
  scan_kernel<false><<<grid, kThreads, kSmemAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace gdn
