// The chunk scan on the 5th-generation tensor cores (tcgen05 + TMEM + bulk
// copies): the part of the forward that carries the state from chunk to
// chunk.
//
// One CTA runs one chain: a run of 64-token chunks of one (sequence, value
// head), with the 128x128 state held on chip.  The same kernel template
// serves two roles:
//
//   scan_kernel<false>  (fused state scan + output, FlashQLA pages section
//     "TileLang warp-specialised kernels", forward pass: V', S and O per
//     chunk): starts from h0, from the exactly combined segment start state,
//     or from zero a few chunks early (warmup restart, section "AutoCP"),
//     writes o and, for a sequence's last segment, the final state.
//   scan_kernel<true>   (context-parallel preprocessing, section "AutoCP",
//     the correction term M): for an exact-mode (sequence, head) segment,
//     chain 0 runs the segment's transition (the state started at the
//     identity with no value input, giving M^T) and chain 1 its local
//     state (started at zero).
//
// Everything chunk-local (the gate cumsum, the WY form, P) comes from the
// WY kernel's records as ready-made operand tiles; K and Q come straight
// from the inputs (bf16, rounded to fp16 in shared memory, K scaled by the
// decay to the chunk end on the way).  Here, in the S orientation (rows =
// d_v, columns = d_k), per chunk:
//   V'^T = U^T - S W^T        (U^T added by the state warps)
//   S    = gamma_C S + V'^T (diag(exp(G_last - G)) K)
//   O^T  = scale (S (diag(gamma) Q)^T + V'^T P^T)   (one accumulator)
// All are M = 128 tcgen05 MMAs (fp16 operands, fp32 accumulation in TMEM).
// The state is kept fp32 in registers and rounded to fp16 once per chunk
// into TMEM (two buffers), where the MMAs read it as their A operand; V'
// likewise (two buffers of its fp16 copy beside its fp32 accumulator).  A
// value outside the fp16 range is reported through the status word.
//
// Warp roles (512 threads, four warpgroups): warps 0-7 hold the state (row =
// d_v lane, 64 columns each) and run the V' and state epilogues, the
// critical path from one chunk to the next; warps 8-11 read the output
// accumulator (Y + O2) and stage the chunk's outputs in shared memory and
// store them (TMA) while the state warps go on to the next chunk, and round
// the bf16 Q tiles (times gamma) to fp16 in place two chunks ahead; warp 12
// loads each chunk's record (bulk copies) and its K and Q tiles (TMA); lane
// 0 of warp 13 issues every MMA, in the order A, Y, D3, O2; warps 14-15
// round the bf16 K tiles (times the decay to the chunk end) to fp16 in
// place ahead of the D3 that reads them.
// The state warpgroups raise their register limit to 168 (the state takes
// 64 per thread) and the others lower theirs to 88, within the 128 per
// thread the block is launched with.  The roles hand over through
// mbarriers whose waits are all bounded; every decision to stop after a wait
// gave up is taken alike by all threads that share a warp-collective
// instruction or a named barrier, so a timeout ends in the kernel's own
// exit path.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdn_dev.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 512;
constexpr int kChainThreads = 256;
constexpr int kOutWarp = 8;        // warps 8-11
constexpr int kOutThreads = 128;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kConvertWarp = 14;   // warps 14-15
constexpr int kConvertWarps = 2;
constexpr uint32_t kChainRegs = 168, kOtherRegs = 88;
constexpr int kOutBarrier = 1;     // named barrier of the output warps
static_assert(2 * 128 * kChainRegs + 2 * 128 * kOtherRegs <= 65536 && kThreads * 128 == 65536,
              "register split over the launch's 128 per thread");

// ---- shared memory map (bytes from a 1024-byte aligned base) ----
// Three rings, each slot released as soon as its last reader has run: ring
// A (-W, U^T; two slots) and ring K (two slots) after D3(i), ring B (Q, P;
// three slots) after O2(i).  So the loads of chunk i + 2 (rings A, K) and
// i + 3 (ring B) start as early as they can.
constexpr uint32_t kRingA = 0;            // 2 slots of 32 KB:
constexpr uint32_t kSlotA = 32768;
constexpr uint32_t kAWn = 0;              //   fp16 -W, MN-major B: rows d_k
constexpr uint32_t kAU = 16384;           //   fp16 U^T, K-major A: rows d_v
constexpr uint32_t kRingK = 2 * kSlotA;   // 2 slots of 16 KB: [K d0-63 | K d64-127], 8 KB each, bf16 as
constexpr uint32_t kSlotK = 16384;        //   loaded, then fp16 in place (K times dec)
constexpr uint32_t kRingB = kRingK + 2 * kSlotK;  // 3 slots of 24 KB (chunk i in slot i % 3):
constexpr uint32_t kSlotB = 24576;
constexpr uint32_t kBQ = 0;               //   [Q d0-63 | Q d64-127], 8 KB each, bf16 then fp16 in place
constexpr uint32_t kBP = 16384;           //   fp16 P, K-major B: rows r
constexpr uint32_t kSmO = kRingB + 3 * kSlotB;  // bf16 o of one chunk, [64 tokens][128 d_v] rows of 256 bytes
constexpr uint32_t kSmG = kSmO + 16384;     // 4 slots (chunk i in slot i & 3): fp32 exp(G) [64], exp(G_63 - G) [64]
constexpr uint32_t kSmCtl = kSmG + 4 * 512; // barriers, TMEM base, flags
constexpr uint32_t kSmemUse = kSmCtl + 512;
constexpr uint32_t kSmemAlloc = kSmemUse + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory over the per-block limit");
static_assert(kSlotB % 1024 == 0 && kBP + 8192 <= kSlotB, "ring layout");

// ---- TMEM columns (512 allocated) ----
constexpr uint32_t kTV = 0;     // -S W^T                      128 x 64
constexpr uint32_t kTV16 = 64;  // fp16 V'^T, 2 buffers: 128 x 64 packed in 32 columns each
constexpr uint32_t kTD3 = 128;  // V'^T diag(dec) K            128 x 128
constexpr uint32_t kTO = 256;   // S (gamma Q)^T + V'^T P^T, 2 buffers   128 x 64 each
constexpr uint32_t kTS = 384;   // fp16 state, 2 buffers: 128 x 128 packed in 64 columns each

enum InitKind { kInitZero = 0, kInitIdentity = 1, kInitH0 = 2, kInitStart = 3 };

// mbarrier indices
enum Bar {
  kFull0 = 0, kFull1, kEmpty0, kEmpty1,    // ring A slots (-W, U^T): loaded / released
  kGates0, kGates1, kGates2, kGates3,      // gates ring slots (loaded)
  kVaDone, kVReady, kD3Done, kSReady,      // state pipeline
  kYoDone0, kYoDone1, kYoFree0, kYoFree1,  // output epilogue (two O buffers)
  kKqFull0, kKqFull1,                      // ring K slots loaded (bf16)
  kKReady0, kKReady1, kQReady0, kQReady1,  // K, then Q, rounded to fp16
  kEmptyB0, kEmptyB1, kEmptyB2,            // ring B slots released
  kQFull0, kQFull1, kQFull2,               // ring B slots loaded (Q bf16, P)
  kEmptyK0, kEmptyK1,                      // ring K slots released
  kNumBars
};

struct Ctl {
  uint64_t bar[kNumBars];
  uint32_t tmem;
  int abort;
  int range_bad;
  int skip;
  SegInfo seg;
};
static_assert(sizeof(Ctl) <= kSmemUse - kSmCtl, "control block too large");

__device__ __forceinline__ bool wait_bar(Ctl* ctl, int b, uint32_t parity) {
  return wait_phase(&ctl->bar[b], parity, &ctl->abort, 100 + b);
}

// A warp's outcome of a wait: true only if every lane's wait succeeded, so
// the warp stays converged for its warp-collective instructions.
__device__ __forceinline__ bool warp_ok(bool ok) { return __all_sync(0xffffffffu, ok); }

// Bounded wait that polls without suspending: the single MMA-issuing thread
// uses it so that it reacts to a hand-over as soon as the phase completes.
__device__ __forceinline__ bool spin_bar(Ctl* ctl, int b, uint32_t parity) {
  if (mbar_test_wait(&ctl->bar[b], parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int k = 0; k < 64; ++k)
      if (mbar_test_wait(&ctl->bar[b], parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&ctl->abort, 0, 100 + b);
      return false;
    }
  }
}

struct Chain {
  int64_t bos;  // the sequence's first token
  int run_begin, run_end, out_begin;
  int init;
  bool has_u, write_final;
  int iq;
  int chunk0;  // global index of the sequence's first chunk
};

template <bool PREP>
__device__ __forceinline__ bool want_out(const Chain& ch, int i) {
  return !PREP && ch.run_begin + i >= ch.out_begin;
}

// ----------------------------------------------------------------- producer
// Loads each chunk's K (ring K) and Q (ring B) tiles by TMA, 64 tokens x 64
// dims per box (rows past the end of the input read as zero), its P (ring
// B) and gates by bulk copies, and, a chunk ahead, its ring A tiles (-W,
// U^T; bulk copies).  The waits come in the order the slots are released:
// ring B of chunk i - 3 (after its O2), ring K of chunk i - 2 (after its
// D3), ring A of chunk i - 1 (after its D3).
template <bool PREP>
__device__ __forceinline__ void producer_role(uint8_t* sm, Ctl* ctl, const Problem& p, const Chain& ch, int j,
                                           const CUtensorMap* mq, const CUtensorMap* mk) {
  if ((threadIdx.x & 31) != 0) return;
  const int n = ch.run_end - ch.run_begin;
  auto rec_of = [&](int i) { return p.wy + (((size_t)ch.chunk0 + ch.run_begin + i) * p.h_v + j) * kRecBytes; };
  auto load_a = [&](int i) {
    uint8_t* slot = sm + kRingA + (i & 1) * kSlotA;
    uint64_t* bar = &ctl->bar[kFull0 + (i & 1)];
    mbar_arrive_expect_tx(bar, ch.has_u ? 32768u : 16384u);
    bulk_load(slot + kAWn, rec_of(i) + kRecWn, 16384u, bar);
    if (ch.has_u) bulk_load(slot + kAU, rec_of(i) + kRecU, 16384u, bar);
  };
  if (n > 0) load_a(0);
  for (int i = 0; i < n; ++i) {
    const int t0 = (int)(ch.bos + (int64_t)(ch.run_begin + i) * kChunk);
    // ring B (Q and P, only where the chunk's output is written) and the gates
    const int sb = i % 3;
    if (i >= 3 && !wait_bar(ctl, kEmptyB0 + sb, (uint32_t)(((i - 3) / 3) & 1))) return;
    uint8_t* bslot = sm + kRingB + sb * kSlotB;
    uint64_t* qbar = &ctl->bar[kQFull0 + sb];
    if (want_out<PREP>(ch, i)) {
      mbar_arrive_expect_tx(qbar, 24576u);
      tma_load_3d(bslot + kBQ, mq, qbar, 0, ch.iq, t0);
      tma_load_3d(bslot + kBQ + 8192, mq, qbar, 64, ch.iq, t0);
      bulk_load(bslot + kBP, rec_of(i) + kRecP, 8192u, qbar);
    } else {
      mbar_arrive(qbar);  // nothing to load: the phase completes, keeping the slot's phases per chunk
    }
    // The gates go to ring slot i & 3.  Its readers of chunk i - 4 are done:
    // the converter before k_ready(i - 4), the state warps in the V' epilogue
    // of chunk i - 4 (before v_ready(i - 4)), the output warps before
    // q_ready(i - 4), all waited for before O2(i - 3) was issued, and ring B
    // of chunk i - 3 is released after O2(i - 3).
    uint64_t* gbar = &ctl->bar[kGates0 + (i & 3)];
    mbar_arrive_expect_tx(gbar, 512u);
    bulk_load(sm + kSmG + (i & 3) * 512, rec_of(i) + kRecGam, 512u, gbar);
    // ring K
    if (i >= 2 && !wait_bar(ctl, kEmptyK0 + (i & 1), (uint32_t)(((i - 2) >> 1) & 1))) return;
    uint8_t* kslot = sm + kRingK + (i & 1) * kSlotK;
    uint64_t* kbar = &ctl->bar[kKqFull0 + (i & 1)];
    mbar_arrive_expect_tx(kbar, 16384u);
    tma_load_3d(kslot, mk, kbar, 0, ch.iq, t0);
    tma_load_3d(kslot + 8192, mk, kbar, 64, ch.iq, t0);
    if (i + 1 < n) {
      if (i + 1 >= 2 && !wait_bar(ctl, kEmpty0 + ((i + 1) & 1), (uint32_t)(((i - 1) >> 1) & 1))) return;
      load_a(i + 1);
    }
  }
}

// ----------------------------------------------------------------- K and Q rounding
// bf16 tiles are rounded to fp16 in place (same byte layout): the state's
// fp16 operand copy keeps 11 significant bits, so the MMAs with K and Q run
// in fp16.  K is multiplied by dec = exp(G_63 - G) of its row on the way (so
// D3 needs only the plain V'); the converter warps do K and hand it over by
// k_ready, the output warps do Q (two chunks ahead, between their output
// tiles) and hand it over by q_ready.  A value outside the fp16 range turns
// into inf in V', the state or o, which are checked.
// The 16 KB Q tile times gamma (sGam: exp(G) of the 64 rows), 16-byte
// vectors t, t + 128, ... (128 threads; vector v holds 8 dims of row
// (v & 511) >> 3): all eight loads first, then the stores.
__device__ __forceinline__ void round_q_tile(uint32_t base, uint32_t sGam, int t) {
  uint4 u[8];
  float gm[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int v = t + 128 * k;
    u[k] = lds_u32x4(base + (uint32_t)v * 16);
    gm[k] = lds_f32(sGam + (uint32_t)((v & 511) >> 3) * 4);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k)
    st_shared_v4(base + (uint32_t)(t + 128 * k) * 16, bf16x2_to_f16x2_scaled(u[k].x, gm[k]),
                 bf16x2_to_f16x2_scaled(u[k].y, gm[k]), bf16x2_to_f16x2_scaled(u[k].z, gm[k]),
                 bf16x2_to_f16x2_scaled(u[k].w, gm[k]));
}

template <bool PREP>
__device__ __forceinline__ void convert_role(uint8_t* sm, Ctl* ctl, const Chain& ch) {
  const int lane = threadIdx.x & 31, part = (threadIdx.x >> 5) - kConvertWarp;
  const int n = ch.run_end - ch.run_begin;
  for (int i = 0; i < n; ++i) {
    const int st = i & 1;
    if (!warp_ok(wait_bar(ctl, kKqFull0 + st, (uint32_t)((i >> 1) & 1)) &&
                 wait_bar(ctl, kGates0 + (i & 3), (uint32_t)((i >> 2) & 1))))
      break;
    const uint32_t base = smem_u32(sm + kRingK + st * kSlotK);
    const uint32_t sDec = smem_u32(sm + kSmG + (i & 3) * 512 + 256);
    // K halves at 0 and 8 KB: 16-byte vector v holds 8 dims of token row (v & 511) >> 3;
    // eight vectors per thread at a time, loads first
#pragma unroll 1
    for (int v0 = lane + 32 * part; v0 < 1024; v0 += 8 * 32 * kConvertWarps) {
      uint4 u[8];
      float d[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int v = v0 + k * 32 * kConvertWarps;
        u[k] = lds_u32x4(base + (uint32_t)v * 16);
        d[k] = lds_f32(sDec + (uint32_t)((v & 511) >> 3) * 4);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int v = v0 + k * 32 * kConvertWarps;
        st_shared_v4(base + (uint32_t)v * 16, bf16x2_to_f16x2_scaled(u[k].x, d[k]),
                     bf16x2_to_f16x2_scaled(u[k].y, d[k]), bf16x2_to_f16x2_scaled(u[k].z, d[k]),
                     bf16x2_to_f16x2_scaled(u[k].w, d[k]));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->bar[kKReady0 + st]);
  }
}

// ----------------------------------------------------------------- MMA issuer
// Per chunk i, in this order:
//   A(i)  -S W^T, once ring A of chunk i has landed and s_ready(i) has
//         published the state's fp16 copy (TMEM buffer i & 1); commits
//         va_done (the state warps add U^T and write V'(i) in fp16 to TMEM
//         buffer i & 1)
//   Y(i)  O = S (gamma Q)^T into O buffer i & 1, after q_ready(i) and
//         yo_free(i-2), issued while the state warps run the V' epilogue
//   D3(i) V'^T (diag(dec) K), after v_ready(i) and k_ready(i); commits
//         d3_done (which also tells the state warps that Y(i), issued
//         before it, has read state buffer i & 1 before the state of chunk
//         i + 2 goes there) and releases rings K and A (the state warps
//         read U^T before v_ready(i))
//   O2(i) O += V'^T P^T, issued while the state warps update the state;
//         commits yo_done(i) and releases ring B.
// The chain's critical path runs A(i) -> V' epilogue -> D3(i) -> state
// epilogue -> A(i+1); the output products fill the issuer's time in between.
// A(i+2), issued after O2(i), tells the state warps through va_done that V'
// buffer i & 1 has been read.
// The descriptor of the tile at byte offset off from the tile whose
// descriptor is d: the start-address field holds the shared-memory address
// >> 4 in its low 14 bits, and every tile here lies below 256 KB, so adding
// off >> 4 never carries out of the field.  With every descriptor derived
// this way from a few computed once, issuing an MMA costs one add.
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); }

template <bool PREP>
__device__ __forceinline__ void mma_role(uint8_t* sm, Ctl* ctl, const Chain& ch, uint32_t tmem) {
  const int n = ch.run_end - ch.run_begin;
  const uint32_t id_k = idesc_f16(128, 64, false, false);
  const uint32_t id_sw = idesc_f16(128, 64, false, true);
  const uint32_t id_d3 = idesc_f16(128, 128, false, true);
  // SW128 descriptors of the first slot of each ring
  const uint64_t dW0 = sdesc_sw128(smem_u32(sm + kRingA + kAWn), 8192, 1024);
  const uint64_t dK0 = sdesc_sw128(smem_u32(sm + kRingK), 8192, 1024);
  const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + kRingB + kBQ), 16, 1024);
  const uint64_t dP0 = sdesc_sw128(smem_u32(sm + kRingB + kBP), 16, 1024);
  if (n > 0 && !wait_bar(ctl, kFull0, 0u)) return;  // ring A of chunk 0
  for (int i = 0; i < n; ++i) {
    const int sb = i % 3;
    const uint64_t dW = desc_at(dW0, (uint32_t)(i & 1) * kSlotA), dK = desc_at(dK0, (uint32_t)(i & 1) * kSlotK);
    const uint64_t dQ = desc_at(dQ0, (uint32_t)sb * kSlotB), dP = desc_at(dP0, (uint32_t)sb * kSlotB);
    const uint32_t tS = tmem + kTS + (i & 1) * 64;    // the state's fp16 copy, 8 columns per K = 16 step
    const uint32_t tV = tmem + kTV16 + (i & 1) * 32;  // V''s fp16 copy, 8 columns per K = 16 step
    const uint32_t tO = tmem + kTO + (i & 1) * 64;
    const bool out = want_out<PREP>(ch, i);
    if (!spin_bar(ctl, kSReady, (uint32_t)(i & 1))) return;
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)  // -S W^T
      mma_f16_ts(tmem + kTV, tS + ks * 8, desc_at(dW, ks * 2048), id_sw, ks > 0 ? 1u : 0u);
    mma_commit(&ctl->bar[kVaDone]);
    if (out) {
      if (!wait_bar(ctl, kQReady0 + (i & 1), (uint32_t)((i >> 1) & 1))) return;
      if (i >= 2 && !wait_bar(ctl, kYoFree0 + (i & 1), (uint32_t)(((i - 2) >> 1) & 1))) return;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // O = S (gamma Q)^T
        mma_f16_ts(tO, tS + ks * 8, desc_at(dQ, (ks >> 2) * 8192 + (ks & 3) * 32), id_k, ks > 0 ? 1u : 0u);
    }
    if (!wait_bar(ctl, kKReady0 + (i & 1), (uint32_t)((i >> 1) & 1))) return;
    if (!spin_bar(ctl, kVReady, (uint32_t)(i & 1))) return;
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)  // D3 = V'^T diag(dec) K
      mma_f16_ts(tmem + kTD3, tV + ks * 8, desc_at(dK, ks * 2048), id_d3, ks > 0 ? 1u : 0u);
    mma_commit(&ctl->bar[kD3Done]);
    mma_commit(&ctl->bar[kEmptyK0 + (i & 1)]);  // ring K slot read
    mma_commit(&ctl->bar[kEmpty0 + (i & 1)]);   // ring A slot read (A(i); U^T before v_ready(i))
    if (out) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)  // O += V'^T P^T
        mma_f16_ts(tO, tV + ks * 8, desc_at(dP, ks * 32), id_k, 1u);
    }
    mma_commit(&ctl->bar[kYoDone0 + (i & 1)]);
    mma_commit(&ctl->bar[kEmptyB0 + sb]);  // ring B slot read (Y, O2)
    if (i + 1 < n && !wait_bar(ctl, kFull0 + ((i + 1) & 1), (uint32_t)(((i + 1) >> 1) & 1))) return;  // ring A
  }
}

// ----------------------------------------------------------------- output warps
// o = scale O for each chunk whose output is written:
// thread (warp w, lane) takes d_v row 32 (w & 3) + lane and all 64 tokens,
// 16 at a time, into the staging tile o[token][d_v] (a warp writes 64
// contiguous bytes of a token row).  One thread then stores the tile: a
// tensor store for a full chunk, one 256-byte bulk copy per token for a
// sequence's partial last chunk (whose other rows belong to the next
// sequence).  Every chunk, written or not, ends with yo_free, which
// releases Y/O2 buffer i & 1 to the MMA issuer.  The four warps decide
// together (a named barrier with an OR) whether to go on after each wait, so
// none is left behind at the next named barrier.
template <bool PREP>
__device__ __forceinline__ void output_role(uint8_t* sm, Ctl* ctl, const Problem& p, const SegInfo& si,
                                            const Chain& ch, uint32_t tmem, int j, const CUtensorMap* mo) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool issuer = threadIdx.x == kOutWarp * 32;
  const int row = (warp & 3) * 32 + lane;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t sO = smem_u32(sm + kSmO);
  const int n = ch.run_end - ch.run_begin;
  float mx = 0.f;  // largest |o| (inf or NaN when an fp16 operand overflowed)
  auto all_ok = [&](bool ok) { return !named_bar_or(kOutBarrier, kOutThreads, !ok); };
  // Q of chunk c times gamma = exp(G) of its row, rounded to fp16 (chunks
  // with no output: nothing to round), then q_ready(c); every chunk gets its
  // q_ready, so its phases follow c.
  auto round_q = [&](int c) -> bool {
    if (want_out<PREP>(ch, c)) {
      const bool ok = wait_bar(ctl, kQFull0 + c % 3, (uint32_t)((c / 3) & 1)) &&
                      wait_bar(ctl, kGates0 + (c & 3), (uint32_t)((c >> 2) & 1));
      if (!all_ok(ok)) return false;
      round_q_tile(smem_u32(sm + kRingB + (c % 3) * kSlotB + kBQ), smem_u32(sm + kSmG + (c & 3) * 512),
                   threadIdx.x - kOutWarp * 32);
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->bar[kQReady0 + (c & 1)]);
    return true;
  };
  for (int c = 0; c < 2 && c < n; ++c)
    if (!round_q(c)) return;
  for (int i = 0; i < n; ++i) {
    const bool out = want_out<PREP>(ch, i);
    if (!all_ok(wait_bar(ctl, kYoDone0 + (i & 1), (uint32_t)((i >> 1) & 1)))) break;
    if (out) {
      if (issuer) bulk_wait_read_all();  // the previous chunk's stores have read the tile
      named_bar_sync(kOutBarrier, kOutThreads);
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t oa[16], ob[16];
        tmem_ld16(tmem + lane_base + kTO + (i & 1) * 64 + h * 32, oa);
        tmem_ld16(tmem + lane_base + kTO + (i & 1) * 64 + h * 32 + 16, ob);
        tmem_ld_wait(oa, ob);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float o = p.scale * __uint_as_float(e < 16 ? oa[e] : ob[e - 16]);
          mx = absmax_nan(mx, o);
          sts_u16(sO + (uint32_t)(h * 32 + e) * 256u + (uint32_t)row * 2u,
                  __bfloat16_as_ushort(__float2bfloat16_rn(o)));
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(kOutBarrier, kOutThreads);
      if (issuer) {
        const int64_t t0 = si.bos + (int64_t)(ch.run_begin + i) * kChunk;
        const int cv = (int)min((int64_t)kChunk, si.eos - t0);
        if (cv == kChunk) {
          tma_store_3d(mo, sm + kSmO, 0, j, (int)t0);
        } else {
          uint8_t* orow = reinterpret_cast<uint8_t*>(p.out) + ((size_t)t0 * p.h_v + j) * kDim * 2;
          for (int r = 0; r < cv; ++r) bulk_store(orow + (size_t)r * p.h_v * kDim * 2, sm + kSmO + r * 256, 256u);
        }
        bulk_commit();
      }
    }
    tc_fence_before();
    mbar_arrive(&ctl->bar[kYoFree0 + (i & 1)]);  // O buffer i & 1 read
    if (i + 2 < n && !round_q(i + 2)) break;  // its ring B slot was loaded after O2(i - 1)
  }
  if (issuer) bulk_wait_all();  // the stores have landed before the block exits
  if (!(mx <= 3.4028235e38f)) atomicExch(&ctl->range_bad, 1);
}

// ----------------------------------------------------------------- state (chain) warps
template <bool PREP, bool DUMP>
__device__ __forceinline__ void chain_role(uint8_t* sm, Ctl* ctl, const Problem& p, const SegInfo& si,
                                        const Chain& ch, uint32_t tmem, int j, int chain) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127, half = tid >> 7;
  // The state lives only in these warps' registers.
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
  const int n = ch.run_end - ch.run_begin;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  // Largest magnitude this thread rounds to fp16: V' is checked every chunk;
  // the state only at the end, since an fp16 overflow of its operand copy
  // would turn the next V' and so the state into inf/NaN.
  float mx = 0.f;
  // The state's fp16 copy for chunk c into TMEM buffer c & 1: this thread's
  // row, its 64 columns packed into 32 (columns 32 half .. 32 half + 31).
  // DUMP (the backward's recompute): the copy of each output chunk's start
  // state also goes to p.hchunk (row = this thread's d_v, panel = half).
  uint8_t* const hdump = (DUMP && !PREP)
                             ? p.hchunk + ((size_t)(ch.chunk0 + ch.run_begin) * p.h_v + j) * 32768u +
                                   (size_t)half * 16384u
                             : nullptr;
  auto store_state = [&](int c) {
    uint32_t w[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) w[q] = pack_f16x2(S[2 * q], S[2 * q + 1]);
    tmem_st32(tmem + lane_base + kTS + (c & 1) * 64 + half * 32, w);
    if (DUMP && c < n && ch.run_begin + c >= ch.out_begin) {
      uint8_t* dst = hdump + (size_t)c * p.h_v * 32768u;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(dst + sw128_offset(row, q)) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    tmem_st_wait();
  };
  store_state(0);
  tc_fence_before();
  mbar_arrive(&ctl->bar[kSReady]);
  int done = 0;
  for (int i = 0; i < n; ++i) {
    const uint32_t par = (uint32_t)(i & 1);
    const uint32_t sGam = smem_u32(sm + kSmG + (i & 3) * 512);  // exp(G) [64], then dec [64]
    if (!warp_ok(wait_bar(ctl, kGates0 + (i & 3), (uint32_t)((i >> 2) & 1)))) break;
    // U^T of this thread's row and 32 tokens (16-byte chunks half * 4 .. + 3 of
    // the row in ring A), read while A(i) runs
    uint4 uq[4] = {};
    if (ch.has_u) {
      if (!warp_ok(wait_bar(ctl, kFull0 + (i & 1), (uint32_t)((i >> 1) & 1)))) break;
      const uint32_t sU = smem_u32(sm + kRingA + (i & 1) * kSlotA + kAU);
#pragma unroll
      for (int c = 0; c < 4; ++c) uq[c] = lds_u32x4(sU + sw128_offset(row, half * 4 + c));
    }
    if (!warp_ok(wait_bar(ctl, kVaDone, par))) break;
    tc_fence_after();
    const float gC = lds_f32(sGam + 63 * 4);
    // V' = U^T - S W^T, its fp16 copy into TMEM buffer i & 1 (columns 16 half ..
    // 16 half + 15: this thread's 32 tokens), the A operand of D3 and O2 (the
    // decay to the chunk end is in K)
    {
      uint32_t va[16], vb[16], w[16];
      tmem_ld16(tmem + lane_base + kTV + half * 32, va);
      tmem_ld16(tmem + lane_base + kTV + half * 32 + 16, vb);
      tmem_ld_wait(va, vb);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t* acc = q4 < 2 ? &va[q4 * 8] : &vb[(q4 - 2) * 8];
        const uint32_t uw[4] = {uq[q4].x, uq[q4].y, uq[q4].z, uq[q4].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 u2 = __half22float2(*reinterpret_cast<const __half2*>(&uw[e]));
          const float f0 = __uint_as_float(acc[2 * e]) + u2.x, f1 = __uint_as_float(acc[2 * e + 1]) + u2.y;
          mx = absmax_nan(absmax_nan(mx, f0), f1);
          w[q4 * 4 + e] = pack_f16x2(f0, f1);
        }
      }
      tmem_st16(tmem + lane_base + kTV16 + (i & 1) * 32 + half * 16, w);
      tmem_st_wait();
    }
    tc_fence_before();
    mbar_arrive(&ctl->bar[kVReady]);
    // S = gamma_C S + D3
    if (!warp_ok(wait_bar(ctl, kD3Done, par))) break;
    tc_fence_after();
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
    // buffer (i + 1) & 1 was last read by A(i - 1) and Y(i - 1), both issued
    // before D3(i - 1), whose completion this thread has seen
    store_state(i + 1);
    tc_fence_before();
    mbar_arrive(&ctl->bar[kSReady]);
    done = i + 1;
  }
#pragma unroll
  for (int e = 0; e < 64; ++e) mx = absmax_nan(mx, S[e]);
  if (!(mx < 65504.f)) atomicExch(&ctl->range_bad, 1);
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

template <bool PREP, bool DUMP = false>
__global__ void __launch_bounds__(kThreads, 1)
    scan_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mo, const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + kSmCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the preprocessing's two chains of a segment are neighbouring blocks
  // (x = 2 segment + chain), so both of a head's chains come in the same wave
  const int j = blockIdx.y;
  const int chain = PREP ? (int)(blockIdx.x & 1) : 0;
  const int seg = PREP ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_segs = PREP ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // ---- which chain this CTA runs ----
  // The segment comes from the plan's arithmetic and the sequence bounds (an
  // input), so warps 0 and 1 locate it before waiting for the kernel before
  // this one: while that kernel finishes on other SMs.  After the wait, warp
  // 0 fetches the words the set-up depends on together, so that their
  // latencies overlap: the status word, and for the output scan the head's
  // mode and the segment's warmup depth; warp 1 of the preprocessing
  // computes the warmup depths of the head's segments.
  __shared__ int s_mode, s_w, s_exact;
  SegInfo si0;
  bool ok0 = false;
  if (warp < 2) ok0 = locate_segment(p, seg, si0);
  if (tid == 64) {  // the barriers and tensor maps, also before the wait
    const int counts[kNumBars] = {1, 1, 1, 1, 1, 1, 1, 1, 1, kChainThreads, 1, kChainThreads,
                                  1, 1, kOutThreads, kOutThreads, 1, 1, kConvertWarps, kConvertWarps,
                                  kOutThreads / 32, kOutThreads / 32, 1, 1, 1, 1, 1, 1, 1, 1};
    for (int b = 0; b < kNumBars; ++b) mbar_init(&ctl->bar[b], counts[b]);
    ctl->abort = 0;
    ctl->range_bad = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    if (!PREP) tma_prefetch_desc(&mo);
  }
  grid_dependency_wait();  // records, chunk index, segment states: written by the kernels before
  grid_launch_dependents();
  if (warp == 0) {
    SegInfo si = si0;
    const bool ok = ok0;
    int v = 0;
    if (lane == 0) v = earlier_failure(p.status);
    if (!PREP && ok && p.plan_mode != kModeOff) {
      if (lane == 1) v = p.head_mode[si.n * p.h_v + j];
      if (lane == 2 && p.plan_mode == kModeWarmup) v = p.seg_w[(size_t)(si.seg_base + si.s) * p.h_v + j];
    }
    const int mode = __shfl_sync(0xffffffffu, v, 1), w = __shfl_sync(0xffffffffu, v, 2);
    if (lane == 0) {
      if (!ok) si.n = -1;
      ctl->seg = si;
      ctl->skip = v;
      s_mode = mode;
      s_w = w;
    }
  } else if (warp == 1) {
    // warmup depths of every segment of this (sequence, head) from the chunk
    // exponents; the head runs exactly unless all of them found a depth.  The
    // first CTA of each segment records its depth for the combine and the scan.
    bool none = false;
    if (PREP && p.plan_mode == kModeWarmup) {
      const SegInfo si = si0;
      const int chunk0 = ok0 ? seq_first_chunk(p, si.n) : -1;
      if (ok0 && chunk0 >= 0 && chunk0 + si.n_chunks <= p.n_chunks_total) {
        for (int s2 = lane; s2 < si.n_seg; s2 += 32) {
          int w = 0;
          float b = -__int_as_float(0x7f800000);
          if (s2 > 0) seg_warmup_depth(p, chunk0, seg_first(s2, si.n_chunks, si.n_seg), j, w, b);
          none |= w < 0;
          if (s2 == si.s && chain == 0) {
            p.seg_w[(size_t)(si.seg_base + s2) * p.h_v + j] = w;
            p.seg_bound[(size_t)(si.seg_base + s2) * p.h_v + j] = b;
          }
        }
      }
    }
    none = __any_sync(0xffffffffu, none);
    if (lane == 0) s_exact = !PREP || p.plan_mode != kModeWarmup || none;
  }
  __syncthreads();
  if (ctl->skip) return;  // an earlier kernel failed: its results are incomplete
  const SegInfo si = ctl->seg;
  if (si.n < 0) {
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return;
  }
  if (seg == n_segs - 1 && !(si.n == p.n_seqs - 1 && si.s == si.n_seg - 1)) {
    if (tid == 0 && blockIdx.y == 0 && chain == 0) report(p.status, kDevCheck, kDetSegMismatch);
  }
  Chain ch;
  ch.bos = si.bos;
  ch.run_begin = si.cb;
  ch.run_end = si.ce;
  ch.out_begin = si.cb;
  ch.init = kInitZero;
  ch.has_u = true;
  ch.write_final = false;
  if (PREP) {
    if (!s_exact) return;  // a warmup head: no transition or local state needed
    if (si.s == si.n_seg - 1) return;
    if (chain == 0 && si.s == 0 && p.h0 == nullptr) return;  // M of segment 0 unused for a zero start
    ch.init = chain == 0 ? kInitIdentity : kInitZero;
    ch.has_u = chain == 1;
  } else {
    const int mode = p.plan_mode == kModeOff ? kModeOff : s_mode;
    if (si.s == 0) {
      ch.init = kInitH0;
    } else if (mode == kModeWarmup) {
      const int ws = si.cb - s_w;
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
  ch.iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
  ch.chunk0 = seq_first_chunk(p, si.n);
  if (ch.chunk0 < 0 || ch.chunk0 + si.n_chunks > p.n_chunks_total || ch.run_begin < 0 ||
      ch.run_begin > ch.run_end) {  // the chunk index or the warmup depth disagrees with the plan
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return;
  }

  // ---- set-up ----
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  if (warp < 8) {
    setmaxnreg_inc<kChainRegs>();
    chain_role<PREP, DUMP>(sm, ctl, p, si, ch, tmem, j, chain);
  } else {
    setmaxnreg_dec<kOtherRegs>();
    if (warp < kOutWarp + 4) {
      output_role<PREP>(sm, ctl, p, si, ch, tmem, j, &mo);
    } else if (warp == kProducerWarp) {
      producer_role<PREP>(sm, ctl, p, ch, j, &mq, &mk);
    } else if (warp >= kConvertWarp) {
      convert_role<PREP>(sm, ctl, ch);
    } else if (warp == kMmaWarp && lane == 0) {
      mma_role<PREP>(sm, ctl, ch, tmem);
    }
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
  e = cudaFuncSetAttribute(scan_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
}

cudaError_t launch_scan_prep(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, cudaStream_t st) {
  dim3 grid(2 * p.n_seg_total, p.h_v);
  return launch_kernel(scan_kernel<true>, grid, dim3(kThreads), kSmemAlloc, st, true, mq, mk, mq,
                       p);  // writes no output: o's map unused
}

cudaError_t launch_scan_out(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mo,
                            int grid_x, cudaStream_t st) {
  dim3 grid(grid_x, p.h_v, 1);
  if (p.hchunk)  // the backward's recompute: also keeps every chunk's start state
    return launch_kernel(scan_kernel<false, true>, grid, dim3(kThreads), kSmemAlloc, st, true, mq, mk, mo, p);
  return launch_kernel(scan_kernel<false>, grid, dim3(kThreads), kSmemAlloc, st, true, mq, mk, mo, p);
}

}  // namespace gdn
