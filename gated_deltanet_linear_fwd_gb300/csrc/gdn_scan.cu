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
//   A    = (I + L)^{-1}                    (fp32 forward substitution)
//   W^T  = K^T (A diag(beta gamma))^T,  U^T = V^T (A diag(beta))^T
//   V'^T = U^T - S W^T,  Y = S Q^T          (one pass over the bf16 state)
//   O^T  = scale (Y diag(gamma) + V'^T P^T)
//   S    = gamma_C S + V'^T diag(exp(G_last - G)) K
// The state itself stays fp32 in registers.  Every MMA operand derived in
// the kernel (the state, A, V', P) is carried as a pair of bf16 numbers,
// hi = bf16(x) and lo = bf16(x - hi), and its product is the sum of the
// hi*hi, hi*lo and lo*hi terms (inputs q, k, v are exact in bf16 and need one
// term), so each contraction is accurate to about 2^-16 relative; a single
// bf16 rounding of those operands costs more than the whole error budget.
// Only W stays a single bf16 operand.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

// ---- shared memory map (bytes from a 1024-byte aligned base) ----
constexpr uint32_t kStageBytes = 49152;  // per stage: K,Q halves (32 KB) + V halves (16 KB)
constexpr uint32_t kStKQ = 0;            // [K d0-63 | Q d0-63 | K d64-127 | Q d64-127], 8 KB each
constexpr uint32_t kStV = 32768;         // [V d0-63 | V d64-127]
// state operand, K-major A: hi (two 64-column halves of 16 KB) then lo.
// Between the state MMAs and the state update the same 64 KB hold the V'
// operands (K-major A, 16 KB each): V' hi, V' lo, V'dec hi, V'dec lo.
constexpr uint32_t kSmS = 98304;
constexpr uint32_t kSmWn = 163840;       // -W, MN-major B: rows d_k, 64 chunk rows each
constexpr uint32_t kSmP = 180224;        // P hi | P lo, K-major B: rows r
// 32 KB scratch, by phase: fp32 L (row stride 68); then the A operands
// (MN-major B, 8 KB each: A diag(beta gamma) hi, lo, A diag(beta) hi, lo);
// then the bf16 output tile [64][128].
constexpr uint32_t kSmX = 196608;
constexpr uint32_t kLStride = 68;
constexpr uint32_t kSmSmall = 229376;    // G, gamma, decay, beta: 64 floats each
constexpr uint32_t kSmCtl = 230400;      // barriers, TMEM base, flags
constexpr uint32_t kSmemUse = 230656;
constexpr uint32_t kSmemAlloc = kSmemUse + 1024;

// ---- TMEM columns (512 allocated) ----
constexpr uint32_t kTKQ = 0;    // [K K^T ; Q K^T]      128 x 64
constexpr uint32_t kTW = 64;    // W^T                  128 x 64
constexpr uint32_t kTV = 128;   // U^T, then V'^T       128 x 64
constexpr uint32_t kTQ = 192;   // S Q^T                128 x 64
constexpr uint32_t kTO2 = 256;  // V'^T P^T             128 x 64
constexpr uint32_t kTD3 = 320;  // V'^T diag(dec) K     128 x 128

enum InitKind { kInitZero = 0, kInitIdentity = 1, kInitH0 = 2, kInitStart = 3 };

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// hi = bf16(a,b), lo = bf16(a - hi, b - hi): the pair carries ~16 mantissa bits.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}

// Writes 8 consecutive values as a 16-byte chunk of a hi tile and of a lo tile.
__device__ __forceinline__ void store_split8(uint32_t hi_addr, uint32_t lo_addr, const float* f) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split2(f[2 * e], f[2 * e + 1], h[e], l[e]);
  st_shared_v4(hi_addr, h[0], h[1], h[2], h[3]);
  st_shared_v4(lo_addr, l[0], l[1], l[2], l[3]);
}

struct Ctl {
  uint64_t bar[3];  // 0,1: TMA stages; 2: MMA completion
  uint32_t tmem;
  int abort;
  float warp_total[2];
  SegInfo seg;
};

template <bool PREP>
__global__ void __launch_bounds__(256, 1)
    scan_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sG = reinterpret_cast<float*>(sm + kSmSmall);
  float* sGam = sG + 64;
  float* sDec = sG + 128;
  float* sBeta = sG + 192;
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + kSmCtl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127, half = tid >> 7;
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

  int init = kInitZero, run_begin = si.cb, out_begin = si.cb;
  const int run_end = si.ce;
  bool write_final = false;
  bool has_u = true;
  if (PREP) {
    if (head_mode_of(p, si, j) != kModeExact || si.s == si.n_seg - 1) return;
    if (chain == 0 && si.s == 0 && p.h0 == nullptr) return;  // M of segment 0 unused for a zero start
    init = chain == 0 ? kInitIdentity : kInitZero;
    has_u = chain == 1;
  } else {
    const int mode = p.plan_mode == kModeOff ? kModeOff : p.head_mode[si.n * p.h_v + j];
    if (si.s == 0) {
      init = kInitH0;
    } else if (mode == kModeWarmup) {
      const int ws = si.cb - p.warmup_chunks;
      if (ws <= 0) {
        run_begin = 0;
        init = kInitH0;
      } else {
        run_begin = ws;
        init = kInitZero;
      }
    } else {
      init = kInitStart;
    }
    write_final = (p.hT != nullptr) && si.s == si.n_seg - 1;
  }
  if (init == kInitH0 && p.h0 == nullptr) init = kInitZero;
  const bool need_q = !PREP;
  const bool need_v = has_u;
  const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);

  // ---- set-up: barriers, TMEM, initial state ----
  if (tid == 0) {
    mbar_init(&ctl->bar[0], 1);
    mbar_init(&ctl->bar[1], 1);
    mbar_init(&ctl->bar[2], 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mk);
    if (need_q) tma_prefetch_desc(&mq);
    if (need_v) tma_prefetch_desc(&mv);
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }

  float S[64];
  {
    const size_t head_off = (size_t)(si.n * p.h_v + j) * kDim * kDim;
    if (init == kInitH0) {
#pragma unroll
      for (int i = 0; i < 64; ++i) S[i] = p.h0[head_off + (size_t)(half * 64 + i) * kDim + row];
    } else if (init == kInitStart) {
      const float4* src = reinterpret_cast<const float4*>(
          p.Sstart + ((size_t)(si.seg_base + si.s) * p.h_v + j) * kDim * kDim + (size_t)row * kDim + half * 64);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 v4 = src[i];
        S[4 * i] = v4.x;
        S[4 * i + 1] = v4.y;
        S[4 * i + 2] = v4.z;
        S[4 * i + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) S[i] = (init == kInitIdentity && half * 64 + i == row) ? 1.f : 0.f;
    }
  }
  const uint32_t sS = smem_u32(sm + kSmS);  // state hi at +0, lo at +32768
  auto store_state = [&]() {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t off = half * 16384 + sw128_offset(row, q);
      store_split8(sS + off, sS + 32768 + off, &S[8 * q]);
    }
  };
  store_state();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  auto issue_tma = [&](int cid, int stage) {
    uint8_t* st = sm + stage * kStageBytes;
    const int t0 = (int)(si.bos + (int64_t)cid * kChunk);
    const uint32_t bytes = 16384u + (need_q ? 16384u : 0u) + (need_v ? 16384u : 0u);
    mbar_arrive_expect_tx(&ctl->bar[stage], bytes);
    tma_load_3d(st + kStKQ, &mk, &ctl->bar[stage], 0, iq, t0);
    tma_load_3d(st + kStKQ + 16384, &mk, &ctl->bar[stage], 64, iq, t0);
    if (need_q) {
      tma_load_3d(st + kStKQ + 8192, &mq, &ctl->bar[stage], 0, iq, t0);
      tma_load_3d(st + kStKQ + 24576, &mq, &ctl->bar[stage], 64, iq, t0);
    }
    if (need_v) {
      tma_load_3d(st + kStV, &mv, &ctl->bar[stage], 0, j, t0);
      tma_load_3d(st + kStV + 8192, &mv, &ctl->bar[stage], 64, j, t0);
    }
  };

  const uint32_t sWn = smem_u32(sm + kSmWn), sP = smem_u32(sm + kSmP), sX = smem_u32(sm + kSmX);
  // operand addresses inside the aliased regions
  const uint32_t sAbgH = sX, sAbgL = sX + 8192, sAbH = sX + 16384, sAbL = sX + 24576;
  const uint32_t sVpH = sS, sVpL = sS + 16384, sVdH = sS + 32768, sVdL = sS + 49152;
  const uint32_t sPH = sP, sPL = sP + 8192;
  float* sL = reinterpret_cast<float*>(sm + kSmX);
  __nv_bfloat16* sO = reinterpret_cast<__nv_bfloat16*>(sm + kSmX);

  uint32_t mma_phase = 0;
  int pending_stage = -1;  // stage with a TMA in flight not yet waited on
  uint32_t pending_parity = 0;
  bool aborted = false;

  auto wait_mma = [&]() -> bool {
    if (!mbar_wait(&ctl->bar[2], mma_phase, kWaitLimitNs)) ctl->abort = kDetMmaWait;
    mma_phase ^= 1;
    __syncthreads();
    if (ctl->abort) return false;
    tc_fence_after();
    return true;
  };

  if (tid == 0 && run_end > run_begin) issue_tma(run_begin, 0);
  if (run_end > run_begin) {
    pending_stage = 0;
    pending_parity = 0;
  }

  int it = 0;
  for (int cid = run_begin; cid < run_end; ++cid, ++it) {
    const int stage = it & 1;
    const uint32_t stKQ = smem_u32(sm + stage * kStageBytes + kStKQ);
    const uint32_t stV = smem_u32(sm + stage * kStageBytes + kStV);
    const int64_t t0 = si.bos + (int64_t)cid * kChunk;
    const int cv = (int)min((int64_t)kChunk, si.eos - t0);
    const bool want_out = !PREP && cid >= out_begin;

    // (1) gates of this chunk (rows past the sequence end act as g = beta = 0)
    float gval = 0.f, bval = 0.f;
    if (tid < 64 && tid < cv) {
      gval = p.g[(size_t)(t0 + tid) * p.h_v + j];
      bval = p.beta[(size_t)(t0 + tid) * p.h_v + j];
    }
    if (!mbar_wait(&ctl->bar[stage], (uint32_t)((it >> 1) & 1), kWaitLimitNs)) ctl->abort = kDetTmaWait;
    __syncthreads();
    if (ctl->abort) { aborted = true; break; }
    pending_stage = -1;

    // (2) prefetch the next chunk; D_kq = [K;Q] K^T
    if (tid == 0) {
      if (cid + 1 < run_end) issue_tma(cid + 1, stage ^ 1);
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
        mma_bf16(tmem + kTKQ, sdesc_sw128(stKQ + off, 16, 1024), sdesc_sw128(stKQ + off, 16, 1024), idesc,
                 ks > 0);
      }
      mma_commit(&ctl->bar[2]);
    }
    if (cid + 1 < run_end) {
      pending_stage = stage ^ 1;
      pending_parity = (uint32_t)(((it + 1) >> 1) & 1);
    }

    // (3) inclusive gate cumsum within the chunk (warps 0 and 1)
    if (tid < 64) {
      float x = gval;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
      }
      if (lane == 31) ctl->warp_total[warp] = x;
      named_bar_sync(1, 64);
      if (warp == 1) x += ctl->warp_total[0];
      sG[tid] = x;
      sBeta[tid] = bval;
      named_bar_sync(1, 64);
      const float glast = sG[63];
      sGam[tid] = __expf(x);
      sDec[tid] = __expf(glast - x);
    }
    if (!wait_mma()) { aborted = true; break; }

    // (4) L (rows 0-63 of D_kq, fp32) and P (rows 64-127, hi/lo bf16)
    {
      uint32_t r32[32];
      tmem_ld32(tmem + lane_base + kTKQ + half * 32, r32);
      tmem_ld_wait(r32);
      if (row < 64) {
        const int r = row;
        const float br = sBeta[r], Gr = sG[r];
        float* Lrow = sL + r * kLStride + half * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 o4;
          float* o = &o4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = half * 32 + i + e;
            o[e] = (s < r) ? br * __uint_as_float(r32[i + e]) * __expf(Gr - sG[s]) : 0.f;
          }
          *reinterpret_cast<float4*>(Lrow + i) = o4;
        }
      } else if (!PREP) {
        const int r = row - 64;
        const float Gr = sG[r];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = half * 32 + q * 8 + e;
            f[e] = (s <= r) ? __uint_as_float(r32[q * 8 + e]) * __expf(Gr - sG[s]) : 0.f;
          }
          const uint32_t off = sw128_offset(r, half * 4 + q);
          store_split8(sPH + off, sPL + off, f);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // (5) A = (I + L)^{-1} by forward substitution, one column per thread;
    //     the A operands overwrite L, so the solvers sync before writing.
    if (tid < 64) {
      float x[64];
#pragma unroll
      for (int r = 0; r < 64; ++r) x[r] = 0.f;
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        float a0 = (r == tid) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int s = 0; s < r; s += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(sL + r * kLStride + s);
          a0 -= l4.x * x[s];
          a1 -= l4.y * x[s + 1];
          a2 -= l4.z * x[s + 2];
          a3 -= l4.w * x[s + 3];
        }
        x[r] = (a0 + a1) + (a2 + a3);
      }
      named_bar_sync(1, 64);
      // column `tid` of A -> row `tid` of the MN-major B operands
      const float bg = sBeta[tid] * sGam[tid], b = sBeta[tid];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float f[8];
        const uint32_t off = sw128_offset(tid, q);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = x[8 * q + e] * bg;
        store_split8(sAbgH + off, sAbgL + off, f);
        if (has_u) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = x[8 * q + e] * b;
          store_split8(sAbH + off, sAbL + off, f);
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // (6) W^T = K^T (A diag(beta gamma))^T ; U^T = V^T (A diag(beta))^T   (A as hi + lo)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_mn = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t kk = (uint32_t)(ks & 3) * 2048u;
        mma_bf16(tmem + kTW, sdesc_sw128(stKQ + kk, 16384, 1024),
                 sdesc_sw128((ks < 4 ? sAbgH : sAbgL) + kk, 8192, 1024), id_mn, ks > 0);
      }
      if (has_u) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t kk = (uint32_t)(ks & 3) * 2048u;
          mma_bf16(tmem + kTV, sdesc_sw128(stV + kk, 8192, 1024),
                   sdesc_sw128((ks < 4 ? sAbH : sAbL) + kk, 8192, 1024), id_mn, ks > 0);
        }
      }
      mma_commit(&ctl->bar[2]);
    }
    if (!wait_mma()) { aborted = true; break; }

    // (7) -W into the MN-major B operand (row d_k, 64 chunk rows)
    {
      uint32_t r32[32];
      tmem_ld32(tmem + lane_base + kTW + half * 32, r32);
      tmem_ld_wait(r32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float* f = reinterpret_cast<const float*>(&r32[q * 8]);
        st_shared_v4(sWn + sw128_offset(row, half * 4 + q), pack_bf16x2(-f[0], -f[1]), pack_bf16x2(-f[2], -f[3]),
                     pack_bf16x2(-f[4], -f[5]), pack_bf16x2(-f[6], -f[7]));
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // (8) V'^T = U^T - S W^T ; Y = S Q^T    (S as hi + lo)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_a = idesc_bf16_f32(128, 64, false, true);
      const uint32_t id_q = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        const uint32_t kin = (uint32_t)(ks & 7);
        const uint32_t aoff = (ks < 8 ? 0u : 32768u) + (kin >> 2) * 16384u + (kin & 3) * 32u;
        const uint64_t a = sdesc_sw128(sS + aoff, 16, 1024);
        mma_bf16(tmem + kTV, a, sdesc_sw128(sWn + kin * 2048, 8192, 1024), id_a, (has_u || ks > 0) ? 1u : 0u);
        if (want_out) {
          const uint32_t boff = (kin >> 2) * 16384u + (kin & 3) * 32u;
          mma_bf16(tmem + kTQ, a, sdesc_sw128(stKQ + 8192 + boff, 16, 1024), id_q, ks > 0);
        }
      }
      mma_commit(&ctl->bar[2]);
    }
    if (!wait_mma()) { aborted = true; break; }

    // (9) V' operands (hi/lo): plain (for O) and decayed to the chunk end (for S).
    //     They overwrite the state operand, which the MMAs above have consumed.
    {
      uint32_t r32[32];
      tmem_ld32(tmem + lane_base + kTV + half * 32, r32);
      tmem_ld_wait(r32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float* f = reinterpret_cast<const float*>(&r32[q * 8]);
        const float* d = sDec + half * 32 + q * 8;
        const uint32_t off = sw128_offset(row, half * 4 + q);
        if (want_out) store_split8(sVpH + off, sVpL + off, f);
        float fd[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) fd[e] = f[e] * d[e];
        store_split8(sVdH + off, sVdL + off, fd);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // (10) O2 = V'^T P^T (hi*hi + hi*lo + lo*hi) ; D3 = V'^T diag(dec) K (hi + lo)
    if (tid == 0) {
      tc_fence_after();
      if (want_out) {
        const uint32_t id_o = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < 12; ++ks) {
          const int term = ks >> 2;  // 0: hi*hi, 1: hi*lo, 2: lo*hi
          const uint32_t kk = (uint32_t)(ks & 3) * 32u;
          const uint32_t a = (term == 2 ? sVpL : sVpH) + kk, b = (term == 1 ? sPL : sPH) + kk;
          mma_bf16(tmem + kTO2, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), id_o, ks > 0);
        }
      }
      const uint32_t id_c = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t kk = (uint32_t)(ks & 3);
        mma_bf16(tmem + kTD3, sdesc_sw128((ks < 4 ? sVdH : sVdL) + kk * 32u, 16, 1024),
                 sdesc_sw128(stKQ + kk * 2048u, 16384, 1024), id_c, ks > 0);
      }
      mma_commit(&ctl->bar[2]);
    }
    if (!wait_mma()) { aborted = true; break; }

    // (11) S = gamma_C S + D3 ; output staging
    {
      const float gC = __expf(sG[63]);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t r32[32];
        tmem_ld32(tmem + lane_base + kTD3 + half * 64 + h2 * 32, r32);
        tmem_ld_wait(r32);
#pragma unroll
        for (int i = 0; i < 32; ++i) S[h2 * 32 + i] = fmaf(gC, S[h2 * 32 + i], __uint_as_float(r32[i]));
      }
      store_state();
      if (want_out) {
        uint32_t yq[32], o2[32];
        tmem_ld32(tmem + lane_base + kTQ + half * 32, yq);
        tmem_ld_wait(yq);
        tmem_ld32(tmem + lane_base + kTO2 + half * 32, o2);
        tmem_ld_wait(o2);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = half * 32 + i;
          const float o = p.scale * fmaf(sGam[c], __uint_as_float(yq[i]), __uint_as_float(o2[i]));
          sO[c * kDim + row] = __float2bfloat16_rn(o);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (want_out) {
      __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = tid + q * 256;
        const int r = idx >> 4, c16 = idx & 15;
        if (r < cv) {
          const uint4 val = *reinterpret_cast<const uint4*>(sO + r * kDim + c16 * 8);
          *reinterpret_cast<uint4*>(outp + ((size_t)(t0 + r) * p.h_v + j) * kDim + c16 * 8) = val;
        }
      }
    }
  }

  // ---- results ----
  if (aborted) {
    if (tid == 0) {
      report(p.status, kDevTimeout, ctl->abort);
      if (pending_stage >= 0) mbar_wait(&ctl->bar[pending_stage], pending_parity, kWaitLimitNs);
      mbar_wait(&ctl->bar[2], mma_phase, kWaitLimitNs);
    }
  } else if (PREP) {
    float* dst = (chain == 0 ? p.R : p.Sloc) + ((size_t)(si.seg_base + si.s) * p.h_v + j) * kDim * kDim +
                 (size_t)row * kDim + half * 64;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      reinterpret_cast<float4*>(dst)[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
  } else if (write_final) {
    float* dst = p.hT + (size_t)(si.n * p.h_v + j) * kDim * kDim;
#pragma unroll
    for (int i = 0; i < 64; ++i) dst[(size_t)(half * 64 + i) * kDim + row] = S[i];
  }
  tc_fence_before();
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
  scan_kernel<true><<<grid, 256, kSmemAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

cudaError_t launch_scan_out(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            int grid_x, cudaStream_t st) {
  dim3 grid(grid_x, p.h_v, 1);
  scan_kernel<false><<<grid, 256, kSmemAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace gdn
