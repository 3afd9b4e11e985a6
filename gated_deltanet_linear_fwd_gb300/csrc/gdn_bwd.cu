// Backward of the chunked GDN forward: gradients of  sum(o * do) + sum(h_T * dh_T)
// with respect to q, k, v, g, beta and h0.
//
// The FlashQLA pages (section "TileLang warp-specialised kernels", the
// backward-pass bullet) fuse the dv, dh, dq/dk/dw/dg and WY gradient steps into
// one kernel; they give no formulas.  The gradients here follow the chunk-level
// derivation through the WY form (one chunk, C rows, chunk-start state H,
// gradient D of the chunk-end state; W, U, P, Ktil, gamma, dec as in the
// forward's records):
//   dV'  = scale P^T dO + Ktil D                 D_prev = gamma_C D + E + T' D
//   E    = scale (diag(gamma) Q)^T dO - W^T (scale P^T dO),   T' = -W^T Ktil
//   dQ   = scale diag(gamma) dO H^T + (dP * Gam) K,            dP = scale dO V'^T
//   dK   = (dP * Gam)^T Q + diag(dec) V' D^T - diag(beta gamma) Y_U H^T + (dKK + dKK^T) K
//   Y_U  = A^T dV',  dV = diag(beta) Y_U,  dL = -A^T dV' V'^T (strict lower)
//   dKK  = dL * beta * Gam;  the gates through dG and a reverse cumulative sum.
//
// Three stages (five kernels) after a forward pass, in the plan's mode, that
// also leaves each chunk's start state and A^T (fp16), all on the 5th-generation
// tensor cores (tcgen05, accumulators
// in TMEM; fp16 operands in the forward's 128-byte-swizzled tile image; tiles
// by bulk copies on mbarriers; every wait bounded):
//   bwd_pre_tc_kernel    per (chunk, value head): T' and E (chunk-parallel)
//   bwd_chain2_tc_kernel, the combine run backwards, bwd_chain_tc_kernel:
//                        the state gradient D over each segment's chunks in
//                        reverse, in fp32 registers, context parallel like the
//                        forward (per segment the transition and the local
//                        offset together, the segments' end-state gradients by
//                        the combine, then the final pass writing every chunk's
//                        D (fp16) and dh0)
//   bwd_local_tc_kernel  per (chunk, q/k head), over the value heads of the
//                        group: every other gradient
//
// The chunk-local gradients, one CTA per (chunk, q/k head), the value heads of
// the group one after the other:
//   V'^T = U^T - S W^T                      (S = H^T, the chunk-start state)
//   dV'^T = scale dO^T P + D^T Ktil^T
//   dq^T += scale H dO^T diag(gamma) + K^T (dP * Gam)^T
//   dk^T += Q^T (dP * Gam) + D V'^T diag(dec) - H Y_U^T diag(beta gamma)
//           + K^T (dKK^T + dKK)
//   Y_U^T = dV'^T A,  dv = diag(beta) Y_U
//   [dP; dL_raw] = scale [dO; dV'] V'^T (lower triangles),  dL = -A^T dL_raw
// Products have M = 128: a head dimension (d_k or d_v) as rows and the 64
// tokens as columns, or two stacked 64-row operands ([dO; dV'], [Q; K]).  The
// per-token sums over a head dimension (dgamma, ddec, <Y_U, V>, <Y_W, K>) are
// column sums across TMEM lanes: a 31-shuffle butterfly per warp, then the
// four lane quarters through shared memory.  16 warps: four per lane quarter,
// each thread taking 16 of a 64-column accumulator.  Operand tiles are fp16 in the
// forward's 128-byte-swizzled image (bulk copies of the records and states,
// the rest written by the epilogues); one thread issues the MMAs and commits
// each phase to an mbarrier; every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdn_dev.cuh"

namespace gdn {
namespace {

constexpr int kTcThreads = 256;
constexpr int kLocThreads = 512;  // the chunk-local kernel: 16 warps (4 per lane quarter)

// ---- shared memory (bytes from a 1024-byte aligned base) ----
constexpr uint32_t sQK = 0;          // [Q d0-63 | K d0-63 | Q d64-127 | K d64-127], 64 rows each
constexpr uint32_t sS = 32768;       // S = H^T: 128 (d_v) x 128 (d_k), panels d_k 0-63 | 64-127
constexpr uint32_t sD = 65536;       // D: 128 (d_k) x 128 (d_v), panels d_v 0-63 | 64-127
constexpr uint32_t sWt = 98304;      // -W^T record tile 128 (d_k) x 64; then dV'^T 128 (d_v) x 64
constexpr uint32_t sUt = 114688;     // U^T record tile 128 (d_v) x 64; then Y_U^T 128 (d_v) x 64
constexpr uint32_t sP = 131072;      // P record tile 64 x 64; then dL_raw
constexpr uint32_t sPG = 139264;     // dP * Gam 64 x 64 (also rows 0-63 of the padded dL product); then dKK
constexpr uint32_t sAT = 147456;     // A^T 64 x 64
constexpr uint32_t sDOV = 155648;    // [dO d0-63 | dV' d0-63 | dO d64-127 | dV' d64-127], 64 rows each
constexpr uint32_t sVpT = 188416;    // V'^T 128 (d_v) x 64; then dv staged (64 rows x 128 bf16, row-major)
constexpr uint32_t sV = 204800;      // V: 64 rows x 128 bf16, plain row-major (bulk copies of its rows)
constexpr uint32_t sF = 221184;      // fp32: G, exp(G), dec, beta [64 each]
constexpr uint32_t sRed = sF + 1024; // fp32 reductions (below)
constexpr int kRedCol = 0;           //   [4 kinds][4 lane quarters][64]: dgamma gamma, ddec, t1, t2
constexpr int kRedRowE = 1024;       //   [2 sources][4 column groups][64]: row sums of dGam * Gam
constexpr int kRedColE = 1536;       //   [4 quarters][64]: column sums of dGam * Gam
constexpr int kRedRowB = 1792;       //   [4 column groups][64]: sum_s dL KK Gam
constexpr int kRedMisc = 2048;       //   [20]: scan carry, gate sums, <D, H> per warp for two heads
constexpr int kGate0 = 256;          // warps 8 and 9 (threads 256-319) scan the gates and reduce dg, dbeta
constexpr uint32_t sCtl = sRed + 8448;
constexpr uint32_t kTcSmem = sCtl + 256 + 1024;
static_assert(kTcSmem <= 232448, "shared memory over the per-block limit");

// ---- TMEM columns (512: one CTA per SM) ----
constexpr uint32_t tQK = 0;     // lanes 0-63: Q K^T [r][s]; lanes 64-127: K K^T [r][s]
constexpr uint32_t tDQ = 64;    // dq^T [k][r], summed over the group's heads
constexpr uint32_t tDK = 128;   // dk^T [k][s]
constexpr uint32_t tA = 192;    // -S W^T, then Y_U^T
constexpr uint32_t tB = 256;    // dO^T P, then H Y_U^T
constexpr uint32_t tC = 320;    // D^T K^T, then [dP_raw; dL_raw]
constexpr uint32_t tE = 384;    // H dO^T, then A^T dL_raw (lanes 64-127)
constexpr uint32_t tF = 448;    // D V'^T

// Loads of a head's tiles, in groups issued as their slots free up in the
// head before: A (D, -W^T) once phase 2's products are done, B (S, U^T, A^T,
// V) and C (P) once phase 3's are.
struct TcCtl {
  uint64_t loadA, loadB, loadC, ph[5];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint8_t* tc_smem_base() {
  extern __shared__ uint8_t smem_raw[];
  return smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
}

// K-major operand (rows run along M or N, 64 K-elements a row per panel):
// K step ks (16 elements) of a tile whose 64-wide K panels are panel_bytes apart.
__device__ __forceinline__ uint64_t dk_(uint32_t base, int ks, uint32_t panel_bytes) {
  return sdesc_sw128(base + (uint32_t)(ks >> 2) * panel_bytes + (uint32_t)(ks & 3) * 32u, 16, 1024);
}
// MN-major operand (rows run along K, 64 M/N-elements a row per block; blocks
// lbo bytes apart): K step ks = 16 rows.
__device__ __forceinline__ uint64_t dmn_(uint32_t base, int ks, uint32_t lbo) {
  return sdesc_sw128(base + (uint32_t)ks * 2048u, lbo, 1024);
}

__device__ __forceinline__ bool tc_wait(TcCtl* c, int b, uint32_t parity) {
  return wait_phase(&c->ph[b], parity, &c->abort, 200 + b);
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&x)[32]) {
  uint32_t a[16], b[16];
  tmem_ld16(taddr, a);
  tmem_ld16(taddr + 16, b);
  tmem_ld_wait(a, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[i] = __uint_as_float(a[i]);
    x[16 + i] = __uint_as_float(b[i]);
  }
}
// One recursive-halving step of a column sum over the lanes of a warp (see
// butterfly16): lanes with bit OFF set keep the upper half of their values.
template <int OFF>
__device__ __forceinline__ void butterfly_step16(float (&x)[16], int lane) {
  const bool up = (lane & OFF) != 0;
#pragma unroll
  for (int i = 0; i < OFF; ++i) {
    const float send = up ? x[i] : x[i + OFF];
    const float keep = up ? x[i + OFF] : x[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
  }
}

// 32 fp16 values (x, optionally scaled per column) as row `row` of an fp16
// tile, columns c0 .. c0 + 31 (c0 a multiple of 8, within one 64-wide panel).
__device__ __forceinline__ void row_f16(uint32_t panel, int row, int c0, const float (&x)[32], float& mx) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx = absmax_nan(absmax_nan(mx, x[8 * q + 2 * e]), x[8 * q + 2 * e + 1]);
      w[e] = pack_f16x2(x[8 * q + 2 * e], x[8 * q + 2 * e + 1]);
    }
    st_shared_v4(panel + sw128_offset((uint32_t)row, (uint32_t)((c0 >> 3) + q)), w[0], w[1], w[2], w[3]);
  }
}

// Element (row, col) of a one-panel fp16 tile.
__device__ __forceinline__ uint32_t el(uint32_t panel, int row, int col) {
  return panel + sw128_offset((uint32_t)row, (uint32_t)(col >> 3)) + (uint32_t)(col & 7) * 2u;
}
__device__ __forceinline__ float ld_h(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ void st_h(uint32_t addr, float x) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(__half_as_ushort(__float2half_rn(x))) : "memory");
}

// 64 rows x 128 bf16 of a [tokens, heads, 128] tensor into two fp16 panels
// (panel stride pstride; rows >= cv are zero), in two halves: the loads into
// registers (issued together, and before any row scale is known), then the
// conversion and the stores.
template <int NT>
struct RowLoads {
  uint4 raw[64 * 16 / NT];
};
template <int NT>
__device__ __forceinline__ void rows_load(RowLoads<NT>& L, const __nv_bfloat16* src, int64_t t0, int heads, int head,
                                          int cv) {
#pragma unroll
  for (int u = 0; u < 64 * 16 / NT; ++u) {
    const int idx = threadIdx.x + u * NT, r = idx >> 4, c = idx & 15;
    L.raw[u] = make_uint4(0, 0, 0, 0);
    if (r < cv) L.raw[u] = *reinterpret_cast<const uint4*>(src + ((size_t)(t0 + r) * heads + head) * kDim + c * 8);
  }
}
template <int NT>
__device__ __forceinline__ void rows_store(const RowLoads<NT>& L, uint32_t base, uint32_t pstride, float& mx,
                                           const float* row_scale = nullptr) {
#pragma unroll
  for (int u = 0; u < 64 * 16 / NT; ++u) {
    const int idx = threadIdx.x + u * NT, r = idx >> 4, c = idx & 15;
    const uint32_t w[4] = {L.raw[u].x, L.raw[u].y, L.raw[u].z, L.raw[u].w};
    const float sc = row_scale ? row_scale[r] : 1.f;
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      mx = absmax_nan(absmax_nan(mx, f.x * sc), f.y * sc);
      o[e] = pack_f16x2(f.x * sc, f.y * sc);
    }
    st_shared_v4(base + (uint32_t)(c >> 3) * pstride + sw128_offset((uint32_t)r, (uint32_t)(c & 7)), o[0], o[1],
                 o[2], o[3]);
  }
}

// 16-column variants (the chunk-local kernel: 16 warps, a thread takes 16 of a
// 64-column accumulator)
__device__ __forceinline__ void ld16f(uint32_t taddr, float (&x)[16]) {
  uint32_t a[16];
  tmem_ld16(taddr, a);
  tmem_ld_wait(a);
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(a[i]);
}
// Two 16-column loads in flight together, one wait.
__device__ __forceinline__ void ld16f2(uint32_t ta, float (&x)[16], uint32_t tb, float (&y)[16]) {
  uint32_t a[16], b[16];
  tmem_ld16(ta, a);
  tmem_ld16(tb, b);
  tmem_ld_wait(a, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[i] = __uint_as_float(a[i]);
    y[i] = __uint_as_float(b[i]);
  }
}
__device__ __forceinline__ void st16f(uint32_t taddr, const float (&x)[16]) {
  uint32_t a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = __float_as_uint(x[i]);
  tmem_st16(taddr, a);
}
// Column sums of x[0..15] over the 32 lanes of a warp: lanes l and l + 16 return
// the sum of column l (the halves added first, then recursive halving).
__device__ __forceinline__ float butterfly16(float (&x)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], 16);
  butterfly_step16<8>(x, lane);
  butterfly_step16<4>(x, lane);
  butterfly_step16<2>(x, lane);
  butterfly_step16<1>(x, lane);
  return x[0];
}
__device__ __forceinline__ void row_f16_16(uint32_t panel, int row, int c0, const float (&x)[16], float& mx) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx = absmax_nan(absmax_nan(mx, x[8 * q + 2 * e]), x[8 * q + 2 * e + 1]);
      w[e] = pack_f16x2(x[8 * q + 2 * e], x[8 * q + 2 * e + 1]);
    }
    st_shared_v4(panel + sw128_offset((uint32_t)row, (uint32_t)((c0 >> 3) + q)), w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ bool tc_chunk_rows(const Problem& p, int gc, int& n, int64_t& t0, int& cv) {
  if (p.cu) {
    const int4 ci = p.chunk_info[gc];
    n = ci.x;
    cv = ci.y;
    t0 = (int64_t)(((uint64_t)(uint32_t)ci.w << 32) | (uint32_t)ci.z);
  } else {
    const int cps = chunks_of(p.T_row);
    n = gc / cps;
    t0 = (int64_t)n * p.T_row + (int64_t)(gc - n * cps) * kChunk;
    cv = (int)min((int64_t)kChunk, (int64_t)(n + 1) * p.T_row - t0);
  }
  return n >= 0 && n < p.n_seqs && cv > 0 && cv <= kChunk;
}

__global__ void __launch_bounds__(kLocThreads, 1) bwd_local_tc_kernel(const Problem p, const BwdArgs b) {
  uint8_t* sm = tc_smem_base();
  const uint32_t s0 = smem_u32(sm);
  TcCtl* ctl = reinterpret_cast<TcCtl*>(sm + sCtl);
  float* sG = reinterpret_cast<float*>(sm + sF);
  float* sGam = sG + 64;
  float* sDec = sG + 128;
  float* sBeta = sG + 192;
  float* red = reinterpret_cast<float*>(sm + sRed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, h = warp >> 2;         // TMEM lane quarter, group of 16 columns
  const int d = 32 * q + lane;                   // this thread's TMEM lane
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const int gc = (int)(blockIdx.x / (unsigned)p.h_qk), iq = (int)(blockIdx.x % (unsigned)p.h_qk);
  if (tid == 0) {
    mbar_init(&ctl->loadA, 1);
    mbar_init(&ctl->loadB, 1);
    mbar_init(&ctl->loadC, 1);
    for (int i = 0; i < 5; ++i) mbar_init(&ctl->ph[i], 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  int n, cv;
  int64_t t0;
  const bool rows_ok = tc_chunk_rows(p, gc, n, t0, cv);
  tc_fence_before();
  const bool skip = __syncthreads_or(tid == 0 && (!rows_ok || earlier_failure(p.status)));
  tc_fence_after();
  const uint32_t tmem = ctl->tmem + lane_base;
  const int j_lo = (int)(((int64_t)iq * p.h_v + p.h_qk - 1) / p.h_qk);
  const int j_hi = (int)(((int64_t)(iq + 1) * p.h_v + p.h_qk - 1) / p.h_qk);
  float mx = 0.f;
  bool ok = !skip;
  int n_heads = 0;
  // (one thread) head jj's tile groups
  auto issue_A = [&](int jj) {
    const size_t slot = (size_t)gc * p.h_v + jj;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&ctl->loadA, 32768u + 16384u);
    bulk_load(sm + sD, b.dstate + slot * 32768u, 32768u, &ctl->loadA);
    bulk_load(sm + sWt, p.wy + slot * kRecBytes + kRecWn, 16384u, &ctl->loadA);
  };
  auto issue_B = [&](int jj) {  // (the 32 lanes of one warp: V's rows spread over them)
    const size_t slot = (size_t)gc * p.h_v + jj;
    if (lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&ctl->loadB, 32768u + 16384u + 8192u + (uint32_t)cv * 256u);
      bulk_load(sm + sS, p.hchunk + slot * 32768u, 32768u, &ctl->loadB);
      bulk_load(sm + sUt, p.wy + slot * kRecBytes + kRecU, 16384u, &ctl->loadB);
      bulk_load(sm + sAT, p.wyA + slot * 8192u, 8192u, &ctl->loadB);
    }
    __syncwarp();
    const uint8_t* vrow = reinterpret_cast<const uint8_t*>(p.v) + ((size_t)t0 * p.h_v + jj) * (kDim * 2);
    for (int r = lane; r < cv; r += 32)
      bulk_load(sm + sV + r * 256, vrow + (size_t)r * p.h_v * (kDim * 2), 256u, &ctl->loadB);
  };
  auto issue_C = [&](int jj) {
    const size_t slot = (size_t)gc * p.h_v + jj;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&ctl->loadC, 8192u);
    bulk_load(sm + sP, p.wy + slot * kRecBytes + kRecP, 8192u, &ctl->loadC);
  };
  if (ok) {
    // the first head's tiles need nothing of Q and K: their copies start first
    if (j_lo < j_hi) {
      if (tid == 0) {
        issue_A(j_lo);
        issue_C(j_lo);
      }
      if (warp == 0) issue_B(j_lo);
    }
    // dq^T and dk^T accumulators start at zero
    {
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.f;
      st16f(tmem + tDQ + 16 * h, z);
      st16f(tmem + tDK + 16 * h, z);
    }
    // Q, K and the first head's dO rows: every load in flight before any store
    RowLoads<kLocThreads> lq, lk, ldo;
    rows_load(lq, reinterpret_cast<const __nv_bfloat16*>(p.q), t0, p.h_qk, iq, cv);
    rows_load(lk, reinterpret_cast<const __nv_bfloat16*>(p.k), t0, p.h_qk, iq, cv);
    if (j_lo < j_hi) rows_load(ldo, reinterpret_cast<const __nv_bfloat16*>(b.dout), t0, p.h_v, j_lo, cv);
    rows_store(lq, s0 + sQK, 16384, mx);
    rows_store(lk, s0 + sQK + 8192, 16384, mx);
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // [Q; K] K^T: Q K^T on lanes 0-63, K K^T on lanes 64-127
      tc_fence_after();
      const uint32_t id = idesc_f16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(ctl->tmem + tQK, dk_(s0 + sQK, ks, 16384), dk_(s0 + sQK + 8192, ks, 16384), id, ks > 0);
      mma_commit(&ctl->ph[0]);
    }
    if (j_lo < j_hi) rows_store(ldo, s0 + sDOV, 16384, mx);
  }
  // The gate threads: row gr of the chunk.  They hold this head's g and beta (prefetched
  // during the head before); a head's dg and dbeta are reduced while the next head's
  // first products run.
  const bool gate_thr = tid >= kGate0 && tid < kGate0 + 64;
  const int gr = tid - kGate0, gw = warp - (kGate0 >> 5);
  float g_cur = 0.f, b_cur = 0.f;
  if (gate_thr && j_lo < j_hi && gr < cv) {
    g_cur = p.g[(size_t)(t0 + gr) * p.h_v + j_lo];
    b_cur = p.beta[(size_t)(t0 + gr) * p.h_v + j_lo];
  }
  // dG, dg = its reverse cumulative sum, and dbeta of head jj from the epilogues' sums
  // and that head's gates in sBeta, sGam, sDec; dh_par selects its <D, H> slots.
  auto gates = [&](int jj, uint32_t dh_par) {
    const int r = gr;
    auto col = [&](int kind) {
      return red[kRedCol + (kind * 4 + 0) * 64 + r] + red[kRedCol + (kind * 4 + 1) * 64 + r] +
             red[kRedCol + (kind * 4 + 2) * 64 + r] + red[kRedCol + (kind * 4 + 3) * 64 + r];
    };
    const float t2 = col(3);
    float erow = 0.f;
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) erow += red[kRedRowE + g8 * 64 + r];
    const float ecol = red[kRedColE + r] + red[kRedColE + 64 + r] + red[kRedColE + 128 + r] +
                       red[kRedColE + 192 + r];
    const float ddec = col(1) * sDec[r];
    float dG = col(0) + sBeta[r] * t2 * sGam[r] + erow - ecol - ddec;
    const float dbeta = col(2) + sGam[r] * t2 + red[kRedRowB + r] + red[kRedRowB + 64 + r] +
                        red[kRedRowB + 128 + r] + red[kRedRowB + 192 + r];
    float dd = ddec;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
    if (lane == 0) red[kRedMisc + 1 + gw] = dd;
    named_bar_sync(1, 64);
    if (r == 63) {
      float dgc = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) dgc += red[kRedMisc + 4 + 8 * dh_par + w];
      dG += dgc * sGam[63] + red[kRedMisc + 1] + red[kRedMisc + 2];
    }
    float x = dG;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x += y;
    }
    if (gw == 1 && lane == 0) red[kRedMisc + 3] = x;
    named_bar_sync(1, 64);
    if (gw == 0) x += red[kRedMisc + 3];
    if (r < cv) {
      b.dg[(size_t)(t0 + r) * p.h_v + jj] = x;
      b.dbeta[(size_t)(t0 + r) * p.h_v + jj] = dbeta;
    }
  };
  for (int j = j_lo; ok && j < j_hi; ++j, ++n_heads) {
    const uint32_t par = (uint32_t)(n_heads & 1);
    // the previous head's last products (they read K and dKK) are done
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    // (this head's tiles came during the head before)
    const bool landed = mbar_wait(&ctl->loadA, par, kWaitLimitNs) && mbar_wait(&ctl->loadB, par, kWaitLimitNs) &&
                        mbar_wait(&ctl->loadC, par, kWaitLimitNs);
    if (!landed) atomicCAS(&ctl->abort, 0, kDetTmaWait);
    if (n_heads == 0 && !tc_wait(ctl, 0, 0)) ok = false;
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!landed || !ok)) {
      ok = false;
      break;
    }
    // ---- phase 1: -S W^T, dO^T P, D^T K^T, H dO^T ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t t = ctl->tmem;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(t + tA, dk_(s0 + sS, ks, 16384), dmn_(s0 + sWt, ks, 16384), idesc_f16(128, 64, false, true), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tB, dmn_(s0 + sDOV, ks, 16384), dmn_(s0 + sP, ks, 8192), idesc_f16(128, 64, true, true), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(t + tC, dmn_(s0 + sD, ks, 16384), dk_(s0 + sQK + 8192, ks, 16384), idesc_f16(128, 64, true, false),
                 ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(t + tE, dmn_(s0 + sS, ks, 16384), dk_(s0 + sDOV, ks, 16384), idesc_f16(128, 64, true, false), ks > 0);
      mma_commit(&ctl->ph[1]);
    }
    // the previous head's dg and dbeta while these products run
    if (gate_thr) {
      if (n_heads > 0) gates(j - 1, par ^ 1u);
      // then this head's G = inclusive cumulative gate (two warps, as the forward)
      const int r = gr;
      float x = g_cur;
      sBeta[r] = b_cur;
#pragma unroll
      for (int dd = 1; dd < 32; dd <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, dd);
        if (lane >= dd) x += y;
      }
      if (lane == 31 && gw == 0) red[kRedMisc] = x;
      named_bar_sync(1, 64);
      if (gw == 1) x += red[kRedMisc];
      sG[r] = x;
      sGam[r] = __expf(x);
      named_bar_sync(1, 64);
      sDec[r] = __expf(sG[63] - x);
    }
    // <D, H> = sum D[k][v] S[v][k] (the gradient of gamma_C) while the products run:
    // thread = one 8 x 8 block, rows k0.. of D against rows v0.. of S
    if (tid < 256) {  // 16 x 16 blocks of 8 x 8: the first eight warps
      const int k0 = 8 * (tid >> 4), v0 = 8 * (tid & 15);
      const uint32_t dpanel = s0 + sD + (uint32_t)(v0 >> 6) * 16384u;
      const uint32_t spanel = s0 + sS + (uint32_t)(k0 >> 6) * 16384u;
      float dblk[8][8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const uint4 w = lds_u32x4(dpanel + sw128_offset((uint32_t)(k0 + a), (uint32_t)((v0 & 63) >> 3)));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
          dblk[a][2 * e] = f.x;
          dblk[a][2 * e + 1] = f.y;
        }
      }
      float dh = 0.f;
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) {  // row v0 + bb of S: S[v][k0 .. k0 + 7]
        const uint4 w = lds_u32x4(spanel + sw128_offset((uint32_t)(v0 + bb), (uint32_t)((k0 & 63) >> 3)));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
          dh = fmaf(dblk[2 * e][bb], f.x, fmaf(dblk[2 * e + 1][bb], f.y, dh));
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dh += __shfl_xor_sync(0xffffffffu, dh, o);
      if (lane == 0) red[kRedMisc + 4 + 8 * par + warp] = dh;
    }
    if (!tc_wait(ctl, 1, par)) ok = false;
    tc_fence_after();
    // the previous head's sums are read and this head's gates written before the epilogue
    __syncthreads();
    if (ok) {
      // V'^T = U^T - S W^T (lane = d_v)
      float x[16];
      ld16f(tmem + tA + 16 * h, x);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 u = lds_u32x4(s0 + sUt + sw128_offset((uint32_t)d, (uint32_t)(2 * h + c)));
        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 u2 = __half22float2(*reinterpret_cast<const __half2*>(&uw[e]));
          x[8 * c + 2 * e] += u2.x;
          x[8 * c + 2 * e + 1] += u2.y;
        }
      }
      row_f16_16(s0 + sVpT, d, 16 * h, x, mx);
      // dV'^T = scale dO^T P + diag(dec) applied to D^T K^T's columns; also dV' (rows r)
      float y[16];
      ld16f2(tmem + tB + 16 * h, x, tmem + tC + 16 * h, y);
      const uint32_t dvp = s0 + sDOV + 8192u + (uint32_t)(d >> 6) * 16384u;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] = fmaf(p.scale, x[i], sDec[16 * h + i] * y[i]);
        st_h(el(dvp, 16 * h + i, d & 63), x[i]);
      }
      row_f16_16(s0 + sWt, d, 16 * h, x, mx);
      // H dO^T (lane = d_k): dq^T += scale gamma_r (H dO^T); dgamma_r gamma_r = <Q_r, that>
      ld16f2(tmem + tE + 16 * h, x, tmem + tDQ + 16 * h, y);
      const uint32_t qpanel = s0 + sQK + (uint32_t)(d >> 6) * 16384u;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] *= p.scale * sGam[16 * h + i];
        y[i] += x[i];
        x[i] *= ld_h(el(qpanel, 16 * h + i, d & 63));
      }
      st16f(tmem + tDQ + 16 * h, y);
      {
        const float cs_ = butterfly16(x);
        if (lane < 16) red[kRedCol + (0 * 4 + q) * 64 + 16 * h + lane] = cs_;
      }
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    // ---- phase 2: D V'^T, [dO; dV'] V'^T, dV'^T A ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t t = ctl->tmem;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(t + tF, dk_(s0 + sD, ks, 16384), dmn_(s0 + sVpT, ks, 16384), idesc_f16(128, 64, false, true), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(t + tC, dk_(s0 + sDOV, ks, 16384), dmn_(s0 + sVpT, ks, 16384), idesc_f16(128, 64, false, true),
                 ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tA, dk_(s0 + sWt, ks, 16384), dk_(s0 + sAT, ks, 8192), idesc_f16(128, 64, false, false), ks > 0);
      mma_commit(&ctl->ph[2]);
    }
    if (!tc_wait(ctl, 2, par)) ok = false;
    // the previous head's last products (they read dKK and update dk^T) are done
    if (n_heads > 0 && !tc_wait(ctl, 4, par ^ 1u)) ok = false;
    if (tid == 0 && ok && j + 1 < j_hi) issue_A(j + 1);  // D and -W^T are read
    tc_fence_after();
    // the next head's dO rows, in flight during this epilogue (its slots were last
    // read by phase 2; they are written at the epilogue's end)
    const bool next_do = ok && j + 1 < j_hi;
    uint4 dro[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (next_do) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = tid + u * kLocThreads, r = idx >> 4, c = idx & 15;
        if (r < cv)
          dro[u] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(b.dout) +
                                                   ((size_t)(t0 + r) * p.h_v + j + 1) * kDim + c * 8);
      }
    }
    if (ok) {
      float x[16], y[16];
      // D V'^T (lane = d_k): dk^T += dec_r (.); ddec_r = <K_r, .>
      ld16f2(tmem + tF + 16 * h, x, tmem + tDK + 16 * h, y);
      const uint32_t kpanel = s0 + sQK + 8192u + (uint32_t)(d >> 6) * 16384u;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        y[i] = fmaf(sDec[16 * h + i], x[i], y[i]);
        x[i] *= ld_h(el(kpanel, 16 * h + i, d & 63));
      }
      st16f(tmem + tDK + 16 * h, y);
      {
        const float cs_ = butterfly16(x);
        if (lane < 16) red[kRedCol + (1 * 4 + q) * 64 + 16 * h + lane] = cs_;
      }
      // Y_U^T (lane = d_v): dv = beta_r Y_U; t1_r = <Y_U_r, V_r>; Y_U^T into the U^T slot
      ld16f(tmem + tA + 16 * h, x);
      row_f16_16(s0 + sUt, d, 16 * h, x, mx);
      {  // dv staged in the V'^T slot (read by phase 2), stored in epilogue 3
        const unsigned short* vcol = reinterpret_cast<const unsigned short*>(sm + sV) + d;
        unsigned short* dvcol = reinterpret_cast<unsigned short*>(sm + sVpT) + d;
        unsigned short vb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) vb[i] = vcol[(16 * h + i) * 128];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = 16 * h + i;
          const __nv_bfloat16 dvb = __float2bfloat16_rn(sBeta[r] * x[i]);
          dvcol[r * 128] = *reinterpret_cast<const unsigned short*>(&dvb);
          x[i] = r < cv ? x[i] * __uint_as_float((uint32_t)vb[i] << 16) : 0.f;
        }
      }
      {
        const float cs_ = butterfly16(x);
        if (lane < 16) red[kRedCol + (2 * 4 + q) * 64 + 16 * h + lane] = cs_;
      }
      // [dP_raw; dL_raw] (lane = token r, or 64 + r)
      if (q < 2)
        ld16f2(tmem + tC + 16 * h, x, tmem + tQK + 16 * h, y);
      else
        ld16f(tmem + tC + 16 * h, x);
      if (q < 2) {
        const int r = d;
        float rowsum = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int s = 16 * h + i;
          const float gam = s <= r ? __expf(sG[r] - sG[s]) : 0.f;
          const float dP = s <= r ? p.scale * x[i] : 0.f;
          const float e = dP * y[i] * gam;
          rowsum += e;
          x[i] = dP * gam;
          y[i] = e;
        }
        row_f16_16(s0 + sPG, r, 16 * h, x, mx);
        red[kRedRowE + (0 * 4 + h) * 64 + r] = rowsum;
        {
        const float cs_ = butterfly16(y);
        if (lane < 16) red[kRedColE + q * 64 + 16 * h + lane] = cs_;
      }
      } else {
        row_f16_16(s0 + sP, d - 64, 16 * h, x, mx);
      }
    }
    if (next_do) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = tid + u * kLocThreads, r = idx >> 4, c = idx & 15;
        const uint32_t w[4] = {dro[u].x, dro[u].y, dro[u].z, dro[u].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
          mx = absmax_nan(absmax_nan(mx, f.x), f.y);
          o[e] = pack_f16x2(f.x, f.y);
        }
        st_shared_v4(s0 + sDOV + (uint32_t)(c >> 3) * 16384u + sw128_offset((uint32_t)r, (uint32_t)(c & 7)), o[0], o[1],
                     o[2], o[3]);
      }
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    // ---- phase 3: H Y_U^T; dq^T += K^T (dP*Gam)^T; dk^T += Q^T (dP*Gam); A^T dL_raw ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t t = ctl->tmem;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(t + tB, dmn_(s0 + sS, ks, 16384), dmn_(s0 + sUt, ks, 16384), idesc_f16(128, 64, true, true), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tDQ, dmn_(s0 + sQK + 8192, ks, 16384), dk_(s0 + sPG, ks, 8192), idesc_f16(128, 64, true, false), 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tDK, dmn_(s0 + sQK, ks, 16384), dmn_(s0 + sPG, ks, 8192), idesc_f16(128, 64, true, true), 1);
      // rows 64-127 of this A operand are A^T (rows 0-63 read the tile before it and are discarded)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tE, dk_(s0 + sPG, ks, 16384), dmn_(s0 + sP, ks, 8192), idesc_f16(128, 64, false, true), ks > 0);
      mma_commit(&ctl->ph[3]);
    }
    if (!tc_wait(ctl, 3, par)) ok = false;
    if (warp == 0) {  // S, U^T / Y_U^T, A^T, V and P / dL_raw are read
      if (__all_sync(0xffffffffu, ok) && j + 1 < j_hi) {
        issue_B(j + 1);
        if (lane == 0) issue_C(j + 1);
      }
    }
    tc_fence_after();
    if (ok) {  // dv of this head from its staging rows: 16-byte stores, whole rows per warp
      uint8_t* dvo = reinterpret_cast<uint8_t*>(b.dv);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = tid + u * kLocThreads, r = idx >> 4, c = idx & 15;
        const uint4 w = lds_u32x4(s0 + sVpT + (uint32_t)(r * 256 + c * 16));
        if (r < cv) *reinterpret_cast<uint4*>(dvo + (((size_t)(t0 + r) * p.h_v + j) * kDim) * 2 + c * 16) = w;
      }
    }
    // the next head's g and beta, in flight during this epilogue
    float g_next = 0.f, b_next = 0.f;
    if (gate_thr && j + 1 < j_hi && gr < cv) {
      g_next = p.g[(size_t)(t0 + gr) * p.h_v + j + 1];
      b_next = p.beta[(size_t)(t0 + gr) * p.h_v + j + 1];
    }
    if (ok) {
      float x[16], y[16];
      // Y_W^T = -H Y_U^T (lane = d_k): dk^T += beta_r gamma_r Y_W^T; t2_r = <Y_W_r, K_r>
      ld16f2(tmem + tB + 16 * h, x, tmem + tDK + 16 * h, y);
      const uint32_t kpanel = s0 + sQK + 8192u + (uint32_t)(d >> 6) * 16384u;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 16 * h + i;
        y[i] = fmaf(-sBeta[r] * sGam[r], x[i], y[i]);
        x[i] = -x[i] * ld_h(el(kpanel, r, d & 63));
      }
      st16f(tmem + tDK + 16 * h, y);
      {
        const float cs_ = butterfly16(x);
        if (lane < 16) red[kRedCol + (3 * 4 + q) * 64 + 16 * h + lane] = cs_;
      }
      // dL = -A^T dL_raw, s < r (lanes 64-127: r = lane - 64)
      if (q >= 2) {
        const int r = d - 64;
        ld16f2(tmem + tE + 16 * h, x, tmem + tQK + 16 * h, y);  // y: K K^T [r][s]
        const float br = sBeta[r];
        float rowb = 0.f, rowe = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int s = 16 * h + i;
          const float gam = s < r ? __expf(sG[r] - sG[s]) : 0.f;
          const float dL = s < r ? -x[i] : 0.f;
          const float xb = dL * y[i] * gam;
          rowb += xb;
          rowe += br * xb;
          x[i] = dL * br * gam;
          y[i] = br * xb;
        }
        row_f16_16(s0 + sPG, r, 16 * h, x, mx);
        red[kRedRowB + h * 64 + r] = rowb;
        red[kRedRowE + (1 * 4 + h) * 64 + r] = rowe;
        {
        const float cs_ = butterfly16(y);
        if (lane < 16) red[kRedColE + q * 64 + 16 * h + lane] = cs_;
      }
      }
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    // ---- phase 4: dk^T += K^T (dKK^T + dKK) ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t t = ctl->tmem;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tDK, dmn_(s0 + sQK + 8192, ks, 16384), dk_(s0 + sPG, ks, 8192), idesc_f16(128, 64, true, false), 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(t + tDK, dmn_(s0 + sQK + 8192, ks, 16384), dmn_(s0 + sPG, ks, 8192), idesc_f16(128, 64, true, true), 1);
      mma_commit(&ctl->ph[4]);
    }
    g_cur = g_next;
    b_cur = b_next;
  }
  // the last head's dg and dbeta
  if (ok && n_heads > 0 && gate_thr) gates(j_lo + n_heads - 1, (uint32_t)((n_heads - 1) & 1));
  // ---- dq, dk (bf16) from their accumulators ----
  if (ok && n_heads > 0 && !tc_wait(ctl, 4, (uint32_t)((n_heads - 1) & 1))) ok = false;
  if (ok && n_heads == 0 && !tc_wait(ctl, 0, 0)) ok = false;  // [Q; K] K^T done before TMEM is freed
  tc_fence_after();
  if (__syncthreads_or(!ok) == 0 && !skip) {
    float x[16], y[16];
    ld16f(tmem + tDQ + 16 * h, x);
    ld16f(tmem + tDK + 16 * h, y);
    __nv_bfloat16* dqo = reinterpret_cast<__nv_bfloat16*>(b.dq);
    __nv_bfloat16* dko = reinterpret_cast<__nv_bfloat16*>(b.dk);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = 16 * h + i;
      if (r < cv) {
        const size_t o = ((size_t)(t0 + r) * p.h_qk + iq) * kDim + d;
        dqo[o] = __float2bfloat16_rn(x[i]);
        dko[o] = __float2bfloat16_rn(y[i]);
      }
    }
  }
  if (skip && tid == 0 && !rows_ok) report(p.status, kDevCheck, kDetSegMismatch);
  tc_fence_before();
  __syncthreads();
  if (ctl->abort || (!ok && !skip)) {
    if (tid == 0) report(p.status, kDevTimeout, ctl->abort ? ctl->abort : kDetMmaWait);
    // let copies and MMAs already in flight land before the memory is released
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
    __syncthreads();
  }
  if (!(mx < 65504.f)) report(p.status, kDevCheck, kDetFp16Range);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(ctl->tmem, 512);
  }
}


// ------------------------------------------------------------ per-chunk T' and E
// For one (chunk, value head): T' = -W^T Ktil (the chunk's map of the state
// gradient) and E = scale (diag(gamma) Q)^T dO - W^T Y with Y = scale P^T dO,
// both fp16 in the tile image the chain reads (rows d_k; panels d_k resp. d_v).
// Products (M = 128 rows of d): Y^T = dO^T P; T' = (-W^T) Ktil;
// E = Qg^T dO + (-W^T) Y  (Qg = scale diag(gamma) Q).  Two CTAs per SM.
constexpr uint32_t pWt = 0;        // -W^T record tile 128 (d_k) x 64
constexpr uint32_t pKt = 16384;    // Ktil = diag(dec) K: 64 x 128, panels d_k 0-63 | 64-127 (8 KB)
constexpr uint32_t pQg = 32768;    // Qg: 64 x 128
constexpr uint32_t pDo = 49152;    // dO: 64 x 128
constexpr uint32_t pYt = 65536;    // Y^T: 128 (d_v) x 64
constexpr uint32_t pP = 81920;     // P record tile 64 x 64
constexpr uint32_t pGam = 90112;   // record gates: exp(G) [64], dec [64]
constexpr uint32_t pSc = pGam + 512;   // scale exp(G) [64]
constexpr uint32_t pCtl = pSc + 256;
constexpr uint32_t kPreTcSmem = pCtl + 64 + 1024;
constexpr uint32_t qT = 0, qE = 128;   // TMEM columns: T' [0, 128); Y^T then E [128, 256)

struct PreCtl {
  uint64_t load, mma1, mma2;
  uint32_t tmem;
  int abort;
};

__global__ void __launch_bounds__(kTcThreads, 2) bwd_pre_tc_kernel(const Problem p, const BwdArgs b) {
  uint8_t* sm = tc_smem_base();
  const uint32_t s0 = smem_u32(sm);
  PreCtl* ctl = reinterpret_cast<PreCtl*>(sm + pCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, h = warp >> 2, d = 32 * q + lane;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const int gc = (int)(blockIdx.x / (unsigned)p.h_v), j = (int)(blockIdx.x % (unsigned)p.h_v);
  if (tid == 0) {
    mbar_init(&ctl->load, 1);
    mbar_init(&ctl->mma1, 1);
    mbar_init(&ctl->mma2, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 256);
    tmem_relinquish();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  int n, cv;
  int64_t t0;
  const bool rows_ok = tc_chunk_rows(p, gc, n, t0, cv);
  tc_fence_before();
  const bool skip = __syncthreads_or(tid == 0 && (!rows_ok || earlier_failure(p.status)));
  tc_fence_after();
  const uint32_t tm = ctl->tmem;
  float mx = 0.f;
  bool ok = !skip;
  if (ok) {
    const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
    const uint8_t* rec = p.wy + ((size_t)gc * p.h_v + j) * kRecBytes;
    if (tid == 0) {
      mbar_arrive_expect_tx(&ctl->load, 16384u + 8192u + 512u);
      bulk_load(sm + pWt, rec + kRecWn, 16384u, &ctl->load);
      bulk_load(sm + pP, rec + kRecP, 8192u, &ctl->load);
      bulk_load(sm + pGam, rec + kRecGam, 512u, &ctl->load);
    }
    // all row loads in flight before the gates (which scale K and Q) have landed
    RowLoads<kTcThreads> lo_do, lo_k, lo_q;
    rows_load(lo_do, reinterpret_cast<const __nv_bfloat16*>(b.dout), t0, p.h_v, j, cv);
    rows_load(lo_k, reinterpret_cast<const __nv_bfloat16*>(p.k), t0, p.h_qk, iq, cv);
    rows_load(lo_q, reinterpret_cast<const __nv_bfloat16*>(p.q), t0, p.h_qk, iq, cv);
    rows_store(lo_do, s0 + pDo, 8192, mx);
    if (!mbar_wait(&ctl->load, 0, kWaitLimitNs)) atomicCAS(&ctl->abort, 0, kDetTmaWait);
    float* gam = reinterpret_cast<float*>(sm + pGam);
    float* qsc = reinterpret_cast<float*>(sm + pSc);
    if (tid < 64) qsc[tid] = p.scale * gam[tid];
    __syncthreads();
    rows_store(lo_k, s0 + pKt, 8192, mx, gam + 64);
    rows_store(lo_q, s0 + pQg, 8192, mx, qsc);
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(ctl->abort != 0)) ok = false;
  }
  if (ok && tid == 0) {  // phase 1: Y^T = dO^T P -> E's columns; T' = (-W^T) Ktil
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tm + qE, dmn_(s0 + pDo, ks, 8192), dmn_(s0 + pP, ks, 8192), idesc_f16(128, 64, true, true), ks > 0);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tm + qT, dk_(s0 + pWt, ks, 16384), dmn_(s0 + pKt, ks, 8192), idesc_f16(128, 128, false, true), ks > 0);
    mma_commit(&ctl->mma1);
  }
  if (ok) {
    if (!wait_phase(&ctl->mma1, 0, &ctl->abort, 220)) ok = false;
    tc_fence_after();
  }
  if (__syncthreads_or(!ok)) ok = false;
  if (ok) {  // Y^T (lane = d_v) scaled, into its K-major tile
    float x[32];
    ld32(tm + lane_base + qE + 32 * h, x);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] *= p.scale;
    row_f16(s0 + pYt, d, 32 * h, x, mx);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (ok && tid == 0) {  // phase 2: E = Qg^T dO + (-W^T) Y
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tm + qE, dmn_(s0 + pQg, ks, 8192), dmn_(s0 + pDo, ks, 8192), idesc_f16(128, 128, true, true), ks > 0);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tm + qE, dk_(s0 + pWt, ks, 16384), dk_(s0 + pYt, ks, 16384), idesc_f16(128, 128, false, false), 1);
    mma_commit(&ctl->mma2);
  }
  const size_t slot = ((size_t)gc * p.h_v + j) * 32768u;
  // T' rows (lane = d_k out) while E's products run: columns 64 h .. 64 h + 63 (panel h)
  auto store_rows = [&](uint32_t col0, uint8_t* dst) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float x[32];
      ld32(tm + lane_base + col0 + 64 * h + 32 * half, x);
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        mx = absmax_nan(absmax_nan(mx, x[2 * e]), x[2 * e + 1]);
        w[e] = pack_f16x2(x[2 * e], x[2 * e + 1]);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(dst + (size_t)h * 16384u + sw128_offset((uint32_t)d, (uint32_t)(4 * half + c))) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
  };
  if (ok) store_rows(qT, b.tmat + slot);
  if (ok) {
    if (!wait_phase(&ctl->mma2, 0, &ctl->abort, 221)) ok = false;
    tc_fence_after();
  }
  if (__syncthreads_or(!ok)) ok = false;
  if (ok) store_rows(qE, b.emat + slot);
  if (skip && tid == 0 && !rows_ok) report(p.status, kDevCheck, kDetSegMismatch);
  tc_fence_before();
  __syncthreads();
  if (!skip && (!ok || ctl->abort)) {
    if (tid == 0) report(p.status, kDevTimeout, ctl->abort ? ctl->abort : kDetMmaWait);
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
    __syncthreads();
  }
  if (!(mx < 65504.f)) report(p.status, kDevCheck, kDetFp16Range);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 256);
  }
}

// ------------------------------------------------------------ state-gradient chain
// The final pass over one segment's chunks in reverse, D <- gamma_C D + E_c +
// T'_c D_c: the product on tcgen05 (M = d_k out, N = d_v, K = d_k in; A = T'
// from the record, B = D's fp16 copy in shared memory), D itself in fp32
// registers (thread: TMEM lane = row d_k, 64 of the 128 columns).  D starts
// from dh_T (a sequence's last segment) or from the combine's D_end; every
// chunk's D is written before its step (fp16 tile image), and dh0 for a
// sequence's first segment.  Without context parallelism every sequence is
// one segment.  (The segments' transitions and local offsets for the combine
// come from bwd_chain2_tc_kernel.)
constexpr uint32_t cT = 0;          // 2 x T' (32 KB): rows d_k out, panels d_k in 0-63 | 64-127
constexpr uint32_t cE = 65536;      // 2 x E (32 KB): rows d_k, panels d_v
constexpr uint32_t cD = 131072;     // D's fp16 copy: rows d_k (K), panels d_v 0-63 | 64-127
constexpr uint32_t cCtl = 163840;
constexpr uint32_t kChainSmem = cCtl + 128 + 1024;

struct ChCtl {
  uint64_t load[2], mma;
  uint32_t tmem;
  int abort;
  SegInfo si;
  int ok;
};

__global__ void __launch_bounds__(kTcThreads, 1) bwd_chain_tc_kernel(const Problem p, const BwdArgs b) {
  uint8_t* sm = tc_smem_base();
  const uint32_t s0 = smem_u32(sm);
  ChCtl* ctl = reinterpret_cast<ChCtl*>(sm + cCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, h = warp >> 2, k = 32 * q + lane;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const int j = blockIdx.y;
  const int seg = (int)blockIdx.x;
  if (warp == 1) {
    SegInfo si;
    const bool okseg = locate_segment(p, seg, si);
    if (lane == 0) {
      ctl->si = si;
      ctl->ok = okseg;
    }
  }
  if (tid == 0) {
    mbar_init(&ctl->load[0], 1);
    mbar_init(&ctl->load[1], 1);
    mbar_init(&ctl->mma, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 128);
    tmem_relinquish();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  tc_fence_before();
  const bool failed = __syncthreads_or(tid == 0 && earlier_failure(p.status));
  tc_fence_after();
  const uint32_t tm = ctl->tmem;
  const SegInfo si = ctl->si;
  bool run = !failed && ctl->ok;
  if (!failed && !ctl->ok && tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
  const bool last_seg = si.s == si.n_seg - 1;
  int c0 = run ? seq_first_chunk(p, si.n) + si.cb : 0, nc = run ? si.ce - si.cb : 0;
  if (run && (c0 < 0 || c0 + nc > p.n_chunks_total)) {  // the chunk index disagrees with the plan
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    run = false;
    c0 = nc = 0;
  }
  const size_t mat = (size_t)kDim * kDim;
  const size_t head_seg = ((size_t)(si.seg_base + si.s) * p.h_v + j) * mat;
  float D[64];  // row k, columns 64 h .. 64 h + 63
  if (run) {
    if (!last_seg) {  // D_end of this segment from the combine, stored transposed (rows d_v)
      const float* src = p.Sstart + head_seg;
#pragma unroll
      for (int e = 0; e < 64; ++e) D[e] = src[(size_t)(64 * h + e) * kDim + k];
    } else if (b.dhT) {
      const float4* src = reinterpret_cast<const float4*>(b.dhT + ((size_t)si.n * p.h_v + j) * mat + (size_t)k * kDim + 64 * h);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float4 v4 = src[e];
        D[4 * e] = v4.x;
        D[4 * e + 1] = v4.y;
        D[4 * e + 2] = v4.z;
        D[4 * e + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 64; ++e) D[e] = 0.f;
    }
  }
  float mx = 0.f;
  // D's fp16 copy as row k of the tile (panel h), and as chunk c's record when asked
  auto store_d = [&](uint8_t* global_row) {
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      mx = absmax_nan(absmax_nan(mx, D[2 * e]), D[2 * e + 1]);
      w[e] = pack_f16x2(D[2 * e], D[2 * e + 1]);
    }
    const uint32_t panel = s0 + cD + (uint32_t)h * 16384u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      st_shared_v4(panel + sw128_offset((uint32_t)k, (uint32_t)c), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      if (global_row)
        *reinterpret_cast<uint4*>(global_row + sw128_offset((uint32_t)k, (uint32_t)c)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
  };
  auto issue = [&](int it) {  // T' (and E) of step it into buffer it & 1 (one thread)
    const int c = c0 + nc - 1 - it;
    const size_t slot = ((size_t)c * p.h_v + j) * 32768u;
    const uint32_t buf = (uint32_t)(it & 1) * 32768u;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&ctl->load[it & 1], 65536u);
    bulk_load(sm + cT + buf, b.tmat + slot, 32768u, &ctl->load[it & 1]);
    bulk_load(sm + cE + buf, b.emat + slot, 32768u, &ctl->load[it & 1]);
  };
  if (tid == 0 && nc > 0) issue(0);
  bool ok = true;
  if (nc > 0) {
    // the first step's D_c is D itself
    store_d(b.dstate + ((size_t)(c0 + nc - 1) * p.h_v + j) * 32768u + (size_t)h * 16384u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  for (int it = 0; it < nc && ok; ++it) {
    const int c = c0 + nc - 1 - it;
    const uint32_t buf = (uint32_t)(it & 1) * 32768u;
    const float gC = reinterpret_cast<const float*>(p.wy + ((size_t)c * p.h_v + j) * kRecBytes + kRecGam)[63];
    if (!mbar_wait(&ctl->load[it & 1], (uint32_t)((it >> 1) & 1), kWaitLimitNs)) atomicCAS(&ctl->abort, 0, kDetTmaWait);
    if (tid == 0 && !ctl->abort) {  // T'_c D_c
      tc_fence_after();
      const uint32_t id = idesc_f16(128, 128, false, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tm, dk_(s0 + cT + buf, ks, 16384), dmn_(s0 + cD, ks, 16384), id, ks > 0);
      mma_commit(&ctl->mma);
      if (it + 1 < nc) issue(it + 1);  // buffer (it + 1) & 1 was last read in step it - 1
    }
    // E_c and gamma_C D while the product runs
    {
      const uint32_t epanel = s0 + cE + buf + (uint32_t)h * 16384u;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 w = lds_u32x4(epanel + sw128_offset((uint32_t)k, (uint32_t)c8));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
          D[8 * c8 + 2 * e] = fmaf(gC, D[8 * c8 + 2 * e], f.x);
          D[8 * c8 + 2 * e + 1] = fmaf(gC, D[8 * c8 + 2 * e + 1], f.y);
        }
      }
    }
    if (!wait_phase(&ctl->mma, (uint32_t)(it & 1), &ctl->abort, 210)) ok = false;
    tc_fence_after();
    if (__syncthreads_or(!ok || ctl->abort)) {
      ok = false;
      break;
    }
    {
      float a[32];
      ld32(tm + lane_base + 64 * h, a);
#pragma unroll
      for (int e = 0; e < 32; ++e) D[e] += a[e];
      ld32(tm + lane_base + 64 * h + 32, a);
#pragma unroll
      for (int e = 0; e < 32; ++e) D[32 + e] += a[e];
    }
    // D_{c-1} for the next step (and as the previous chunk's record)
    if (it + 1 < nc)
      store_d(b.dstate + ((size_t)(c - 1) * p.h_v + j) * 32768u + (size_t)h * 16384u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  }
  if (run && ok && !ctl->abort) {
    if (si.s == 0 && b.dh0) {
      float4* dst = reinterpret_cast<float4*>(b.dh0 + ((size_t)si.n * p.h_v + j) * mat + (size_t)k * kDim + 64 * h);
#pragma unroll
      for (int e = 0; e < 16; ++e) dst[e] = make_float4(D[4 * e], D[4 * e + 1], D[4 * e + 2], D[4 * e + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (ctl->abort || !ok) {
    if (tid == 0) report(p.status, kDevTimeout, ctl->abort ? ctl->abort : kDetMmaWait);
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
    __syncthreads();
  }
  if (!(mx < 65504.f)) report(p.status, kDevCheck, kDetFp16Range);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 128);
  }
}


// The preprocessing's two chains of one segment in one CTA: the transition X0
// (from I, no E) and the local offset X1 (from 0, with E) share each step's T'
// as the A operand of one N = 256 product T' [X0 | X1]; both stay in fp32
// registers.  Stored transposed for the combine (p.R, p.Sloc).
constexpr uint32_t c2T = 0;          // 2 x T' (32 KB)
constexpr uint32_t c2E = 65536;      // 2 x E (32 KB)
constexpr uint32_t c2D = 131072;     // [X0 | X1] fp16: four 64-column panels of 128 rows (16 KB each)
constexpr uint32_t c2Ctl = 196608;
constexpr uint32_t kChain2Smem = c2Ctl + 128 + 1024;

__global__ void __launch_bounds__(kTcThreads, 1) bwd_chain2_tc_kernel(const Problem p, const BwdArgs b) {
  uint8_t* sm = tc_smem_base();
  const uint32_t s0 = smem_u32(sm);
  ChCtl* ctl = reinterpret_cast<ChCtl*>(sm + c2Ctl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, h = warp >> 2, k = 32 * q + lane;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const int j = blockIdx.y, seg = blockIdx.x;
  if (warp == 1) {
    SegInfo si;
    const bool okseg = locate_segment(p, seg, si);
    if (lane == 0) {
      ctl->si = si;
      ctl->ok = okseg;
    }
  }
  if (tid == 0) {
    mbar_init(&ctl->load[0], 1);
    mbar_init(&ctl->load[1], 1);
    mbar_init(&ctl->mma, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, 256);
    tmem_relinquish();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  tc_fence_before();
  const bool failed = __syncthreads_or(tid == 0 && earlier_failure(p.status));
  tc_fence_after();
  const uint32_t tm = ctl->tmem;
  const SegInfo si = ctl->si;
  bool run = !failed && ctl->ok;
  if (!failed && !ctl->ok && tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
  if (run && si.s == 0) run = false;  // segment 0 is taken by the final pass
  int c0 = run ? seq_first_chunk(p, si.n) + si.cb : 0, nc = run ? si.ce - si.cb : 0;
  if (run && (c0 < 0 || c0 + nc > p.n_chunks_total)) {  // the chunk index disagrees with the plan
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    run = false;
    c0 = nc = 0;
  }
  const size_t mat = (size_t)kDim * kDim;
  const size_t head_seg = ((size_t)(si.seg_base + si.s) * p.h_v + j) * mat;
  float X0[64], X1[64];  // row k, columns 64 h .. 64 h + 63
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    X0[e] = (64 * h + e == k) ? 1.f : 0.f;
    X1[e] = 0.f;
  }
  float mx = 0.f;
  auto store_x = [&]() {  // both as row k of their tiles (panels h and 2 + h)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const float* X = m ? X1 : X0;
      const uint32_t panel = s0 + c2D + (uint32_t)(2 * m + h) * 16384u;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          mx = absmax_nan(absmax_nan(mx, X[8 * c + 2 * e]), X[8 * c + 2 * e + 1]);
          w[e] = pack_f16x2(X[8 * c + 2 * e], X[8 * c + 2 * e + 1]);
        }
        st_shared_v4(panel + sw128_offset((uint32_t)k, (uint32_t)c), w[0], w[1], w[2], w[3]);
      }
    }
  };
  auto issue = [&](int it) {  // T' and E of step it into buffer it & 1 (one thread)
    const int c = c0 + nc - 1 - it;
    const size_t slot = ((size_t)c * p.h_v + j) * 32768u;
    const uint32_t buf = (uint32_t)(it & 1) * 32768u;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&ctl->load[it & 1], 65536u);
    bulk_load(sm + c2T + buf, b.tmat + slot, 32768u, &ctl->load[it & 1]);
    bulk_load(sm + c2E + buf, b.emat + slot, 32768u, &ctl->load[it & 1]);
  };
  if (tid == 0 && nc > 0) issue(0);
  if (nc > 0) {
    store_x();
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  bool ok = true;
  for (int it = 0; it < nc && ok; ++it) {
    const int c = c0 + nc - 1 - it;
    const uint32_t buf = (uint32_t)(it & 1) * 32768u;
    const float gC = reinterpret_cast<const float*>(p.wy + ((size_t)c * p.h_v + j) * kRecBytes + kRecGam)[63];
    if (!mbar_wait(&ctl->load[it & 1], (uint32_t)((it >> 1) & 1), kWaitLimitNs)) atomicCAS(&ctl->abort, 0, kDetTmaWait);
    if (tid == 0 && !ctl->abort) {  // T'_c [X0 | X1]
      tc_fence_after();
      const uint32_t id = idesc_f16(128, 256, false, true);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tm, dk_(s0 + c2T + buf, ks, 16384), dmn_(s0 + c2D, ks, 16384), id, ks > 0);
      mma_commit(&ctl->mma);
      if (it + 1 < nc) issue(it + 1);  // buffer (it + 1) & 1 was last read in step it - 1
    }
    {  // gamma_C X0, gamma_C X1 + E_c while the product runs
      const uint32_t epanel = s0 + c2E + buf + (uint32_t)h * 16384u;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 w = lds_u32x4(epanel + sw128_offset((uint32_t)k, (uint32_t)c8));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
          X1[8 * c8 + 2 * e] = fmaf(gC, X1[8 * c8 + 2 * e], f.x);
          X1[8 * c8 + 2 * e + 1] = fmaf(gC, X1[8 * c8 + 2 * e + 1], f.y);
        }
      }
#pragma unroll
      for (int e = 0; e < 64; ++e) X0[e] *= gC;
    }
    if (!wait_phase(&ctl->mma, (uint32_t)(it & 1), &ctl->abort, 211)) ok = false;
    tc_fence_after();
    if (__syncthreads_or(!ok || ctl->abort)) {
      ok = false;
      break;
    }
    {
      float a[32];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float* X = m ? X1 : X0;
        ld32(tm + lane_base + 128 * m + 64 * h, a);
#pragma unroll
        for (int e = 0; e < 32; ++e) X[e] += a[e];
        ld32(tm + lane_base + 128 * m + 64 * h + 32, a);
#pragma unroll
        for (int e = 0; e < 32; ++e) X[32 + e] += a[e];
      }
    }
    if (it + 1 < nc) store_x();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  }
  if (run && ok && !ctl->abort) {  // transposed (rows d_v, or the transition's column index) for the combine
#pragma unroll
    for (int e = 0; e < 64; ++e) {
      p.R[head_seg + (size_t)(64 * h + e) * kDim + k] = X0[e];
      p.Sloc[head_seg + (size_t)(64 * h + e) * kDim + k] = X1[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (ctl->abort || !ok) {
    if (tid == 0) report(p.status, kDevTimeout, ctl->abort ? ctl->abort : kDetMmaWait);
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
    __syncthreads();
  }
  if (!(mx < 65504.f)) report(p.status, kDevCheck, kDetFp16Range);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 256);
  }
}

}  // namespace

cudaError_t bwd_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(bwd_pre_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPreTcSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChainSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_chain2_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChain2Smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_local_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  return e;
}

cudaError_t launch_bwd_pre_tc(const Problem& p, const BwdArgs& b, cudaStream_t st) {
  const unsigned grid = (unsigned)p.n_chunks_total * (unsigned)p.h_v;
  return launch_kernel(bwd_pre_tc_kernel, dim3(grid), dim3(kTcThreads), kPreTcSmem, st, true, p, b);
}

cudaError_t launch_bwd_chain_tc(const Problem& p, const BwdArgs& b, bool prep, cudaStream_t st) {
  if (prep)
    return launch_kernel(bwd_chain2_tc_kernel, dim3(p.n_seg_total, p.h_v), dim3(kTcThreads), kChain2Smem, st, true, p,
                         b);
  return launch_kernel(bwd_chain_tc_kernel, dim3(p.n_seg_total, p.h_v), dim3(kTcThreads), kChainSmem, st, true, p, b);
}

cudaError_t launch_bwd_local_tc(const Problem& p, const BwdArgs& b, cudaStream_t st) {
  const unsigned grid = (unsigned)p.n_chunks_total * (unsigned)p.h_qk;
  return launch_kernel(bwd_local_tc_kernel, dim3(grid), dim3(kLocThreads), kTcSmem, st, true, p, b);
}

}  // namespace gdn
