// The chunk-local WY/gate kernel (FlashQLA pages, section "Optimising GDN
// chunked prefill": gate cumsum and the WY form of each 64-token chunk), and
// the small chunk-index kernel it reads.
//
// Everything a chunk contributes that does not depend on the state is
// computed here, for every (chunk, value head) at once, so that the scans
// that carry the state from chunk to chunk do only the state-dependent
// products.  Per chunk (G = inclusive cumsum of g, gamma = exp(G),
// dec = exp(G_63 - G)):
//   D    = [K;Q] K^T                       (bf16 MMA, exact inputs)
//   L    = strict_lower(diag(beta) D_kk . exp(G_r - G_s))
//   P    = lower(D_qk . exp(G_r - G_s))    (diagonal included)
//   A    = (I + L)^{-1}                    (fp32, blocked)
//   W^T  = K^T (A diag(beta gamma))^T,  U^T = V^T (A diag(beta))^T
// (bf16 MMAs on the exact K and V, with the A operands split into bf16 high
// parts and remainders, so W and U keep about 16 significant bits of A)
// and writes -W, U^T, P and (gamma, dec) as one record per (chunk, value
// head), each tile in the 128-byte-swizzled layout the scan's MMAs read.
//
// One CTA of 256 threads per (chunk, value head), four CTAs per SM: the
// shared-memory regions are reused as the work moves on (V lands where Q
// was once D has read it, the A operands of W and then of U go where L was,
// -W and U^T go where K and V were), and P and the gates go straight to
// global memory.
#include <cuda_bf16.h>

#include "gdn_dev.cuh"

namespace gdn {
namespace {

constexpr int kWyThreads = 256;

// ---- shared memory map (bytes from a 1024-byte aligned base) ----
constexpr uint32_t kWyKQ = 0;          // bf16 [K d0-63 | Q d0-63 | K d64-127 | Q d64-127] (TMA).  Once D
                                       // has read Q, V d0-63 | V d64-127 land in the Q slots; once W and
                                       // U are computed, the K slots take the two row halves of the -W
                                       // tile and the Q slots those of the U^T tile
constexpr uint32_t kWyV0 = 8192, kWyV1 = 24576;
constexpr uint32_t kWyF = 32768;       // fp32 [64][68]: L below the diagonal, A^T on and above it; then
                                       // the A operand hi | lo (8 KB each): A diag(beta gamma) for W,
                                       // then A diag(beta) for U
constexpr uint32_t kFStride = 68;
constexpr uint32_t kWyScr = kWyF + 64 * kFStride * 4;  // fp32 solve scratch (4.5 KB): T blocks, rows
                                                        // padded against bank conflicts
constexpr uint32_t kWyGates = kWyScr + 4608;  // G | exp(G) | exp(G_63 - G) | beta | exp(-G), 64 floats each
constexpr uint32_t kWyCtl = kWyGates + 1280;
constexpr uint32_t kWySmemUse = kWyCtl + 64;
constexpr uint32_t kWySmemAlloc = kWySmemUse + 1024;
static_assert(4 * (kWySmemAlloc + 1024) <= 233472, "four CTAs per SM must fit");

// ---- TMEM columns ----
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kTD = 0;    // [K K^T ; Q K^T]   128 x 64
constexpr uint32_t kTW = 64;   // W^T               128 x 64
constexpr uint32_t kTU = 0;    // U^T               128 x 64 (over D, read by then)

struct WyCtl {
  uint64_t full, vfull, kq, w, u;  // K|Q landed, V landed, D done, W done, U done
  uint64_t stall;                  // the test hook's barrier (nothing arrives on it)
  uint32_t tmem;
  int abort;
  float warp_total[2];
};
static_assert(sizeof(WyCtl) <= kWySmemUse - kWyCtl, "control block too large");

// ---------------------------------------------------------------- solve
// A = (I + L)^{-1} for the unit lower-triangular 64 x 64 matrix held
// strictly below the diagonal of F.  A^T is written on and above the
// diagonal (F[s][r] = A[r][s], r >= s).  Diagonal 16 x 16 blocks by forward
// substitution (one column per thread), then two merge levels:
//   A_10 = -D_1 L_10 D_0, A_32 = -D_3 L_32 D_2       (16 x 16 blocks)
//   A_hl = -A_hh L_hl A_ll                           (32 x 32 blocks)
// The strict lower parts of the diagonal 32 x 32 blocks are cleared once
// consumed, so every product runs over full ranges without masks.
// Row strides of the T blocks in the scratch: 18 (16 x 16, float2 stores of
// 16 rows hit 16 different bank pairs) and 36 (32 x 32, float4 stores of 32
// rows spread over all 32 banks).
constexpr int kTs1 = 18, kTs2 = 36;
static_assert(2 * 16 * kTs1 * 4 <= 4608 && 32 * kTs2 * 4 <= 4608, "solve scratch");

__device__ __forceinline__ void solve_unit_lower(float* F, float* scratch, int tid) {
  // ---- diagonal blocks ----
  {
    float x[16];
    const int b = tid >> 4, c = tid & 15;
    if (tid < 64) {
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
    __syncthreads();
    if (tid < 64) {  // row c of D_b^T; zero below the diagonal (L_bb has been consumed)
      float* Dt = F + (16 * b + c) * kFStride + 16 * b;
#pragma unroll
      for (int r4 = 0; r4 < 16; r4 += 4)
        *reinterpret_cast<float4*>(Dt + r4) =
            make_float4(r4 + 0 >= c ? x[r4] : 0.f, r4 + 1 >= c ? x[r4 + 1] : 0.f,
                        r4 + 2 >= c ? x[r4 + 2] : 0.f, r4 + 3 >= c ? x[r4 + 3] : 0.f);
    }
    __syncthreads();
  }
  // ---- level 1: T = L_{ib,jb} D_jb, then A_{ib,jb} = -D_ib T, for (ib, jb) = (1, 0), (3, 2);
  //      four warps per pair, each on four columns of T (four rows of A_{ib,jb}) ----
  {
    const int mat = tid >> 7, w = (tid >> 5) & 3, lane = tid & 31;
    const int ib = 2 * mat + 1, jb = 2 * mat;
    float* Ts = scratch + mat * 16 * kTs1;  // [16][kTs1]
    {
      // T[r][c], c = 4w + 2 (lane >> 4) + {0, 1}, r = lane & 15: sum over m >= 4w (D_jb[m][c] = 0 for m < c)
      const int r = lane & 15, c = 4 * w + 2 * (lane >> 4);
      const float* Lr = F + (16 * ib + r) * kFStride + 16 * jb;
      const float* D0 = F + (16 * jb + c) * kFStride + 16 * jb;  // D_jb column c as a row of D^T
      float t0 = 0.f, t1 = 0.f;
#pragma unroll
      for (int m = 0; m < 16; m += 4) {
        if (m < 4 * w) continue;
        const float4 l4 = *reinterpret_cast<const float4*>(Lr + m);
        const float4 a0 = *reinterpret_cast<const float4*>(D0 + m);
        const float4 a1 = *reinterpret_cast<const float4*>(D0 + kFStride + m);
        t0 = fmaf(l4.x, a0.x, fmaf(l4.y, a0.y, fmaf(l4.z, a0.z, fmaf(l4.w, a0.w, t0))));
        t1 = fmaf(l4.x, a1.x, fmaf(l4.y, a1.y, fmaf(l4.z, a1.z, fmaf(l4.w, a1.w, t1))));
      }
      *reinterpret_cast<float2*>(Ts + r * kTs1 + c) = make_float2(t0, t1);
    }
    __syncthreads();
    {
      // A_{ib,jb}[r][c], r = 4w + 2 (lane >> 4) + {0, 1}, c = lane & 15: sum over m <= 4w + 3
      // (D_ib[r][m] = 0 for m > r)
      const int r = 4 * w + 2 * (lane >> 4), c = lane & 15;
      float x0 = 0.f, x1 = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        if (m >= 4 * w + 4) break;
        const float2 d = *reinterpret_cast<const float2*>(F + (16 * ib + m) * kFStride + 16 * ib + r);
        const float tv = Ts[m * kTs1 + c];
        x0 = fmaf(d.x, tv, x0);
        x1 = fmaf(d.y, tv, x1);
      }
      *reinterpret_cast<float2*>(F + (16 * jb + c) * kFStride + 16 * ib + r) = make_float2(-x0, -x1);
      // L_{ib,jb} has been consumed: clear it
      const int idx = tid & 127, rz = idx >> 3, cz = (idx & 7) * 2;
      *reinterpret_cast<float2*>(F + (16 * ib + rz) * kFStride + 16 * jb + cz) = make_float2(0.f, 0.f);
    }
    __syncthreads();
  }
  // ---- level 2: T = L_hl A_ll (32 x 32), then A_hl = -A_hh T.  Each warp
  //      takes four columns of T (four rows of A_hl), so the triangular
  //      bounds of A_ll and A_hh are the same across the warp ----
  {
    const int w = tid >> 5, lane = tid & 31;
    float* Tb = scratch;  // [32][kTs2]
    {
      // T[lane][4w .. 4w+3] = sum_{m >= 4w} L[32 + lane][m] A_ll[m][c]   (A_ll[m][c] = 0 for m < c)
      const float* Lr = F + (32 + lane) * kFStride;
      float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int m = 4 * w; m < 32; m += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(Lr + m);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 a4 = *reinterpret_cast<const float4*>(F + (4 * w + c) * kFStride + m);  // A_ll[m..m+3][4w+c]
          t[c] = fmaf(l4.x, a4.x, fmaf(l4.y, a4.y, fmaf(l4.z, a4.z, fmaf(l4.w, a4.w, t[c]))));
        }
      }
      *reinterpret_cast<float4*>(Tb + lane * kTs2 + 4 * w) = make_float4(t[0], t[1], t[2], t[3]);
    }
    __syncthreads();
    {
      // A_hl[4w .. 4w+3][lane] = -sum_{m <= 4w+3} A_hh[r][m] T[m][lane]   (A_hh[r][m] = 0 for m > r)
      float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int m = 0; m < 4 * w + 4; ++m) {
        const float4 a4 = *reinterpret_cast<const float4*>(F + (32 + m) * kFStride + 32 + 4 * w);  // A_hh[4w..4w+3][m]
        const float tv = Tb[m * kTs2 + lane];
        x[0] = fmaf(a4.x, tv, x[0]);
        x[1] = fmaf(a4.y, tv, x[1]);
        x[2] = fmaf(a4.z, tv, x[2]);
        x[3] = fmaf(a4.w, tv, x[3]);
      }
      *reinterpret_cast<float4*>(F + lane * kFStride + 32 + 4 * w) = make_float4(-x[0], -x[1], -x[2], -x[3]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void seq_bounds(const Problem& p, int n, int64_t& bos, int64_t& eos) {
  if (p.cu) {
    bos = p.cu[n];
    eos = p.cu[n + 1];
  } else {
    bos = (int64_t)n * p.T_row;
    eos = bos + p.T_row;
  }
}

// Returns false (in every thread alike) when a wait gave up.
__device__ __forceinline__ bool wy_body(uint8_t* sm, WyCtl* ctl, const Problem& p, const CUtensorMap* mq,
                                     const CUtensorMap* mk, const CUtensorMap* mv, uint32_t tmem, float& mx) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gc = (int)(blockIdx.x / (unsigned)p.h_v), j = (int)(blockIdx.x % (unsigned)p.h_v);
  if (p.stall_ns) {  // test hook: a wait that nothing ends, bounded by stall_ns
    bool ok = true;
    if (tid == 0 && !mbar_wait(&ctl->stall, 0, p.stall_ns)) {
      atomicCAS(&ctl->abort, 0, kDetStallTest);
      ok = false;
    }
    if (__syncthreads_or(!ok)) return false;
  }
  int n, cv;
  int64_t t0;
  if (p.cu) {  // one 16-byte load: {sequence, valid tokens, first token}
    const int4 ci = p.chunk_info[gc];
    n = ci.x;
    cv = ci.y;
    t0 = (int64_t)(((uint64_t)(uint32_t)ci.w << 32) | (uint32_t)ci.z);
  } else {     // fixed-length rows
    const int cps = chunks_of(p.T_row);
    n = gc / cps;
    t0 = (int64_t)n * p.T_row + (int64_t)(gc - n * cps) * kChunk;
    cv = (int)min((int64_t)kChunk, (int64_t)(n + 1) * p.T_row - t0);
  }
  if (n < 0 || n >= p.n_seqs || cv <= 0 || cv > kChunk) {  // the chunk index disagrees with the plan
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return false;
  }
  const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
  float* gts = reinterpret_cast<float*>(sm + kWyGates);
  float* sG = gts;
  float* sGam = gts + 64;
  float* sDec = gts + 128;
  float* sBeta = gts + 192;
  float* sEm = gts + 256;
  float* F = reinterpret_cast<float*>(sm + kWyF);
  float* scratch = reinterpret_cast<float*>(sm + kWyScr);
  const uint32_t sKQ = smem_u32(sm + kWyKQ), sF = smem_u32(sm + kWyF);
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  uint8_t* rec = p.wy + ((size_t)gc * p.h_v + j) * kRecBytes;

  // ---- loads; D = [K;Q] K^T as soon as they land ----
  if (tid == 0) {
    mbar_arrive_expect_tx(&ctl->full, 32768u);
    tma_load_3d(sm + kWyKQ, mk, &ctl->full, 0, iq, (int)t0);
    tma_load_3d(sm + kWyKQ + 16384, mk, &ctl->full, 64, iq, (int)t0);
    tma_load_3d(sm + kWyKQ + 8192, mq, &ctl->full, 0, iq, (int)t0);
    tma_load_3d(sm + kWyKQ + 24576, mq, &ctl->full, 64, iq, (int)t0);
  }
  if (warp == 2 || warp == 3) {  // gate cumsum; rows past the sequence end act as g = beta = 0
    const int r = tid - 64;
    const bool ok = r < cv;
    float x = ok ? p.g[(size_t)(t0 + r) * p.h_v + j] : 0.f;
    const float b = ok ? p.beta[(size_t)(t0 + r) * p.h_v + j] : 0.f;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) ctl->warp_total[warp - 2] = x;
    named_bar_sync(1, 64);
    if (warp == 3) x += ctl->warp_total[0];
    sG[r] = x;
    sGam[r] = __expf(x);
    sBeta[r] = b;
    sEm[r] = __expf(-x);
    named_bar_sync(1, 64);
    const float dec = __expf(sG[63] - x);
    sDec[r] = dec;
    reinterpret_cast<float*>(rec + kRecGam)[r] = sGam[r];  // the record's gates
    reinterpret_cast<float*>(rec + kRecGam)[64 + r] = dec;
  }
  if (tid == 32) {
    if (wait_phase(&ctl->full, 0, &ctl->abort, 100)) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u;
        mma_bf16(tmem + kTD, sdesc_sw128(sKQ + off, 16, 1024), sdesc_sw128(sKQ + off, 16, 1024), id, ks > 0);
      }
      mma_commit(&ctl->kq);
    }
  }
  bool ok = wait_phase(&ctl->kq, 0, &ctl->abort, 101);
  if (__syncthreads_or(!ok)) return false;
  tc_fence_after();
  if (tid == 0) {  // D has read Q: V into its slots (needed only by U, after the inverse)
    mbar_arrive_expect_tx(&ctl->vfull, 16384u);
    tma_load_3d(sm + kWyV0, mv, &ctl->vfull, 0, j, (int)t0);
    tma_load_3d(sm + kWyV1, mv, &ctl->vfull, 64, j, (int)t0);
  }

  // ---- L (TMEM lanes 0-63) into F; P (lanes 64-127) into the record, as its
  //      swizzled operand tile ----
  {
    const bool factored = fabsf(sG[0]) < 80.f && fabsf(sG[63]) < 80.f;  // exp(G_r) exp(-G_s) cannot overflow
    const int R = (warp & 3) * 32 + lane, ch = warp >> 2;                 // columns 32 ch .. 32 ch + 31
    uint32_t rk[2][16];
    tmem_ld16(tmem + lane_base + kTD + ch * 32, rk[0]);
    tmem_ld16(tmem + lane_base + kTD + ch * 32 + 16, rk[1]);
    tmem_ld_wait(rk[0], rk[1]);
    if (p.plan_mode == kModeWarmup && R < 64 && (R >> 5) == ch) {  // warps 0 and 5 hold the diagonal
      // the chunk's warmup exponent: G_63 + sum_r log max(1, |1 - beta_r ||k_r||^2|), ||k_r||^2 = D[r][r]
      float kk = 0.f;
#pragma unroll
      for (int sl = 0; sl < 32; ++sl)
        if (sl == (R & 31)) kk = __uint_as_float(rk[sl >> 4][sl & 15]);
      float t = __logf(fmaxf(1.f, fabsf(1.f - sBeta[R] * kk)));  // 0 past the sequence end (beta = 0)
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) t += __shfl_xor_sync(0xffffffffu, t, d);
      if (lane == 0) ctl->warp_total[ch] = t;
    }
    if (R < 64) {
      const int r = R;
      const float br = sBeta[r], Gr = sG[r], brE = sBeta[r] * sGam[r];
      float* Lr = F + r * kFStride + ch * 32;
      if (factored) {  // separate loops: a select between the two would evaluate both
#pragma unroll
        for (int s4 = 0; s4 < 32; s4 += 4) {
          const float4 em = *reinterpret_cast<const float4*>(sEm + ch * 32 + s4);
          const float* emv = &em.x;
          float4 o4;
          float* o = &o4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int sl = s4 + e;
            o[e] = (ch * 32 + sl < r) ? brE * __uint_as_float(rk[sl >> 4][sl & 15]) * emv[e] : 0.f;
          }
          *reinterpret_cast<float4*>(Lr + s4) = o4;
        }
      } else {
#pragma unroll
        for (int s4 = 0; s4 < 32; s4 += 4) {
          float4 o4;
          float* o = &o4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int sl = s4 + e, s = ch * 32 + sl;
            o[e] = (s < r) ? br * __uint_as_float(rk[sl >> 4][sl & 15]) * __expf(Gr - sG[s]) : 0.f;
          }
          *reinterpret_cast<float4*>(Lr + s4) = o4;
        }
      }
    } else {
      const int r = R - 64;
      const float Er = sGam[r], Gr = sG[r];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
        if (factored) {
          const float4 e0 = *reinterpret_cast<const float4*>(sEm + ch * 32 + 8 * q);
          const float4 e1 = *reinterpret_cast<const float4*>(sEm + ch * 32 + 8 * q + 4);
          const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int sl = 8 * q + e;
            f[e] = (ch * 32 + sl <= r) ? __uint_as_float(rk[sl >> 4][sl & 15]) * Er * ev[e] : 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int sl = 8 * q + e, s = ch * 32 + sl;
            f[e] = (s <= r) ? __uint_as_float(rk[sl >> 4][sl & 15]) * __expf(Gr - sG[s]) : 0.f;
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) mx = absmax_nan(mx, f[e]);
        *reinterpret_cast<uint4*>(rec + kRecP + sw128_offset(r, ch * 4 + q)) =
            make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && p.plan_mode == kModeWarmup)
    p.chunk_exp[(size_t)gc * p.h_v + j] = sG[63] + ctl->warp_total[0] + ctl->warp_total[1];

  // ---- A = (I + L)^{-1} ----
  solve_unit_lower(F, scratch, tid);

  // ---- A operands: quarter c of row s of A^T, scaled by beta gamma (for W),
  //      then by beta (for U), split into bf16 high parts and remainders, in
  //      the hi | lo buffer over F; W^T = K^T (A diag(beta gamma))^T and
  //      U^T = V^T (A diag(beta))^T take it in turn (A = hi + lo) ----
  const int s = tid >> 2, qc = tid & 3;  // columns 16 qc .. 16 qc + 15 of row s
  float a[16];
  {
    const float* At = F + s * kFStride + 16 * qc;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const float4 a4 = *reinterpret_cast<const float4*>(At + 4 * q4);
      a[4 * q4] = (16 * qc + 4 * q4 + 0 >= s) ? a4.x : 0.f;
      a[4 * q4 + 1] = (16 * qc + 4 * q4 + 1 >= s) ? a4.y : 0.f;
      a[4 * q4 + 2] = (16 * qc + 4 * q4 + 2 >= s) ? a4.z : 0.f;
      a[4 * q4 + 3] = (16 * qc + 4 * q4 + 3 >= s) ? a4.w : 0.f;
    }
  }
  if (p.wyA) {  // A^T for the backward: row s, columns 16 qc .. 16 qc + 15, fp16
    uint8_t* dst = p.wyA + ((size_t)gc * p.h_v + j) * 8192u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 8; ++e) mx = absmax_nan(mx, a[8 * h + e]);
      *reinterpret_cast<uint4*>(dst + sw128_offset(s, 2 * qc + h)) =
          make_uint4(pack_f16x2(a[8 * h], a[8 * h + 1]), pack_f16x2(a[8 * h + 2], a[8 * h + 3]),
                     pack_f16x2(a[8 * h + 4], a[8 * h + 5]), pack_f16x2(a[8 * h + 6], a[8 * h + 7]));
    }
  }
  auto store_operand = [&](float sc) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = a[8 * h + e] * sc;
      store_bf16x8_hilo(sF + sw128_offset(s, 2 * qc + h), sF + 8192 + sw128_offset(s, 2 * qc + h), f);
    }
  };
  const uint32_t id_mn = idesc_bf16_f32(128, 64, true, true);
  __syncthreads();  // F is read: its first 16 KB take the operand
  store_operand(sBeta[s] * sGam[s]);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 32) {
    tc_fence_after();
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kTW, sdesc_sw128(sKQ + ks * 2048, 16384, 1024),
                 sdesc_sw128(sF + part * 8192 + ks * 2048, 8192, 1024), id_mn, (part | ks) > 0);
    mma_commit(&ctl->w);
  }
  ok = wait_phase(&ctl->w, 0, &ctl->abort, 102);
  if (__syncthreads_or(!ok)) return false;
  tc_fence_after();
  store_operand(sBeta[s]);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 32) {
    if (wait_phase(&ctl->vfull, 0, &ctl->abort, 103)) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTU, sdesc_sw128(sKQ + kWyV0 + ks * 2048, 16384, 1024),
                   sdesc_sw128(sF + part * 8192 + ks * 2048, 8192, 1024), id_mn, (part | ks) > 0);
    }
    mma_commit(&ctl->u);
  }

  // ---- -W and U^T tiles, row halves d 0-63 | 64-127 in the slots of K (read
  //      by W) and of V (read by U).  No range check here: an fp16 overflow of
  //      either becomes inf in the scan's V' = U - W S, which the scan checks
  //      every chunk. ----
  {
    const int d = (warp & 3) * 32 + lane, ch = warp >> 2;
    const uint32_t half = (uint32_t)(d >> 6) * 16384u;
    uint32_t ra[16], rb[16];
    tmem_ld16(tmem + lane_base + kTW + ch * 32, ra);
    tmem_ld16(tmem + lane_base + kTW + ch * 32 + 16, rb);
    tmem_ld_wait(ra, rb);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = -__uint_as_float(q < 2 ? ra[8 * q + e] : rb[8 * (q - 2) + e]);
      st_shared_v4(sKQ + half + sw128_offset(d & 63, ch * 4 + q), pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]),
                   pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
    }
    fence_proxy_async_smem();
    ok = wait_phase(&ctl->u, 0, &ctl->abort, 104);
    if (__syncthreads_or(!ok)) return false;  // also: every thread's -W rows are written
    tc_fence_after();
    if (tid == 64) {  // -W into the record while U is read back
      bulk_store(rec + kRecWn, sm + kWyKQ, 8192);
      bulk_store(rec + kRecWn + 8192, sm + kWyKQ + 16384, 8192);
      bulk_commit();
    }
    tmem_ld16(tmem + lane_base + kTU + ch * 32, ra);
    tmem_ld16(tmem + lane_base + kTU + ch * 32 + 16, rb);
    tmem_ld_wait(ra, rb);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(q < 2 ? ra[8 * q + e] : rb[8 * (q - 2) + e]);
      st_shared_v4(sKQ + kWyV0 + half + sw128_offset(d & 63, ch * 4 + q), pack_f16x2(f[0], f[1]),
                   pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 64) {
    bulk_store(rec + kRecU, sm + kWyV0, 8192);
    bulk_store(rec + kRecU + 8192, sm + kWyV1, 8192);
    bulk_commit();
  }
  return true;
}

__global__ void __launch_bounds__(kWyThreads, 4)
    wy_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned
  WyCtl* ctl = reinterpret_cast<WyCtl*>(sm + kWyCtl);
  const int tid = threadIdx.x, warp = tid >> 5;
  grid_dependency_wait();  // the chunk index (varlen) is written by the kernel before
  grid_launch_dependents();
  if (tid == 0) {
    mbar_init(&ctl->stall, 1);
    mbar_init(&ctl->full, 1);
    mbar_init(&ctl->vfull, 1);
    mbar_init(&ctl->kq, 1);
    mbar_init(&ctl->w, 1);
    mbar_init(&ctl->u, 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mv);
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  float mx = 0.f;  // largest magnitude rounded to fp16 by this thread
  wy_body(sm, ctl, p, &mq, &mk, &mv, tmem, mx);
  // the record's bulk stores have read shared memory before it is released (the
  // grid completes only once they have landed)
  if (tid == 64) bulk_wait_read_all();
  tc_fence_before();
  __syncthreads();
  if (ctl->abort) {
    if (tid == 0) report(p.status, kDevTimeout, ctl->abort);
    // let copies and MMAs already in flight land before the memory is released
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
    __syncthreads();
  }
  if (!(mx < 65504.f)) report(p.status, kDevCheck, kDetFp16Range);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- chunk index
// Varlen chunk index: seq_chunk_base[n] = chunks of sequences 0..n-1;
// chunk_info[c] = {sequence, valid tokens, first token} of global chunk c.
// One CTA.  (Fixed-length rows need no index: it is arithmetic.)
constexpr int kMapThreads = 1024;

__global__ void __launch_bounds__(kMapThreads) chunk_map_kernel(const Problem p) {
  __shared__ int warp_sum[32];
  __shared__ int carry, seg_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_launch_dependents();
  if (tid == 0) {
    carry = 0;
    seg_total = 0;
  }
  __syncthreads();
  // The device offsets must be the plan's: sequence bounds that run from 0 to
  // T without going back, and the plan's numbers of chunks and segments.
  int bad = 0;
  for (int n0 = 0; n0 < p.n_seqs; n0 += kMapThreads) {
    const int n = n0 + tid;
    int cnt = 0;
    if (n < p.n_seqs) {
      int64_t bos, eos;
      seq_bounds(p, n, bos, eos);
      if (bos < 0 || eos < bos || eos > (int64_t)p.T_row || (n == 0 && bos != 0) ||
          (n == p.n_seqs - 1 && eos != (int64_t)p.T_row)) {
        bad = 1;
      } else {
        cnt = chunks_of(eos - bos);
        atomicAdd(&seg_total, seg_count(cnt, p.lambda_q8, p.plan_mode == kModeOff));
      }
    }
    int x = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += y;
      }
      warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? warp_sum[warp - 1] : 0) + carry;
    if (n < p.n_seqs) p.seq_chunk_base[n] = incl - cnt;
    __syncthreads();
    if (tid == kMapThreads - 1) carry = incl;
    __syncthreads();
  }
  const int total = carry;
  const bool valid =
      __syncthreads_or(bad) == 0 && total == p.n_chunks_total && seg_total == p.n_seg_total;
  if (!valid) {  // nothing later may follow these offsets: every chunk is marked as outside the plan
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    for (int n = tid; n <= p.n_seqs; n += kMapThreads) p.seq_chunk_base[n] = -1;
    for (int gc = tid; gc < p.n_chunks_total; gc += kMapThreads) p.chunk_info[gc] = make_int4(-1, 0, 0, 0);
    return;
  }
  if (tid == 0) p.seq_chunk_base[p.n_seqs] = total;
  __syncthreads();
  for (int gc = tid; gc < total; gc += kMapThreads) {
    int lo = 0, hi = p.n_seqs - 1;  // last n with base[n] <= gc
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.seq_chunk_base[mid] <= gc) lo = mid;
      else hi = mid - 1;
    }
    int64_t bos, eos;
    seq_bounds(p, lo, bos, eos);
    const int64_t t0 = bos + (int64_t)(gc - p.seq_chunk_base[lo]) * kChunk;
    p.chunk_info[gc] = make_int4(lo, (int)min((int64_t)kChunk, eos - t0), (int)(uint32_t)(uint64_t)t0,
                                 (int)(uint32_t)((uint64_t)t0 >> 32));
  }
}

}  // namespace

cudaError_t wy_kernel_setup() {
  return cudaFuncSetAttribute(wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWySmemAlloc);
}

cudaError_t launch_chunk_map(const Problem& p, cudaStream_t st) {
  chunk_map_kernel<<<1, kMapThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wy(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      cudaStream_t st, bool dependent) {
  if (p.n_chunks_total == 0) return cudaSuccess;
  const unsigned grid = (unsigned)p.n_chunks_total * (unsigned)p.h_v;
  return launch_kernel(wy_kernel, dim3(grid), dim3(kWyThreads), kWySmemAlloc, st, dependent, mq, mk, mv, p);
}

}  // namespace gdn
