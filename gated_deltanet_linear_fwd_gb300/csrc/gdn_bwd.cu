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
// Three kernels after a forward pass that also leaves each chunk's start state
// and A^T (fp16):
//   bwd_pre_kernel    per (chunk, value head): T' and E            (chunk-parallel)
//   bwd_chain_tc_kernel (gdn_bwd_tc.cu) per segment and value head: D over the
//                     chunks in reverse, D kept in fp32; writes every chunk's D
//                     (fp16) and dh0; context parallel like the forward
//   bwd_local_tc_kernel (gdn_bwd_tc.cu) per (chunk, q/k head), over the value
//                     heads of the group: every other gradient on tcgen05
// bwd_pre_kernel runs its products on the tensor cores through mma.sync
// m16n8k16 (fp16 operands in the forward's 128-byte-swizzled tile image, fp32
// accumulators); tiles arrive by bulk copies on an mbarrier with a bounded wait.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "gdn_dev.cuh"

namespace gdn {
namespace {

constexpr int kBwdThreads = 256;

// ---------------------------------------------------------------- fragments
// An fp16 tile of `rows` rows and 64 * panels columns, stored as panels of
// rows x 64 (128 bytes a row, 16-byte chunk c of row r at chunk c ^ (r & 7)).
struct Tile {
  uint32_t base;
  uint32_t panel_bytes;  // rows * 128
  __device__ __forceinline__ uint32_t at(int row, int col) const {
    return base + (uint32_t)(col >> 6) * panel_bytes + sw128_offset((uint32_t)row, (uint32_t)((col & 63) >> 3)) +
           (uint32_t)(col & 7) * 2u;
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc[NT][4] += A[m0 .. m0+15][k0 .. k0+16 KS) * B[k0 ..][n0 .. n0 + 8 NT), one warp.
// TA: A is stored transposed (tile rows index k); TB: B is stored with rows
// indexing k (else rows index n).  Accumulator element e of n-tile t sits at
// row m0 + lane/4 + 8 (e >> 1), column n0 + 8 t + 2 (lane % 4) + (e & 1).
template <int NT, int KS, bool TA, bool TB>
__device__ __forceinline__ void warp_mma(float (&acc)[NT][4], const Tile& ta, const Tile& tb, int m0, int n0,
                                         int k0) {
  static_assert(NT % 2 == 0, "n-tiles come in pairs");
  const int lane = threadIdx.x & 31, i = lane & 7, q = lane >> 3;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int kk = k0 + 16 * ks;
    uint32_t a[4];
    if (!TA)
      ldsm_x4(ta.at(m0 + i + (q & 1) * 8, kk + (q >> 1) * 8), a);
    else
      ldsm_x4_t(ta.at(kk + i + (q >> 1) * 8, m0 + (q & 1) * 8), a);
#pragma unroll
    for (int t = 0; t < NT; t += 2) {
      const int nn = n0 + 8 * t;
      uint32_t b[4];
      if (!TB)
        ldsm_x4(tb.at(nn + i + (q >> 1) * 8, kk + (q & 1) * 8), b);
      else
        ldsm_x4_t(tb.at(kk + i + (q & 1) * 8, nn + (q >> 1) * 8), b);
      mma16816(acc[t], a, b[0], b[1]);
      mma16816(acc[t + 1], a, b[2], b[3]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 h2f(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The fragment of a 16 x 8 NT accumulator as fp16 pairs into a tile (scaled per row).
template <int NT>
__device__ __forceinline__ void store_frag(const Tile& t, const float (&acc)[NT][4], int m0, int n0, float& mx) {
  const int lane = threadIdx.x & 31, r = m0 + (lane >> 2), c = n0 + 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = absmax_nan(mx, acc[nt][e]);
    sts_u32(t.at(r, c + 8 * nt), pack_f16x2(acc[nt][0], acc[nt][1]));
    sts_u32(t.at(r + 8, c + 8 * nt), pack_f16x2(acc[nt][2], acc[nt][3]));
  }
}

// ------------------------------------------------------------------- chunks
// Sequence, first token and valid rows of global chunk gc (as the forward).
__device__ __forceinline__ bool chunk_rows(const Problem& p, int gc, int& n, int64_t& t0, int& cv) {
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

// 64 rows x 128 bf16 of a [tokens, heads, 128] tensor into an fp16 tile (two
// panels), row r scaled by row_scale[r] (null: 1); rows >= cv are zero.
__device__ __forceinline__ void load_rows_f16(const Tile& t, const __nv_bfloat16* src, int64_t t0, int heads, int head,
                                              int cv, const float* row_scale, float& mx) {
  // all loads in flight before the first store (the stores are ordered memory operations)
  constexpr int kPer = 64 * 16 / kBwdThreads;
  uint4 raw[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int idx = threadIdx.x + u * kBwdThreads, r = idx >> 4, c = idx & 15;
    raw[u] = make_uint4(0, 0, 0, 0);
    if (r < cv) raw[u] = *reinterpret_cast<const uint4*>(src + ((size_t)(t0 + r) * heads + head) * kDim + c * 8);
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int idx = threadIdx.x + u * kBwdThreads, r = idx >> 4, c = idx & 15;
    const float sc = row_scale ? row_scale[r] : 1.f;
    const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      mx = absmax_nan(absmax_nan(mx, f.x * sc), f.y * sc);
      o[e] = pack_f16x2(f.x * sc, f.y * sc);
    }
    st_shared_v4(t.at(r, c * 8), o[0], o[1], o[2], o[3]);
  }
}

// A bounded wait on a load barrier by every thread; false (in every thread
// alike) when it ran out, after recording the timeout.
__device__ __forceinline__ bool loads_landed(uint64_t* bar, uint32_t parity, const Problem& p) {
  const bool ok = mbar_wait(bar, parity, kWaitLimitNs);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) report(p.status, kDevTimeout, kDetTmaWait);
    // let copies still in flight land before the shared memory is released
    const uint64_t t_start = globaltimer_ns();
    while (globaltimer_ns() - t_start < 2000000ull) {
    }
    return false;
  }
  return true;
}

__device__ __forceinline__ uint8_t* smem_base() {
  extern __shared__ uint8_t smem_raw[];
  return smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
}

// ------------------------------------------------------------------ bwd_pre
// T' = -W^T Ktil (128 x 128) and E = scale (diag(gamma) Q)^T dO + (-W^T) Y with
// Y = scale P^T dO, for one (chunk, value head); both fp16 in the tile image
// (rows d_k; panels d_k resp. d_v 0-63 | 64-127).
constexpr uint32_t kPreWt = 0;                 // -W^T record tile: 128 rows (d_k) x 64 (r)
constexpr uint32_t kPreP = kPreWt + 16384;     // P record tile: 64 x 64
constexpr uint32_t kPreKt = kPreP + 8192;      // diag(dec) K: 64 x 128
constexpr uint32_t kPreQ = kPreKt + 16384;     // scale diag(gamma) Q: 64 x 128
constexpr uint32_t kPreDo = kPreQ + 16384;     // dO: 64 x 128
constexpr uint32_t kPreY = kPreDo + 16384;     // Y: 64 x 128
constexpr uint32_t kPreGam = kPreY + 16384;    // record gates: exp(G) [64], dec [64]
constexpr uint32_t kPreBar = kPreGam + 512;
constexpr uint32_t kPreSmem = kPreBar + 64 + 1024;

__global__ void __launch_bounds__(kBwdThreads, 2) bwd_pre_kernel(const Problem p, const BwdArgs b) {
  uint8_t* sm = smem_base();
  const uint32_t s0 = smem_u32(sm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kPreBar);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int gc = (int)(blockIdx.x / (unsigned)p.h_v), j = (int)(blockIdx.x % (unsigned)p.h_v);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  int n, cv;
  int64_t t0;
  if (!chunk_rows(p, gc, n, t0, cv)) {
    if (tid == 0) report(p.status, kDevCheck, kDetSegMismatch);
    return;
  }
  // one read of the status word per CTA: an earlier kernel's failure means incomplete inputs
  if (__syncthreads_or(tid == 0 && earlier_failure(p.status))) return;  // (also: barrier initialised)
  const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
  const uint8_t* rec = p.wy + ((size_t)gc * p.h_v + j) * kRecBytes;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, 16384u + 8192u + 512u);
    bulk_load(sm + kPreWt, rec + kRecWn, 16384u, bar);
    bulk_load(sm + kPreP, rec + kRecP, 8192u, bar);
    bulk_load(sm + kPreGam, rec + kRecGam, 512u, bar);
  }
  float mx = 0.f;
  const Tile tWt{s0 + kPreWt, 16384}, tP{s0 + kPreP, 8192}, tKt{s0 + kPreKt, 8192}, tQ{s0 + kPreQ, 8192},
      tDo{s0 + kPreDo, 8192}, tY{s0 + kPreY, 8192};
  load_rows_f16(tDo, reinterpret_cast<const __nv_bfloat16*>(b.dout), t0, p.h_v, j, cv, nullptr, mx);
  if (!loads_landed(bar, 0, p)) return;
  float* gam = reinterpret_cast<float*>(sm + kPreGam);  // exp(G) [64], dec [64]
  {
    // rows scaled: K by dec, Q by scale * exp(G)
    __shared__ float qsc[64];
    if (tid < 64) qsc[tid] = p.scale * gam[tid];
    __syncthreads();
    load_rows_f16(tKt, reinterpret_cast<const __nv_bfloat16*>(p.k), t0, p.h_qk, iq, cv, gam + 64, mx);
    load_rows_f16(tQ, reinterpret_cast<const __nv_bfloat16*>(p.q), t0, p.h_qk, iq, cv, qsc, mx);
  }
  __syncthreads();
  // Y = scale P^T dO: warp (rows 16 (w & 3), columns 64 (w >> 2))
  {
    const int m0 = 16 * (warp & 3), n0 = 64 * (warp >> 2);
    float acc[8][4];
    zero(acc);
    warp_mma<8, 4, true, true>(acc, tP, tDo, m0, n0, 0);
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] *= p.scale;
    store_frag(tY, acc, m0, n0, mx);
  }
  __syncthreads();
  // T' and E: warp w owns rows 16 w .. 16 w + 15 (d_k), all 128 columns
  const size_t slot = ((size_t)gc * p.h_v + j) * 32768u;
  const int m0 = 16 * warp, lane = tid & 31;
  auto store_global = [&](uint8_t* dst, const float(&acc)[16][4]) {
    const int r = m0 + (lane >> 2), c = 2 * (lane & 3);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int col = 8 * t + c;
      const uint32_t off0 = (uint32_t)(col >> 6) * 16384u + sw128_offset(r, (col & 63) >> 3) + (col & 7) * 2;
      const uint32_t off1 = (uint32_t)(col >> 6) * 16384u + sw128_offset(r + 8, (col & 63) >> 3) + (col & 7) * 2;
#pragma unroll
      for (int e = 0; e < 4; ++e) mx = absmax_nan(mx, acc[t][e]);
      *reinterpret_cast<uint32_t*>(dst + off0) = pack_f16x2(acc[t][0], acc[t][1]);
      *reinterpret_cast<uint32_t*>(dst + off1) = pack_f16x2(acc[t][2], acc[t][3]);
    }
  };
  {
    float acc[16][4];
    zero(acc);
    warp_mma<16, 4, false, true>(acc, tWt, tKt, m0, 0, 0);
    store_global(b.tmat + slot, acc);
  }
  {
    float acc[16][4];
    zero(acc);
    warp_mma<16, 4, true, true>(acc, tQ, tDo, m0, 0, 0);
    warp_mma<16, 4, false, true>(acc, tWt, tY, m0, 0, 0);
    store_global(b.emat + slot, acc);
  }
  if (!(mx < 65504.f)) report(p.status, kDevCheck, kDetFp16Range);
}

}  // namespace

namespace {
cudaError_t bwd_attrs() {
  static cudaError_t once = [] {
    cudaError_t e = cudaFuncSetAttribute(bwd_pre_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPreSmem);
    return e;
  }();
  return once;
}
}  // namespace

cudaError_t launch_bwd_pre(const Problem& p, const BwdArgs& b, cudaStream_t st) {
  cudaError_t e = bwd_attrs();
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.n_chunks_total * (unsigned)p.h_v;
  return launch_kernel(bwd_pre_kernel, dim3(grid), dim3(kBwdThreads), kPreSmem, st, true, p, b);
}



}  // namespace gdn
