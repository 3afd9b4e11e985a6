// fp32 path of the forward (all of q, k, v, o in fp32), for callers that need
// results within 1e-4 of the exact recurrence.  The tensor-core path rounds
// its operands to fp16 and cannot reach that, so this path runs the gated
// delta rule itself in fp32 on the CUDA cores:
//   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//   o_t = scale S_t q_t.
// Chunking and context parallelism are exact re-associations of this same
// recurrence (FlashQLA pages, sections "Optimising GDN chunked prefill" and
// "AutoCP"); here the parallelism comes instead from the d_v rows of the
// state, which evolve independently given k, g and beta.  One CTA owns 16 rows
// of one (sequence, value head): 16 threads per row, 8 columns each.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRowsPerCta = 16;

__global__ void __launch_bounds__(256) recurrence_f32_kernel(const Problem p) {
  const int tid = threadIdx.x;
  const int rr = tid >> 4;         // row within the CTA
  const int cg = tid & 15;         // column group: columns 8 cg .. 8 cg + 7
  const int n = blockIdx.x, j = blockIdx.y;
  const int dv = blockIdx.z * kRowsPerCta + rr;
  const int iq = (int)(((int64_t)j * p.h_qk) / p.h_v);
  int64_t bos, eos;
  if (p.cu) {
    bos = p.cu[n];
    eos = p.cu[n + 1];
  } else {
    bos = (int64_t)n * p.T_row;
    eos = bos + p.T_row;
  }
  const float* q = reinterpret_cast<const float*>(p.q);
  const float* k = reinterpret_cast<const float*>(p.k);
  const float* v = reinterpret_cast<const float*>(p.v);
  float* o = reinterpret_cast<float*>(p.out);
  const size_t head_off = (size_t)(n * p.h_v + j) * kDim * kDim;

  float S[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) S[e] = p.h0 ? p.h0[head_off + (size_t)(8 * cg + e) * kDim + dv] : 0.f;

  auto load = [&](int64_t t, float4& k0, float4& k1, float4& q0, float4& q1, float& vv, float& a, float& b) {
    const float4* kr = reinterpret_cast<const float4*>(k + ((size_t)t * p.h_qk + iq) * kDim + 8 * cg);
    const float4* qr = reinterpret_cast<const float4*>(q + ((size_t)t * p.h_qk + iq) * kDim + 8 * cg);
    k0 = kr[0];
    k1 = kr[1];
    q0 = qr[0];
    q1 = qr[1];
    vv = v[((size_t)t * p.h_v + j) * kDim + dv];
    a = p.g[(size_t)t * p.h_v + j];
    b = p.beta[(size_t)t * p.h_v + j];
  };
  float4 k0, k1, q0, q1;
  float vv = 0.f, gg = 0.f, bb = 0.f;
  if (bos < eos) load(bos, k0, k1, q0, q1, vv, gg, bb);
  for (int64_t t = bos; t < eos; ++t) {
    const float kc[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    const float qc[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const float vt = vv, alpha = expf(gg), beta = bb;
    if (t + 1 < eos) load(t + 1, k0, k1, q0, q1, vv, gg, bb);  // next token in flight
    // S_{t-1} k_t, reduced over the 16 column groups of this row
    float sk = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) sk = fmaf(S[e], kc[e], sk);
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, d);
    // S_t = alpha (S_{t-1} - beta (S_{t-1} k) k^T) + beta v k^T
    const float bsk = beta * sk, bv = beta * vt;
    float so = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      S[e] = fmaf(alpha, fmaf(-bsk, kc[e], S[e]), bv * kc[e]);
      so = fmaf(S[e], qc[e], so);
    }
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) so += __shfl_xor_sync(0xffffffffu, so, d);
    if (cg == 0) o[((size_t)t * p.h_v + j) * kDim + dv] = p.scale * so;
  }
  if (p.hT) {
#pragma unroll
    for (int e = 0; e < 8; ++e) p.hT[head_off + (size_t)(8 * cg + e) * kDim + dv] = S[e];
  }
}

}  // namespace

cudaError_t launch_recurrence_f32(const Problem& p, cudaStream_t st) {
  dim3 grid(p.n_seqs, p.h_v, kDim / kRowsPerCta);
  recurrence_f32_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
