// Segmentation rule of intra-card context parallelism, shared by the host
// planner and the kernels so both derive identical segments from the same
// cu_seqlens (integer arithmetic only: no floating-point rounding can differ).
//
// FlashQLA pages, section "AutoCP": the CP degree follows L = lambda * sqrt(N),
// N = chunks of the sequence, L = chunks per CP segment.
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define GDN_HD __host__ __device__ __forceinline__
#else
#define GDN_HD inline
#endif

namespace gdn {

constexpr int kChunk = 64;  // tokens per chunk
constexpr int kDim = 128;   // d_k = d_v

// floor(sqrt(x)), exact, by the digit-by-digit method.
GDN_HD uint64_t isqrt_u64(uint64_t x) {
  uint64_t r = 0, bit = 1ull << 62;
  while (bit > x) bit >>= 2;
  while (bit != 0) {
    if (x >= r + bit) {
      x -= r + bit;
      r = (r >> 1) + bit;
    } else {
      r >>= 1;
    }
    bit >>= 2;
  }
  return r;
}

GDN_HD int chunks_of(int64_t n_tokens) { return (int)((n_tokens + kChunk - 1) / kChunk); }

// L = round(lambda * sqrt(N)) with lambda = lambda_q8 / 256, at least 1.
GDN_HD int seg_len_chunks(int n_chunks, int lambda_q8) {
  const uint64_t X = (uint64_t)lambda_q8 * (uint64_t)lambda_q8 * (uint64_t)n_chunks;
  const int L = (int)((isqrt_u64(X) + 128) / 256);
  return L < 1 ? 1 : L;
}

// Segments of one sequence: one when CP is off, else ceil(N / L), at least one.
GDN_HD int seg_count(int n_chunks, int lambda_q8, bool cp_off) {
  if (cp_off || n_chunks <= 1) return 1;
  const int L = seg_len_chunks(n_chunks, lambda_q8);
  const int n = (n_chunks + L - 1) / L;
  return n < 1 ? 1 : n;
}

// First chunk of segment s (balanced split); seg_first(n_seg) == n_chunks.
GDN_HD int seg_first(int s, int n_chunks, int n_seg) {
  return (int)(((int64_t)s * n_chunks) / n_seg);
}

}  // namespace gdn
