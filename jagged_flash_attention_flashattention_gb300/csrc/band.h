// band.h -- the band mask and the tile ranges it implies, shared by the host
// scheduler and the kernels so that both walk exactly the same work.
//
// "Desarrollo de Jagged Flash Attention para el modelo GEM", section "Impacto
// en el desarrollo de modelos generativos" names causal, sliding-window and
// block-sparse masks as the extensions of the jagged kernels (built on the
// masked last K/V block, "Optimización del proceso de Backward y dQ"). Reading
// used here, the usual band mask: in a sequence with Lq queries and Lk keys,
// query i sees key j iff
//   (left < 0 || j >= i + shift - left) && (right < 0 || j <= i + shift + right),
// shift = Lk - Lq (bottom-right alignment). (-1, -1) is no mask, (-1, 0) causal.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define JFA_HD __host__ __device__ __forceinline__
#else
#define JFA_HD inline
#endif

namespace jfa {

constexpr int kFwdTileRows = 256;  // forward tile: two 128-row query halves
constexpr int kBwdTileKeys = 128;  // backward tile: 128 keys
constexpr int kBwdQBlock = 64;     // backward query block

JFA_HD int64_t band_max(int64_t a, int64_t b) { return a > b ? a : b; }
JFA_HD int64_t band_min(int64_t a, int64_t b) { return a < b ? a : b; }

// Keys [*lo, *hi) that query rows [r0, r1) can see (r1 > r0).
JFA_HD void fwd_key_range(int64_t r0, int64_t r1, int64_t Lq, int64_t Lk, int left, int right,
                          int64_t *lo, int64_t *hi) {
  const int64_t shift = Lk - Lq;
  const int64_t a = left < 0 ? 0 : band_max(0, r0 + shift - left);
  const int64_t b = right < 0 ? Lk : band_min(Lk, r1 - 1 + shift + right + 1);
  *lo = a;
  *hi = band_max(a, b);
}

// Query rows [*lo, *hi) that can see some key of [k0, k1) (k1 > k0).
JFA_HD void bwd_query_range(int64_t k0, int64_t k1, int64_t Lq, int64_t Lk, int left, int right,
                            int64_t *lo, int64_t *hi) {
  const int64_t shift = Lk - Lq;
  const int64_t a = right < 0 ? 0 : band_max(0, k0 - shift - right);
  const int64_t b = left < 0 ? Lq : band_min(Lq, k1 - 1 - shift + left + 1);
  *lo = a;
  *hi = band_max(a, b);
}

// The 64-row query blocks [*qb0, *qb0 + *nq) that backward key block n walks.
JFA_HD void bwd_query_blocks(int64_t n, int64_t Lq, int64_t Lk, int left, int right, int *qb0,
                             int *nq) {
  const int64_t k0 = n * kBwdTileKeys, k1 = band_min(Lk, k0 + kBwdTileKeys);
  int64_t lo, hi;
  bwd_query_range(k0, k1, Lq, Lk, left, right, &lo, &hi);
  *qb0 = (int)(lo / kBwdQBlock);
  *nq = hi > lo ? (int)((hi + kBwdQBlock - 1) / kBwdQBlock - lo / kBwdQBlock) : 0;
}

}  // namespace jfa
