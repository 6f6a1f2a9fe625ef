// Host LPT tile scheduler with a zigzag (boustrophedon) deal to SMs.
//
// "Desarrollo de Jagged Flash Attention para el modelo GEM", section
// "Optimizaciones específicas para el flujo de trabajo de GEM": all tiles are
// sorted on the host by K/V workload, largest first, and dealt to the SMs
// left to right on even passes and right to left on odd passes, so that the
// heavy tiles of long sequences spread over all SMs and the light ones fill
// in behind them. Readings where the article is silent (tile = (b, h, m),
// stable tie order, naive comparison order) are spelled out in jfa.h.
#include <algorithm>
#include <cstdarg>
#include <cstring>
#include <numeric>
#include <vector>

#include "band.h"
#include "host_common.h"

namespace jfa {

static thread_local char g_err[512] = {0};

jfa_status fail(jfa_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

jfa_status check_host_offsets(const void *off, jfa_index_t idx, int64_t B, int64_t T) {
  if (B < 0) return fail(JFA_ERR_INVALID_ARG, "B = %lld < 0", (long long)B);
  if (!off) return fail(JFA_ERR_INVALID_ARG, "offsets is NULL");
  if (idx != JFA_I32 && idx != JFA_I64) return fail(JFA_ERR_INVALID_ARG, "bad index type");
  if (offset_at(off, idx, 0) != 0) return fail(JFA_ERR_INVALID_ARG, "offsets[0] != 0");
  for (int64_t b = 0; b < B; ++b) {
    if (offset_at(off, idx, b + 1) < offset_at(off, idx, b))
      return fail(JFA_ERR_INVALID_ARG, "offsets decrease at b = %lld", (long long)b);
  }
  if (T >= 0 && offset_at(off, idx, B) != T)
    return fail(JFA_ERR_INVALID_ARG, "offsets[B] = %lld != T = %lld",
                (long long)offset_at(off, idx, B), (long long)T);
  if (offset_at(off, idx, B) >= (int64_t(1) << 31))
    return fail(JFA_ERR_INVALID_ARG, "total length >= 2^31");
  return JFA_OK;
}

}  // namespace jfa

using namespace jfa;

extern "C" const char *jfa_last_error(void) { return g_err; }

extern "C" const char *jfa_status_str(jfa_status s) {
  switch (s) {
    case JFA_OK: return "JFA_OK";
    case JFA_ERR_INVALID_ARG: return "JFA_ERR_INVALID_ARG";
    case JFA_ERR_UNSUPPORTED: return "JFA_ERR_UNSUPPORTED";
    case JFA_ERR_WORKSPACE: return "JFA_ERR_WORKSPACE";
    case JFA_ERR_CUDA: return "JFA_ERR_CUDA";
    case JFA_ERR_TIMEOUT: return "JFA_ERR_TIMEOUT";
  }
  return "JFA_ERR_UNKNOWN";
}

namespace {

struct Tile {
  int32_t b, h, m;
  int64_t work;
};

jfa_status enumerate(int64_t B, int H, int tile_rows, const void *off, jfa_index_t idx,
                     int64_t fixed_rows, int64_t fixed_work, std::vector<Tile> *out,
                     int64_t *count) {
  if (H < 1) return fail(JFA_ERR_INVALID_ARG, "H = %d < 1", H);
  if (tile_rows < 1) return fail(JFA_ERR_INVALID_ARG, "tile_rows = %d < 1", tile_rows);
  if (fixed_rows < 0 || fixed_work < 0) return fail(JFA_ERR_INVALID_ARG, "negative fixed size");
  jfa_status st = check_host_offsets(off, idx, B, -1);
  if (st != JFA_OK) return st;
  int64_t n = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t len = offset_at(off, idx, b + 1) - offset_at(off, idx, b);
    const int64_t rows = fixed_rows > 0 ? fixed_rows : len;
    const int64_t work = fixed_work > 0 ? fixed_work : len;
    const int64_t n_m = (rows + tile_rows - 1) / tile_rows;
    if (out) {
      for (int h = 0; h < H; ++h)
        for (int64_t m = 0; m < n_m; ++m) out->push_back({(int32_t)b, h, (int32_t)m, work});
    }
    n += n_m * H;
  }
  if (n >= (int64_t(1) << 31) / 3) return fail(JFA_ERR_INVALID_ARG, "too many tiles");
  *count = n;
  return JFA_OK;
}

}  // namespace

namespace {

// Tiles of the masked / cross (varlen) forward (tiles of 256 query rows) or
// backward (tiles of 128 keys); work = the length of the key range the
// tile's query rows can see (forward) or of the query range that can see the
// tile's keys (backward), both from band.h. Tiles with no work are kept: the
// forward writes O = 0 for their rows, the backward dK = dV = 0.
jfa_status enumerate_varlen(int64_t B, int H, jfa_op op, const void *q_off, const void *kv_off,
                            jfa_index_t idx, int left, int right, std::vector<Tile> *out,
                            int64_t *count) {
  if (H < 1) return fail(JFA_ERR_INVALID_ARG, "H = %d < 1", H);
  if (op != JFA_OP_FWD && op != JFA_OP_BWD)
    return fail(JFA_ERR_INVALID_ARG, "op must be JFA_OP_FWD or JFA_OP_BWD");
  if (left < -1 || right < -1) return fail(JFA_ERR_INVALID_ARG, "window bounds must be >= -1");
  if (!q_off) q_off = kv_off;
  jfa_status st = check_host_offsets(kv_off, idx, B, -1);
  if (st != JFA_OK) return st;
  st = check_host_offsets(q_off, idx, B, -1);
  if (st != JFA_OK) return st;
  int64_t n = 0;
  std::vector<int64_t> work;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t Lq = offset_at(q_off, idx, b + 1) - offset_at(q_off, idx, b);
    const int64_t Lk = offset_at(kv_off, idx, b + 1) - offset_at(kv_off, idx, b);
    const int64_t rows = op == JFA_OP_FWD ? Lq : Lk;
    const int64_t tr = op == JFA_OP_FWD ? kFwdTileRows : kBwdTileKeys;
    const int64_t n_m = (rows + tr - 1) / tr;
    if (out) {  // enumeration order b, h, m (the tie order of the stable sort)
      work.resize(n_m);
      for (int64_t m = 0; m < n_m; ++m) {
        int64_t lo, hi;
        if (op == JFA_OP_FWD)
          fwd_key_range(m * tr, band_min(Lq, m * tr + tr), Lq, Lk, left, right, &lo, &hi);
        else
          bwd_query_range(m * tr, band_min(Lk, m * tr + tr), Lq, Lk, left, right, &lo, &hi);
        work[m] = hi - lo;
      }
      for (int h = 0; h < H; ++h)
        for (int64_t m = 0; m < n_m; ++m) out->push_back({(int32_t)b, h, (int32_t)m, work[m]});
    }
    n += n_m * H;
    if (n >= (int64_t(1) << 31) / 3) return fail(JFA_ERR_INVALID_ARG, "too many tiles");
  }
  *count = n;
  return JFA_OK;
}

// Sorts (LPT, stable) or keeps the enumeration order and deals the tiles to
// the SMs, zigzag or round-robin, into the CSR output.
void deal(const std::vector<Tile> &all, int num_sms, int zigzag, int32_t *sm_ptr,
          int32_t *tiles) {
  const int64_t n = (int64_t)all.size();
  std::vector<int32_t> order(n);
  std::iota(order.begin(), order.end(), 0);
  if (zigzag) {
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return all[a].work > all[b].work; });
  }
  std::vector<int32_t> sm_of(n);
  std::vector<int32_t> cnt(num_sms, 0);
  for (int64_t i = 0; i < n; ++i) {
    const int64_t pass = i / num_sms;
    const int32_t j = (int32_t)(i % num_sms);
    const int32_t sm = (zigzag && (pass & 1)) ? num_sms - 1 - j : j;
    sm_of[i] = sm;
    ++cnt[sm];
  }
  sm_ptr[0] = 0;
  for (int s = 0; s < num_sms; ++s) sm_ptr[s + 1] = sm_ptr[s] + cnt[s];
  std::vector<int32_t> fill(sm_ptr, sm_ptr + num_sms);
  for (int64_t i = 0; i < n; ++i) {
    const Tile &t = all[order[i]];
    const int32_t pos = fill[sm_of[i]]++;
    tiles[3 * pos + 0] = t.b;
    tiles[3 * pos + 1] = t.h;
    tiles[3 * pos + 2] = t.m;
  }
}

}  // namespace

extern "C" jfa_status jfa_sched_size_varlen(int64_t B, int H, jfa_op op,
                                            const void *host_q_offsets,
                                            const void *host_kv_offsets, jfa_index_t idx,
                                            int64_t *n_tiles) {
  if (!n_tiles) return fail(JFA_ERR_INVALID_ARG, "n_tiles is NULL");
  return enumerate_varlen(B, H, op, host_q_offsets, host_kv_offsets, idx, -1, -1, nullptr,
                          n_tiles);
}

extern "C" jfa_status jfa_sched_build_varlen(int64_t B, int H, jfa_op op, int num_sms,
                                             const void *host_q_offsets,
                                             const void *host_kv_offsets, jfa_index_t idx,
                                             int window_left, int window_right, int zigzag,
                                             int32_t *sm_ptr, int32_t *tiles) {
  if (num_sms < 1) return fail(JFA_ERR_INVALID_ARG, "num_sms = %d < 1", num_sms);
  if (!sm_ptr) return fail(JFA_ERR_INVALID_ARG, "sm_ptr is NULL");
  std::vector<Tile> all;
  int64_t n = 0;
  jfa_status st = enumerate_varlen(B, H, op, host_q_offsets, host_kv_offsets, idx, window_left,
                                   window_right, &all, &n);
  if (st != JFA_OK) return st;
  if (n > 0 && !tiles) return fail(JFA_ERR_INVALID_ARG, "tiles is NULL");
  deal(all, num_sms, zigzag, sm_ptr, tiles);
  return JFA_OK;
}

extern "C" jfa_status jfa_sched_size(int64_t B, int H, int tile_rows, const void *host_offsets,
                                     jfa_index_t idx, int64_t fixed_rows, int64_t *n_tiles) {
  if (!n_tiles) return fail(JFA_ERR_INVALID_ARG, "n_tiles is NULL");
  return enumerate(B, H, tile_rows, host_offsets, idx, fixed_rows, 0, nullptr, n_tiles);
}

extern "C" jfa_status jfa_sched_build(int64_t B, int H, int tile_rows, int num_sms,
                                      const void *host_offsets, jfa_index_t idx,
                                      int64_t fixed_rows, int64_t fixed_work, int zigzag,
                                      int32_t *sm_ptr, int32_t *tiles) {
  if (num_sms < 1) return fail(JFA_ERR_INVALID_ARG, "num_sms = %d < 1", num_sms);
  if (!sm_ptr) return fail(JFA_ERR_INVALID_ARG, "sm_ptr is NULL");
  std::vector<Tile> all;
  int64_t n = 0;
  jfa_status st =
      enumerate(B, H, tile_rows, host_offsets, idx, fixed_rows, fixed_work, &all, &n);
  if (st != JFA_OK) return st;
  if (n > 0 && !tiles) return fail(JFA_ERR_INVALID_ARG, "tiles is NULL");
  deal(all, num_sms, zigzag, sm_ptr, tiles);
  return JFA_OK;
}
