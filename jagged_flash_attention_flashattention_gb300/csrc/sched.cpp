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
          int32_t *tiles, std::vector<int32_t> *src_of = nullptr) {
  const int64_t n = (int64_t)all.size();
  std::vector<int32_t> order(n);
  std::iota(order.begin(), order.end(), 0);
  if (zigzag) {
    // Stable sort by work, largest first: a counting sort when the work
    // values span a modest range (they are token counts), else a merge sort;
    // both keep equal works in enumeration order.
    int64_t wmax = 0;
    bool small = true;
    for (const Tile &t : all) {
      if (t.work < 0) small = false;
      wmax = std::max(wmax, t.work);
    }
    if (small && wmax < (int64_t(1) << 20)) {
      std::vector<int32_t> start(wmax + 2, 0);
      for (const Tile &t : all) ++start[wmax - t.work + 1];  // bucket of work w: wmax - w
      for (int64_t w = 0; w <= wmax; ++w) start[w + 1] += start[w];
      for (int64_t i = 0; i < n; ++i) order[start[wmax - all[i].work]++] = (int32_t)i;
    } else {
      std::stable_sort(order.begin(), order.end(),
                       [&](int32_t a, int32_t b) { return all[a].work > all[b].work; });
    }
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
    if (src_of) (*src_of)[pos] = order[i];
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

namespace {

// Block-sparse attention: masks of 128 x 128 blocks, one [ceil(Lq / 128),
// ceil(Lk / 128)] row-major byte array per sequence (non-zero = the query
// block sees the key block), concatenated in sequence order. Forward tiles
// are 256 query rows (query blocks 2m and 2m + 1, the tile's two halves):
// entries are the key blocks either half sees, increasing, each with a bit
// per half; work = the keys in those blocks. Backward tiles are key blocks:
// entries are the 64-row query blocks whose 128-row block sees the key
// block, increasing; work = the query rows in them.
struct SparseTiles {
  std::vector<Tile> tiles;
  std::vector<int64_t> beg;       // [n + 1] entry ranges in enumeration order
  std::vector<int32_t> entries;
  std::vector<int32_t> meta;      // forward: [4 n] first / end step of half 0, of half 1
};

constexpr uint32_t kBlkSees0 = 1u << 29, kBlkSees1 = 1u << 30;

jfa_status enumerate_sparse(int64_t B, int H, jfa_op op, const void *q_off, const void *kv_off,
                            jfa_index_t idx, const uint8_t *masks, int64_t n_mask, bool fill,
                            SparseTiles *out, int64_t *count, int64_t *n_entries) {
  if (H < 1) return fail(JFA_ERR_INVALID_ARG, "H = %d < 1", H);
  if (op != JFA_OP_FWD && op != JFA_OP_BWD)
    return fail(JFA_ERR_INVALID_ARG, "op must be JFA_OP_FWD or JFA_OP_BWD");
  if (!q_off) q_off = kv_off;
  jfa_status st = check_host_offsets(kv_off, idx, B, -1);
  if (st != JFA_OK) return st;
  st = check_host_offsets(q_off, idx, B, -1);
  if (st != JFA_OK) return st;
  if (n_mask < 0) return fail(JFA_ERR_INVALID_ARG, "n_mask < 0");
  int64_t need = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t Lq = offset_at(q_off, idx, b + 1) - offset_at(q_off, idx, b);
    const int64_t Lk = offset_at(kv_off, idx, b + 1) - offset_at(kv_off, idx, b);
    need += ((Lq + 127) / 128) * ((Lk + 127) / 128);
  }
  if (n_mask != need)
    return fail(JFA_ERR_INVALID_ARG, "masks hold %lld blocks, the offsets need %lld",
                (long long)n_mask, (long long)need);
  if (need > 0 && !masks) return fail(JFA_ERR_INVALID_ARG, "masks is NULL");
  int64_t n = 0, ne = 0, moff = 0;
  std::vector<int32_t> ent;
  std::vector<int64_t> work, tb;
  std::vector<int32_t> meta;
  if (fill) {  // sizes from a counting pass, so the fill never reallocates
    int64_t cn = 0, cne = 0;
    jfa_status cst = enumerate_sparse(B, H, op, q_off, kv_off, idx, masks, n_mask, false, nullptr,
                                      &cn, &cne);
    if (cst != JFA_OK) return cst;
    out->tiles.reserve(cn);
    out->beg.reserve(cn + 1);
    out->entries.reserve(cne);
    if (op == JFA_OP_FWD) out->meta.reserve(4 * cn);
  }
  for (int64_t b = 0; b < B; ++b) {
    const int64_t Lq = offset_at(q_off, idx, b + 1) - offset_at(q_off, idx, b);
    const int64_t Lk = offset_at(kv_off, idx, b + 1) - offset_at(kv_off, idx, b);
    const int64_t nqb = (Lq + 127) / 128, nkb = (Lk + 127) / 128;
    const uint8_t *mk = masks ? masks + moff : nullptr;
    moff += nqb * nkb;
    auto sees = [&](int64_t qb, int64_t kb) { return qb < nqb && mk[qb * nkb + kb] != 0; };
    const int64_t n_m = op == JFA_OP_FWD ? (Lq + kFwdTileRows - 1) / kFwdTileRows : nkb;
    // Per tile of this sequence (shared by its H heads): entries, work, meta.
    tb.assign(n_m + 1, 0);
    ent.clear();
    work.assign(n_m, 0);
    meta.assign(4 * n_m, 0);
    for (int64_t m = 0; m < n_m; ++m) {
      tb[m] = (int64_t)ent.size();
      if (op == JFA_OP_FWD) {
        int first[2] = {-1, -1}, last[2] = {-1, -1};
        for (int64_t j = 0; j < nkb; ++j) {
          const bool s0 = sees(2 * m, j), s1 = sees(2 * m + 1, j);
          if (!s0 && !s1) continue;
          const int step = (int)(ent.size() - tb[m]);
          if (s0) { if (first[0] < 0) first[0] = step; last[0] = step; }
          if (s1) { if (first[1] < 0) first[1] = step; last[1] = step; }
          ent.push_back((int32_t)((uint32_t)j | (s0 ? kBlkSees0 : 0u) | (s1 ? kBlkSees1 : 0u)));
          work[m] += band_min(Lk, j * 128 + 128) - j * 128;
        }
        for (int x = 0; x < 2; ++x) {
          meta[4 * m + 2 * x] = first[x] < 0 ? 0 : first[x];
          meta[4 * m + 2 * x + 1] = first[x] < 0 ? 0 : last[x] + 1;
        }
      } else {
        for (int64_t qb = 0; qb < (Lq + kBwdQBlock - 1) / kBwdQBlock; ++qb) {
          if (!sees(qb / 2, m)) continue;
          ent.push_back((int32_t)qb);
          work[m] += band_min(Lq, qb * kBwdQBlock + kBwdQBlock) - qb * kBwdQBlock;
        }
      }
    }
    tb[n_m] = (int64_t)ent.size();
    n += n_m * H;
    ne += (int64_t)ent.size() * H;
    if (n >= (int64_t(1) << 31) / 3) return fail(JFA_ERR_INVALID_ARG, "too many tiles");
    if (ne >= (int64_t(1) << 31)) return fail(JFA_ERR_INVALID_ARG, "too many list entries");
    if (fill) {  // enumeration order b, h, m (the tie order of the stable sort)
      for (int h = 0; h < H; ++h)
        for (int64_t m = 0; m < n_m; ++m) {
          out->tiles.push_back({(int32_t)b, h, (int32_t)m, work[m]});
          out->beg.push_back((int64_t)out->entries.size());
          out->entries.insert(out->entries.end(), ent.begin() + tb[m], ent.begin() + tb[m + 1]);
          if (op == JFA_OP_FWD) out->meta.insert(out->meta.end(), &meta[4 * m], &meta[4 * m] + 4);
        }
    }
  }
  if (fill) out->beg.push_back((int64_t)out->entries.size());
  *count = n;
  if (n_entries) *n_entries = ne;
  return JFA_OK;
}

}  // namespace

extern "C" jfa_status jfa_sched_size_sparse(int64_t B, int H, jfa_op op,
                                            const void *host_q_offsets,
                                            const void *host_kv_offsets, jfa_index_t idx,
                                            const uint8_t *host_masks, int64_t n_mask,
                                            int64_t *n_tiles, int64_t *n_entries) {
  if (!n_tiles || !n_entries) return fail(JFA_ERR_INVALID_ARG, "n_tiles or n_entries is NULL");
  return enumerate_sparse(B, H, op, host_q_offsets, host_kv_offsets, idx, host_masks, n_mask,
                          false, nullptr, n_tiles, n_entries);
}

extern "C" jfa_status jfa_sched_build_sparse(int64_t B, int H, jfa_op op, int num_sms,
                                             const void *host_q_offsets,
                                             const void *host_kv_offsets, jfa_index_t idx,
                                             const uint8_t *host_masks, int64_t n_mask,
                                             int zigzag, int32_t *sm_ptr, int32_t *tiles,
                                             int32_t *list_ptr, int32_t *list, int32_t *meta) {
  if (num_sms < 1) return fail(JFA_ERR_INVALID_ARG, "num_sms = %d < 1", num_sms);
  if (!sm_ptr || !list_ptr) return fail(JFA_ERR_INVALID_ARG, "sm_ptr or list_ptr is NULL");
  SparseTiles all;
  int64_t n = 0, ne = 0;
  jfa_status st = enumerate_sparse(B, H, op, host_q_offsets, host_kv_offsets, idx, host_masks,
                                   n_mask, true, &all, &n, &ne);
  if (st != JFA_OK) return st;
  if (n > 0 && !tiles) return fail(JFA_ERR_INVALID_ARG, "tiles is NULL");
  if (ne > 0 && !list) return fail(JFA_ERR_INVALID_ARG, "list is NULL");
  if (op == JFA_OP_FWD && n > 0 && !meta) return fail(JFA_ERR_INVALID_ARG, "meta is NULL");
  std::vector<int32_t> src(n);
  deal(all.tiles, num_sms, zigzag, sm_ptr, tiles, &src);
  int64_t pos = 0;
  for (int64_t i = 0; i < n; ++i) {  // lists in dealt order
    const int32_t s = src[i];
    list_ptr[i] = (int32_t)pos;
    for (int64_t e = all.beg[s]; e < all.beg[s + 1]; ++e) list[pos++] = all.entries[e];
    if (op == JFA_OP_FWD)
      for (int c = 0; c < 4; ++c) meta[4 * i + c] = all.meta[4 * (int64_t)s + c];
  }
  list_ptr[n] = (int32_t)pos;
  return JFA_OK;
}
