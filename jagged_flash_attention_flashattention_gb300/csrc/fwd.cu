// fwd.cu -- persistent, warp-specialised attention forward for sm_103a,
// jagged self-attention and broadcast-Q.
//
// Method: "TLX Block Attention", section 2 (the standard FlashAttention loop:
// S = Q K^T per K/V tile, running row max m, correction alpha =
// exp(m_old - m_new), O = alpha O + exp(S - m) V, l = alpha l + rowsum,
// O /= l, L = m + log l stored for the backward pass), run directly on packed
// sequences delimited by an offsets tensor ("Desarrollo de Jagged Flash
// Attention para el modelo GEM", first section).
//
// Structure ("Cambios estructurales y gestión de memoria"; "A TLX nagyobb
// kontrollt ad a Triton fölött": persistent kernel, one CTA per SM working
// through many tiles; dedicated TMA-load, MMA, softmax and epilogue roles;
// multi-buffered K/V; score, P and softmax state sharing one tensor-memory
// allocation while the PV accumulator keeps its own):
//
//   warp 0       TMA producer: Q halves, then K/V tiles into a ring of pair
//                slots (K_j with V_{j-1}: one barrier per K/V step)
//   warp 1       MMA issuer: S = Q K^T into TMEM, O += P V from TMEM P
//   warp 2       owns the tensor-memory allocation
//   warps 2-3    (jagged, workspace sized for the backward) clear the
//                backward's fp32 dQ accumulator with coalesced 16-byte
//                stores, which overlaps that HBM-bound pass with this
//                tensor-bound kernel
//   warps 4-7    softmax + correction + epilogue for query rows   0..127
//   warps 8-11   softmax + correction + epilogue for query rows 128..255
//
// A tile is 256 query rows of one (sequence, head): two 128-row halves that
// share every K/V tile, so the tensor core works on one half while the
// other half's softmax runs. Each softmax thread owns one query row (one
// TMEM lane). P is written back as bf16 over the first half of its own S
// columns and read from there by the PV MMA. The correction is applied
// lazily: the running max is only raised when a tile's max exceeds it by
// more than 2^8 (log2 domain), so O rarely needs rescaling in TMEM; the
// final normalisation by l makes the result identical in exact arithmetic.
// The K/V loop is peeled: only the last K/V tile of a sequence is masked.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128) S/P of half A   [128,256) S/P of half B
//   [256,256+D) O of half A   [384,384+D) O of half B
#include <cuda_bf16.h>

#include "band.h"
#include "kernels.h"
#include "sm103.cuh"

namespace jfa {
namespace {

using namespace dev;

template <int D>
struct FwdCfg {
  static constexpr int TILE_BYTES = 128 * D * 2;  // one 128-row Q, K or V tile
  // K/V ring of pair slots: the slot of K/V step j holds K_j and V_{j-1},
  // the two tiles that step j's products read, so one barrier covers both.
  static constexpr int NSLOT = D == 128 ? 2 : 4;
  static constexpr int PAIR_BYTES = 2 * TILE_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * PAIR_BYTES;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, 0, 1);
};

constexpr int kTileRing = 8;  // dynamic scheduling: tile indices published ahead

struct FwdBars {
  uint64_t q_full[2], q_empty[2], s_full[2], p_ready[2], o_full[2], o_free[2];
  uint64_t drain;
  uint64_t tile_full[kTileRing], tile_empty[kTileRing];  // dynamic scheduling ring
  int4 ring[kTileRing];  // (b, h, m, 1) of a claimed tile, or (-1, 0, 0, 0): no more
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdTile {
  int b, h, n_kv, nrows0, nrows1;
  int kv_len;        // keys from the first loaded key to the end of the sequence
  int diag0;         // key (counted from the first loaded key) aligned with the tile's first query row
  int q_coord;       // row coordinate of the tile's first query row in tm_q
  int kv0;           // first key row loaded, in tm_k / tm_v
  int64_t out_row0;  // row of the tile's first query row in O
  int64_t lse0;      // index of that row's LSE
};

__device__ __forceinline__ int64_t load_off(const void *off, int idx64, int i) {
  return idx64 ? static_cast<const int64_t *>(off)[i] : (int64_t) static_cast<const int *>(off)[i];
}

// (b, h, m) of tile index t: from the list p.tiles, or, dynamic scheduling
// over the device enumeration (p.dyn == 2), from tile_base.
template <bool DYN>
__device__ __forceinline__ int4 tile_bhm(const FwdParams &p, int t) {
  if (DYN && p.dyn == 2) {  // sequence of tile t: the last b with tile_base[b] <= t
    int64_t lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int64_t mid = (lo + hi) >> 1;
      if (p.tile_base[mid] <= t) lo = mid; else hi = mid;
    }
    const int64_t s0 = min(max(load_off(p.offsets, p.idx64, (int)lo), (int64_t)0), p.T);
    const int64_t e0 = min(max(load_off(p.offsets, p.idx64, (int)lo + 1), s0), p.T);
    const int nm = max(1, (int)((e0 - s0 + 255) / 256));
    const int r = (int)(t - p.tile_base[lo]);
    return make_int4((int)lo, r / nm, r % nm, 1);
  }
  return make_int4(p.tiles[3 * t], p.tiles[3 * t + 1], p.tiles[3 * t + 2], 1);
}

// GEN: the band mask is compiled in (jfa_varlen_fwd with a window); without
// it every row sees all of its sequence's keys.
template <bool BCAST, bool GEN>
__device__ __forceinline__ FwdTile decode_bhm(const FwdParams &p, int4 bhm) {
  FwdTile d;
  d.b = bhm.x;
  d.h = bhm.y;
  const int m = bhm.z;
  // A tile outside this batch (a schedule built for another one) is empty,
  // and sequence bounds are clamped to [0, T]: no row past the tensors is
  // read or written whatever the tile list or the offsets hold.
  const bool in = d.b >= 0 && d.b < p.B && d.h >= 0 && d.h < p.H && m >= 0 && m < (1 << 22);
  const int64_t s0 = in ? min(max(load_off(p.offsets, p.idx64, d.b), (int64_t)0), p.T) : 0;
  const int64_t e0 = in ? min(max(load_off(p.offsets, p.idx64, d.b + 1), s0), p.T) : 0;
  const int L = (int)(e0 - s0);
  int64_t qs = 0;
  int Lq;
  if (BCAST) {
    Lq = in ? p.Lq : 0;
  } else {
    qs = in ? min(max(load_off(p.q_offsets, p.idx64, d.b), (int64_t)0), p.Tq) : 0;
    Lq = (int)(in ? min(max(load_off(p.q_offsets, p.idx64, d.b + 1), qs), p.Tq) - qs : 0);
  }
  const int row0 = m * 256;
  d.nrows0 = max(0, min(128, Lq - row0));
  d.nrows1 = max(0, min(128, Lq - row0 - 128));
  // Keys the tile's rows can see (all of them without a band mask), in
  // 128-key tiles: K/V tiles j0 .. j0 + n_kv - 1 of the sequence.
  int64_t lo = 0, hi = 0;
  if (d.nrows0 > 0)
    fwd_key_range(row0, row0 + d.nrows0 + d.nrows1, Lq, L, GEN ? p.win_left : -1,
                  GEN ? p.win_right : -1, &lo, &hi);
  const int j0 = (int)(lo / 128);
  d.n_kv = hi > lo ? (int)((hi + 127) / 128) - j0 : 0;
  d.kv_len = L - j0 * 128;
  d.diag0 = row0 + (L - Lq) - j0 * 128;
  d.kv0 = (int)s0 + j0 * 128;
  if (BCAST) {
    d.q_coord = row0;
    d.out_row0 = (int64_t)d.b * Lq + row0;
    d.lse0 = ((int64_t)d.b * p.H + d.h) * Lq + row0;
  } else {
    d.q_coord = (int)qs + row0;
    d.out_row0 = qs + row0;
    d.lse0 = (int64_t)d.h * p.Tq + qs + row0;
  }
  return d;
}

// decode_tile split in two for the pipelined decode: the loads (the list
// entry, the sequence's offsets as stored, the block list bounds) and the
// arithmetic, so that a role can issue the loads a tile ahead and use them a
// tile later without waiting. finish_tile(fetch_raw(...)) equals decode_tile;
// the one-ahead decode keeps the single function, whose code the masked
// instantiation measured faster with.
struct FwdRaw {
  int4 bhm;
  int64_t s0, e0, qs, qe;
  int ls, le;
};

template <bool BCAST, bool SP>
__device__ __forceinline__ FwdRaw fetch_raw(const FwdParams &p, int4 bhm, int t) {
  FwdRaw r;
  r.bhm = bhm;
  const bool in = bhm.x >= 0 && bhm.x < p.B && bhm.y >= 0 && bhm.y < p.H && bhm.z >= 0 && bhm.z < (1 << 22);
  r.s0 = in ? load_off(p.offsets, p.idx64, bhm.x) : 0;
  r.e0 = in ? load_off(p.offsets, p.idx64, bhm.x + 1) : 0;
  r.qs = (!BCAST && in) ? load_off(p.q_offsets, p.idx64, bhm.x) : 0;
  r.qe = (!BCAST && in) ? load_off(p.q_offsets, p.idx64, bhm.x + 1) : 0;
  r.ls = SP ? p.blk_ptr[t] : 0;
  r.le = SP ? p.blk_ptr[t + 1] : 0;
  return r;
}

// GEN: the band mask is compiled in (jfa_varlen_fwd with a window); without
// it every row sees all of its sequence's keys. SP: block-sparse masks (with
// GEN, no band).
template <bool BCAST, bool GEN, bool SP>
__device__ __forceinline__ FwdTile finish_tile(const FwdParams &p, const FwdRaw &r) {
  FwdTile d;
  d.b = r.bhm.x;
  d.h = r.bhm.y;
  const int m = r.bhm.z;
  // A tile outside this batch (a schedule built for another one) is empty,
  // and sequence bounds are clamped to [0, T]: no row past the tensors is
  // read or written whatever the tile list or the offsets hold.
  const bool in = d.b >= 0 && d.b < p.B && d.h >= 0 && d.h < p.H && m >= 0 && m < (1 << 22);
  const int64_t s0 = in ? min(max(r.s0, (int64_t)0), p.T) : 0;
  const int64_t e0 = in ? min(max(r.e0, s0), p.T) : 0;
  const int L = (int)(e0 - s0);
  int64_t qs = 0;
  int Lq;
  if (BCAST) {
    Lq = in ? p.Lq : 0;
  } else {
    qs = in ? min(max(r.qs, (int64_t)0), p.Tq) : 0;
    Lq = (int)(in ? min(max(r.qe, qs), p.Tq) - qs : 0);
  }
  const int row0 = m * 256;
  d.nrows0 = max(0, min(128, Lq - row0));
  d.nrows1 = max(0, min(128, Lq - row0 - 128));
  // Keys the tile's rows can see (all of them without a band mask), in
  // 128-key tiles: K/V tiles j0 .. j0 + n_kv - 1 of the sequence.
  int64_t lo = 0, hi = 0;
  if (d.nrows0 > 0)
    fwd_key_range(row0, row0 + d.nrows0 + d.nrows1, Lq, L, GEN ? p.win_left : -1,
                  GEN ? p.win_right : -1, &lo, &hi);
  const int j0 = (int)(lo / 128);
  d.n_kv = hi > lo ? (int)((hi + 127) / 128) - j0 : 0;
  d.kv_len = L - j0 * 128;
  d.diag0 = row0 + (L - Lq) - j0 * 128;
  d.kv0 = (int)s0 + j0 * 128;
  if (BCAST) {
    d.q_coord = row0;
    d.out_row0 = (int64_t)d.b * Lq + row0;
    d.lse0 = ((int64_t)d.b * p.H + d.h) * Lq + row0;
  } else {
    d.q_coord = (int)qs + row0;
    d.out_row0 = qs + row0;
    d.lse0 = (int64_t)d.h * p.Tq + qs + row0;
  }
  if (SP) {
    // Block-sparse: the tile's steps are its list entries, at most one per
    // key block of the sequence (no band: the keys start at the sequence's
    // first key, kv_len = the sequence's keys).
    const int nkb = (d.kv_len + 127) / 128;
    d.n_kv = d.nrows0 > 0 ? min(max(r.le - r.ls, 0), nkb) : 0;
  }
  return d;
}

// K/V steps [lo, hi) of the tile (counted from its first loaded K/V tile)
// that query half x can see. Without a band both halves walk every step;
// with one, e.g. causal, the first half skips the last tile. A half with
// rows but no step sees no key (cross attention): its O is 0. With a block
// mask, lo and hi - 1 are the first and last steps the half sees; the steps
// between them that it does not see are skipped by their list entries.
// (t: the tile's index in the list, for the block mask's per-tile steps)
template <bool GEN, bool SP>
__device__ __forceinline__ int2 half_steps(const FwdTile &tl, const FwdParams &p, int x, int t) {
  const int rows = x ? tl.nrows1 : tl.nrows0;
  if (rows == 0 || tl.n_kv == 0) return make_int2(0, 0);
  if (!GEN) return make_int2(0, tl.n_kv);
  if (SP) {
    // The range must start and end on steps the half sees (so that every role
    // takes the same first and last step); otherwise the half walks nothing.
    const int2 m = reinterpret_cast<const int2 *>(p.blk_meta)[2 * t + x];
    const int lo = min(max(m.x, 0), tl.n_kv), hi = min(max(m.y, 0), tl.n_kv);
    if (hi <= lo) return make_int2(0, 0);
    const int lst = p.blk_ptr[t];
    const bool ok = ((__ldg(p.blk_list + lst + lo) & __ldg(p.blk_list + lst + hi - 1)) >>
                     (kBlkSeesShift + x)) & 1;
    return ok ? make_int2(lo, hi) : make_int2(0, 0);
  }
  const int64_t first = (int64_t)tl.diag0 + x * 128, last = first + rows - 1;
  const int64_t lo = p.win_left < 0 ? 0 : max(first - p.win_left, (int64_t)0);
  const int64_t hi = p.win_right < 0 ? (int64_t)tl.kv_len - 1 : min(last + p.win_right, (int64_t)tl.kv_len - 1);
  if (hi < lo) return make_int2(0, 0);
  return make_int2((int)(lo / 128), (int)min(hi / 128 + 1, (int64_t)tl.n_kv));
}

// SP: block-sparse masks compiled in (with GEN, no band).
template <bool BCAST, bool GEN, bool DYN, bool SP>
__device__ __forceinline__ FwdTile decode_tile(const FwdParams &p, int t) {
  FwdTile d = decode_bhm<BCAST, GEN>(p, tile_bhm<DYN>(p, t));
  if (SP) {
    // Block-sparse: the tile's steps are its list entries, at most one per
    // key block of the sequence (no band: the keys start at the sequence's
    // first key, kv_len = the sequence's keys); the halves' step ranges are
    // clamped to the list.
    const int nkb = (d.kv_len + 127) / 128;
    d.n_kv = d.nrows0 > 0 ? min(max(p.blk_ptr[t + 1] - p.blk_ptr[t], 0), nkb) : 0;
  }
  return d;
}

// List entry of step j (lst: the tile's first entry): the key block (clamped
// to the sequence) in the low bits, a bit per query half that sees it.
// Without a block mask step j is key tile j, seen by both halves.
template <bool SP>
__device__ __forceinline__ uint32_t step_entry(const FwdParams &p, const FwdTile &tl, int lst, int j) {
  if (SP) {
    const uint32_t e = (uint32_t)__ldg(p.blk_list + lst + j);
    const uint32_t kb = min(e & kBlkIndex, (uint32_t)max((tl.kv_len - 1) >> 7, 0));
    return kb | (e & ~kBlkIndex);
  }
  return (uint32_t)j | (3u << kBlkSeesShift);
}
__device__ __forceinline__ bool half_sees(uint32_t e, int x) { return (e >> (kBlkSeesShift + x)) & 1u; }

template <int D, bool BCAST, bool GEN, bool DYN, bool SP>
__global__ void __launch_bounds__(384, 1) jfa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  // Static schedule, unmasked: the producer and the MMA thread pipeline their
  // tile decode (measured faster there; slower in the masked instantiation).
  constexpr bool PIPE = !DYN && !GEN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  FwdBars &bars = *reinterpret_cast<FwdBars *>(smem + C::OFF_BAR);
  uint64_t *slot_full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR + sizeof(FwdBars) + 8);
  uint64_t *slot_empty = slot_full + C::NSLOT;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.q_full[x], 1);
      mbar_init(&bars.q_empty[x], 1);
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.p_ready[x], 4);
      mbar_init(&bars.o_full[x], 1);
      mbar_init(&bars.o_free[x], 4);
    }
    mbar_init(&bars.drain, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], 1);
    }
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(&bars.tile_full[s], 1);
      mbar_init(&bars.tile_empty[s], 9);  // the MMA thread and the eight softmax warps
    }
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  if (warp == 2) tmem_alloc(&bars.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  const WaitCtl ctl{p.status, &bars.abort_flag, p.timeout_ns};
  // Static scheduling: this CTA's tiles tbeg .. tend-1 of the CSR lists.
  // Dynamic: ordinal k of this CTA's tiles is the k-th index the producer
  // claimed from the global queue and published in the shared ring.
  const int tbeg = DYN ? 0 : p.sm_ptr[blockIdx.x];
  const int tend = DYN ? 0 : p.sm_ptr[blockIdx.x + 1];
  // Dynamic: (b, h, m) of this CTA's tile k for the MMA thread and the
  // softmax warps (b = -1: no more), as the producer resolved it.
  // `mask`: the lanes that run the role (the whole warp in the softmax warps,
  // lane 0 alone in the MMA warp); lane 0's entry is broadcast to them.
  auto tile_at = [&](int k, unsigned mask) -> int4 {
    int4 v = make_int4(-1, 0, 0, 0);
    if (lane == 0) {
      const int s = k % kTileRing;
      if (mbar_wait(&bars.tile_full[s], (k / kTileRing) & 1, ctl, 4)) {
        const volatile int *e = reinterpret_cast<const volatile int *>(&bars.ring[s]);  // (the wait acquires)
        v = make_int4(e[0], e[1], e[2], 0);
        mbar_arrive(&bars.tile_empty[s]);
      }
    }
    return make_int4(__shfl_sync(mask, v.x, 0), __shfl_sync(mask, v.y, 0), __shfl_sync(mask, v.z, 0), 0);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ArmedLoads armed;  // barriers 0-1 q_full, 2.. slot_full
      uint32_t qph = 0;
      int slot = 0;
      uint32_t sph = 0;
      // Dynamic scheduling: claim tile indices from the global queue and
      // publish them two ordinals ahead of this thread's loads (the other
      // roles read ordinal k + 1 when they start ordinal k).
      int pub = 0;
      bool ended = false;
      const int64_t n_dyn = !DYN ? 0 : (p.dyn == 2 ? p.tile_base[p.B] : p.n_tiles);
      auto produce_at = [&](int k) -> int4 {
        while (pub <= k + 1 && !ended) {
          const int s = pub % kTileRing;
          if (!mbar_wait(&bars.tile_empty[s], ((pub / kTileRing) & 1) ^ 1, ctl, 3))
            return make_int4(-1, 0, 0, 0);
          const int g = atomicAdd(p.queue, 1);
          ended = g >= n_dyn;
          bars.ring[s] = ended ? make_int4(-1, 0, 0, 0) : tile_bhm<DYN>(p, g);
          mbar_arrive(&bars.tile_full[s]);  // (release: the entry is visible to the waiters)
          ++pub;
        }
        return k < pub ? bars.ring[k % kTileRing] : make_int4(-1, 0, 0, 0);
      };
      // The next tile is decoded one tile ahead (its index loads are off the
      // critical path at the tile switch).
      // (Dynamic: t counts this CTA's tiles and id is the index of tile t.)
      // Tile decode as in the MMA thread below.
      int4 bhm = DYN ? produce_at(0) : make_int4(-1, 0, 0, 0);
      FwdTile nxt{};
      if (DYN ? bhm.x >= 0 : (!PIPE && tbeg < tend))
        nxt = DYN ? decode_bhm<BCAST, GEN>(p, bhm) : decode_tile<BCAST, GEN, DYN, SP>(p, tbeg);
      FwdRaw raw{};
      int4 ent = make_int4(-1, 0, 0, 0);
      if (PIPE && tbeg < tend) {
        raw = fetch_raw<BCAST, SP>(p, tile_bhm<DYN>(p, tbeg), tbeg);
        if (tbeg + 1 < tend) ent = tile_bhm<DYN>(p, tbeg + 1);
      }
      for (int t = tbeg; DYN ? bhm.x >= 0 : t < tend; ++t) {
        FwdTile tl;
        if (DYN) {
          tl = nxt;
          bhm = produce_at(t + 1);
          if (bhm.x >= 0) nxt = decode_bhm<BCAST, GEN>(p, bhm);
        } else if (PIPE) {
          tl = finish_tile<BCAST, GEN, SP>(p, raw);
          if (t + 1 < tend) raw = fetch_raw<BCAST, SP>(p, ent, t + 1);
          if (t + 2 < tend) ent = tile_bhm<DYN>(p, t + 2);
        } else {
          tl = nxt;
          if (t + 1 < tend) nxt = decode_tile<BCAST, GEN, DYN, SP>(p, t + 1);
        }
        if (tl.n_kv == 0) continue;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int2 hs = half_steps<GEN, SP>(tl, p, x, t);
          if (hs.y <= hs.x) continue;  // no step: the half's Q is not needed
          if (!mbar_wait(&bars.q_empty[x], ((qph >> x) & 1) ^ 1, ctl, 1)) goto drain;
          qph ^= 1u << x;
          mbar_arrive_expect_tx(&bars.q_full[x], C::TILE_BYTES);
          armed.arm(x);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::OFF_Q + x * C::TILE_BYTES + c * 16384, &p.tm_q,
                        &bars.q_full[x], c * 64, tl.h, tl.q_coord + x * 128);
        }
        // Key tile of each step (its list entry with a block mask).
        const int lst = SP ? p.blk_ptr[t] : 0;
        uint32_t kb_cur = 0, kb_prev = 0;
        for (int j = 0; j <= tl.n_kv; ++j) {  // slot of step j: K_j (j < n) and V_{j-1} (j > 0)
          const bool k_in = j < tl.n_kv, v_in = j > 0;
          kb_prev = kb_cur;
          if (k_in) kb_cur = SP ? step_entry<SP>(p, tl, lst, j) & kBlkIndex : (uint32_t)j;
          if (!mbar_wait(&slot_empty[slot], sph ^ 1, ctl, 2)) goto drain;
          mbar_arrive_expect_tx(&slot_full[slot], (k_in + v_in) * C::TILE_BYTES);
          armed.arm(2 + slot);
          uint8_t *dst = smem + C::OFF_RING + slot * C::PAIR_BYTES;
          for (int c = 0; c < D / 64; ++c) {
            if (k_in)
              tma_load_3d(dst + c * 16384, &p.tm_k, &slot_full[slot], c * 64, tl.h,
                          tl.kv0 + (int)kb_cur * 128);
            if (v_in)
              tma_load_3d(dst + C::TILE_BYTES + c * 16384, &p.tm_v, &slot_full[slot], c * 64, tl.h,
                          tl.kv0 + (int)kb_prev * 128);
          }
          if (++slot == C::NSLOT) {
            slot = 0;
            sph ^= 1;
          }
        }
      }
    drain:  // every armed copy has landed before the CTA can exit
      armed.drain([&](int i) { return i < 2 ? &bars.q_full[i] : &slot_full[i - 2]; }, p.timeout_ns);
    }
  } else if (warp == 2 || warp == 3) {
    // ----------------------------------- backward accumulator pre-clearing
    // No waits here: the zeroing always runs to completion, so the count that
    // block 0 records is true once the kernel has finished.
    if (p.acc_zero != nullptr) {
      const int64_t per = (p.acc_n16 + gridDim.x - 1) / gridDim.x;
      const int64_t beg = (int64_t)blockIdx.x * per;
      const int64_t end = min(p.acc_n16, beg + per);
      uint4 *base = reinterpret_cast<uint4 *>(p.acc_zero);
      for (int64_t i = beg + (warp - 2) * 32 + lane; i < end; i += 64) base[i] = make_uint4(0, 0, 0, 0);
      if (blockIdx.x == 0 && warp == 2 && lane == 0)
        *reinterpret_cast<volatile uint64_t *>(reinterpret_cast<uint8_t *>(p.status) + kAccZeroedOff) =
            (uint64_t)p.acc_n16 * 16;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t qph = 0, pph = 0, oph = 0;  // phase bit x per half
      int slot = 0;
      uint32_t sph = 0;
      const uint32_t q_addr = smem_u32(smem + C::OFF_Q);
      const uint32_t ring = smem_u32(smem + C::OFF_RING);
      // Descriptors are built once; a k-step only adds its byte offset >> 4 to
      // the start-address field (a single add keeps the one issuing thread
      // ahead of the tensor core).
      const uint64_t q_desc = sdesc_sw128(q_addr, 16, 1024);
      const uint64_t ring_kdesc = sdesc_sw128(ring, 16, 1024);
      const uint64_t ring_vdesc = sdesc_sw128(ring, 16384, 1024);
      auto issue_qk = [&](int x, int kslot) {
        const uint64_t qd = q_desc + (uint64_t)(x * (C::TILE_BYTES >> 4));
        const uint64_t kd = ring_kdesc + (uint64_t)(kslot * (C::PAIR_BYTES >> 4));
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
          mma_ss(tmem + x * 128, qd + off, kd + off, C::IDESC_QK, k > 0);
        }
      };
      auto issue_pv = [&](int x, int vslot, bool acc) {
        const uint64_t vd = ring_vdesc + (uint64_t)((vslot * C::PAIR_BYTES + C::TILE_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + 256 + x * 128, tmem + x * 128 + k * 8, vd + (k * 2048 >> 4), C::IDESC_PV,
                 (acc || k > 0) ? 1u : 0u);
      };
      // Dynamic, and masked instantiations: the next tile is decoded one tile
      // ahead. Static unmasked (PIPE): the loads of tile t + 1's decode (its
      // offsets, from its list entry fetched a tile earlier) and of tile
      // t + 2's list entry are issued at the top of tile t and used at the top
      // of tile t + 1, so no dependent load is waited for at a tile switch.
      int4 bhm = DYN ? tile_at(0, 1u) : make_int4(-1, 0, 0, 0);
      FwdTile nxt{};
      if (DYN ? bhm.x >= 0 : (!PIPE && tbeg < tend))
        nxt = DYN ? decode_bhm<BCAST, GEN>(p, bhm) : decode_tile<BCAST, GEN, DYN, SP>(p, tbeg);
      FwdRaw raw{};
      int4 ent = make_int4(-1, 0, 0, 0);
      if (PIPE && tbeg < tend) {
        raw = fetch_raw<BCAST, SP>(p, tile_bhm<DYN>(p, tbeg), tbeg);
        if (tbeg + 1 < tend) ent = tile_bhm<DYN>(p, tbeg + 1);
      }
      for (int t = tbeg; DYN ? bhm.x >= 0 : t < tend; ++t) {
        FwdTile tl;
        if (DYN) {
          tl = nxt;
          bhm = tile_at(t + 1, 1u);
          if (bhm.x >= 0) nxt = decode_bhm<BCAST, GEN>(p, bhm);
        } else if (PIPE) {
          tl = finish_tile<BCAST, GEN, SP>(p, raw);
          if (t + 1 < tend) raw = fetch_raw<BCAST, SP>(p, ent, t + 1);
          if (t + 2 < tend) ent = tile_bhm<DYN>(p, t + 2);
        } else {
          tl = nxt;
          if (t + 1 < tend) nxt = decode_tile<BCAST, GEN, DYN, SP>(p, t + 1);
        }
        if (tl.n_kv == 0) continue;
        // Each half's steps [lo, hi): every step without a band.
        const int2 hs0 = half_steps<GEN, SP>(tl, p, 0, t), hs1 = half_steps<GEN, SP>(tl, p, 1, t);
        const uint32_t has = (hs0.y > hs0.x ? 1u : 0u) | (hs1.y > hs1.x ? 2u : 0u);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!(has >> x & 1)) continue;
          if (!mbar_wait(&bars.q_full[x], (qph >> x) & 1, ctl, 10)) goto done;
          qph ^= 1u << x;
        }
        // S_0 (slot of step 0: K_0 only).
        if (!mbar_wait(&slot_full[slot], sph, ctl, 11)) goto done;
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int2 hs = x ? hs1 : hs0;
          if (!(has >> x & 1) || hs.x != 0) continue;
          issue_qk(x, slot);
          mma_commit(&bars.s_full[x]);
          if (hs.y == 1) mma_commit(&bars.q_empty[x]);
        }
        mma_commit(&slot_empty[slot]);
        if (++slot == C::NSLOT) { slot = 0; sph ^= 1; }
        // List entries of steps j - 1, j and j + 1 (a block mask: which halves
        // see the step; otherwise both), the next one loaded a step ahead.
        uint32_t e_prev = 0, e_cur = 0, e_next = 0;
        const int lst = SP ? p.blk_ptr[t] : 0;
        if constexpr (SP) {
          e_cur = step_entry<SP>(p, tl, lst, 0);
          e_next = tl.n_kv > 1 ? step_entry<SP>(p, tl, lst, 1) : 0u;
        }
        for (int j = 1; j <= tl.n_kv; ++j) {
          if constexpr (SP) {
            e_prev = e_cur;
            e_cur = e_next;
            e_next = j + 1 < tl.n_kv ? step_entry<SP>(p, tl, lst, j + 1) : 0u;
          }
          // One slot: V_{j-1}, and K_j unless this is the last step.
          const int ps = slot;
          if (!mbar_wait(&slot_full[ps], sph, ctl, 12)) goto done;
          if (++slot == C::NSLOT) { slot = 0; sph ^= 1; }
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!(has >> x & 1)) continue;
            const int2 hs = x ? hs1 : hs0;
            if (j - 1 >= hs.x && j - 1 < hs.y && (!SP || half_sees(e_prev, x))) {  // O += P_{j-1} V_{j-1}
              if (!mbar_wait(&bars.p_ready[x], (pph >> x) & 1, ctl, 14)) goto done;
              pph ^= 1u << x;
              if (j - 1 == hs.x) {  // first PV of the tile overwrites O: epilogue must be done with it
                if (!mbar_wait(&bars.o_free[x], ((oph >> x) & 1) ^ 1, ctl, 15)) goto done;
                oph ^= 1u << x;
              }
              tc_fence_after();
              issue_pv(x, ps, j - 1 > hs.x);
              if (j == hs.y) mma_commit(&bars.o_full[x]);
            }
            if (j >= hs.x && j < hs.y && (!SP || half_sees(e_cur, x))) {  // S_j = Q K_j^T
              if (j == hs.x) tc_fence_after();
              issue_qk(x, ps);
              mma_commit(&bars.s_full[x]);
              if (j == hs.y - 1) mma_commit(&bars.q_empty[x]);
            }
          }
          mma_commit(&slot_empty[ps]);
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax + epilogue
    const int x = (warp - 4) >> 2;  // half
    const int wq = warp & 3;        // TMEM lane quarter
    const int r = wq * 32 + lane;   // row within the half
    const uint32_t tS = tmem + ((uint32_t)(wq * 32) << 16) + x * 128;
    const uint32_t tO = tmem + ((uint32_t)(wq * 32) << 16) + 256 + x * 128;
    const float sl2 = p.scale_log2;
    uint32_t sph = 0, oph = 0;
    __nv_bfloat16 *obase = static_cast<__nv_bfloat16 *>(p.o);
    // The next tile is decoded one tile ahead (its index loads are off the
    // critical path at the tile switch).
    // The next tile is decoded one tile ahead (its index loads are off the
    // critical path at the tile switch).
    int4 bhm = DYN ? tile_at(0, 0xffffffffu) : make_int4(-1, 0, 0, 0);
    FwdTile nxt{};
    if (DYN ? bhm.x >= 0 : tbeg < tend)
      nxt = DYN ? decode_bhm<BCAST, GEN>(p, bhm) : decode_tile<BCAST, GEN, DYN, SP>(p, tbeg);
    for (int t = tbeg; DYN ? bhm.x >= 0 : t < tend; ++t) {
      const FwdTile tl = nxt;
      if (DYN) {
        bhm = tile_at(t + 1, 0xffffffffu);
        if (bhm.x >= 0) nxt = decode_bhm<BCAST, GEN>(p, bhm);
      } else if (t + 1 < tend) {
        nxt = decode_tile<BCAST, GEN, DYN, SP>(p, t + 1);
      }
      const int nrows = x ? tl.nrows1 : tl.nrows0;
      if (nrows == 0) continue;
      const bool row_ok = r < nrows;
      const int64_t orow = tl.out_row0 + x * 128 + r;
      uint4 *optr = reinterpret_cast<uint4 *>(obase + (orow * p.H + tl.h) * D);
      const int2 hs = half_steps<GEN, SP>(tl, p, x, t);
      if (hs.y <= hs.x) {  // rows that see no key (no keys, or outside the band): O = 0, LSE = -inf
        if (row_ok) {
          for (int i = 0; i < D / 8; ++i) optr[i] = make_uint4(0, 0, 0, 0);
          p.lse[tl.lse0 + x * 128 + r] = -INFINITY;
        }
        continue;
      }
      // This row's visible keys [vis_lo, vis_hi], counted from the tile's
      // first loaded key: all of them, or the band (the last K/V tile is
      // masked past the sequence end).
      const int dg = tl.diag0 + x * 128 + r;
      const int vis_lo =
          (!GEN || p.win_left < 0) ? 0 : (int)max((int64_t)dg - p.win_left, (int64_t)-1);
      const int vis_hi = (!GEN || p.win_right < 0)
                             ? tl.kv_len - 1
                             : (int)min((int64_t)dg + p.win_right, (int64_t)tl.kv_len - 1);
      float m_run = -INFINITY, l_run = 0.f;
      const int lst = SP ? p.blk_ptr[t] : 0;
      for (int j = hs.x; j < hs.y; ++j) {
        const uint32_t e = SP ? step_entry<SP>(p, tl, lst, j) : 0u;  // key tile of the step, and who sees it
        if (SP && !half_sees(e, x)) continue;
        const int kt = SP ? (int)(e & kBlkIndex) : j;
        if (!mbar_wait(&bars.s_full[x], sph, ctl, 20 + x)) goto done;
        sph ^= 1;
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
        tmem_wait_ld();
        // Masked columns only where some row of the warp needs them: the
        // peeled tail past the sequence end and the edges of a band.
        const int lo_rel = vis_lo - kt * 128, hi_rel = vis_hi - kt * 128;
        // (without a band the condition is the same for every row: no vote)
        if (GEN ? __any_sync(0xffffffffu, lo_rel > 0 || hi_rel < 127) : hi_rel < 127) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i < lo_rel || c * 32 + i > hi_rel) s[c][i] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            mx[i & 7] = max3f(mx[i & 7], __uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1]));
        const float m_tile =
            fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
            sl2;
        float alpha = 1.f;
        if (j == hs.x) {
          m_run = m_tile;
        } else if (m_tile > m_run + 8.f) {  // also when every earlier key was masked (m_run = -inf)
          alpha = ex2(m_run - m_tile);
          m_run = m_tile;
        }
        // A row with every key so far masked keeps m_run = -inf; its
        // exponentials are then exp2(-inf - 0) = 0, not NaN.
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(-m_use, -m_use);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = fma2(make_float2(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])),
                                  sl2v, negm);
            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
            sum2[i & 1] = add2(sum2[i & 1], pp);
            pk[i] = pack_bf16(pp.x, pp.y);
          }
          tmem_st16(tS + c * 16, pk);
        }
        l_run = l_run * alpha + ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y));
        if (j > hs.x && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_ready[x]);
      }
      // epilogue
      if (!mbar_wait(&bars.o_full[x], oph, ctl, 22 + x)) goto done;
      oph ^= 1;
      tc_fence_after();
      {
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;  // a row that saw no key: O = 0
        const float2 inv2 = make_float2(inv_l, inv_l);
#pragma unroll 1
        for (int c = 0; c < D / 32; c += 2) {  // two 32-column chunks in flight
          uint32_t o[2][32];
          tmem_ld32(tO + c * 32, o[0]);
          tmem_ld32(tO + c * 32 + 32, o[1]);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = pack_bf16_mul(o[h][2 * i], o[h][2 * i + 1], inv2);
              st_global_v8(optr + (c + h) * 4, pk);
              st_global_v8(optr + (c + h) * 4 + 2, pk + 8);
            }
          }
        }
        if (row_ok)
          p.lse[tl.lse0 + x * 128 + r] =
              l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.o_free[x]);
    }
  }
done:
  if (warp == 1 && lane == 0 && bars.abort_flag) {
    // Let any MMA still in flight finish before the tensor memory is freed.
    mma_commit(&bars.drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars.drain, 0) && globaltimer() - t0 < p.timeout_ns) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BCAST, bool GEN, bool DYN, bool SP = false>
cudaError_t launch_t(const FwdParams &p, int num_sms, cudaStream_t st) {
  auto kern = jfa_fwd_kernel<D, BCAST, GEN, DYN, SP>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, 384, FwdCfg<D>::SMEM, st>>>(p);
  return cudaGetLastError();
}

// Per-sequence forward tile counts (H * ceil(L / 256)) as exclusive prefix
// sums, and the queue counter zeroed.
__global__ void __launch_bounds__(1024) fwd_enum_kernel(const FwdParams p, int64_t *tile_base,
                                                        int *queue) {
  __shared__ int64_t s_n[1024];
  const int t = threadIdx.x;
  const int64_t chunk = (p.B + 1023) / 1024;
  const int64_t b0 = min(p.B, (int64_t)t * chunk), b1 = min(p.B, b0 + chunk);
  auto count = [&](int64_t b) {
    const int64_t s0 = min(max(load_off(p.offsets, p.idx64, (int)b), (int64_t)0), p.T);
    const int64_t e0 = min(max(load_off(p.offsets, p.idx64, (int)b + 1), s0), p.T);
    return (int64_t)p.H * ((e0 - s0 + 255) / 256);
  };
  int64_t n = 0;
  for (int64_t b = b0; b < b1; ++b) n += count(b);
  s_n[t] = n;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int64_t a = t >= off ? s_n[t - off] : 0;
    __syncthreads();
    s_n[t] += a;
    __syncthreads();
  }
  int64_t base = s_n[t] - n;
  for (int64_t b = b0; b < b1; ++b) {
    tile_base[b] = base;
    base += count(b);
  }
  if (t == 1023) tile_base[p.B] = s_n[1023];
  if (t == 0) *queue = 0;
}

}  // namespace

cudaError_t launch_fwd(const FwdParams &p, int D, int num_sms, cudaStream_t st) {
  const bool bcast = p.Lq > 0;
  const bool gen = !bcast && (p.win_left >= 0 || p.win_right >= 0);
  if (p.blk_ptr != nullptr) {  // block-sparse: jagged, no band, static schedule
    if (bcast || gen || p.dyn) return cudaErrorNotSupported;
    return D == 128 ? launch_t<128, false, true, false, true>(p, num_sms, st)
                    : launch_t<64, false, true, false, true>(p, num_sms, st);
  }
  if (p.dyn) {  // dynamic scheduling: jagged without a band only
    if (bcast || gen) return cudaErrorNotSupported;
    return D == 128 ? launch_t<128, false, false, true>(p, num_sms, st)
                    : launch_t<64, false, false, true>(p, num_sms, st);
  }
  if (D == 128) {
    if (bcast) return launch_t<128, true, false, false>(p, num_sms, st);
    return gen ? launch_t<128, false, true, false>(p, num_sms, st)
               : launch_t<128, false, false, false>(p, num_sms, st);
  }
  if (bcast) return launch_t<64, true, false, false>(p, num_sms, st);
  return gen ? launch_t<64, false, true, false>(p, num_sms, st)
             : launch_t<64, false, false, false>(p, num_sms, st);
}

cudaError_t launch_fwd_enum(const FwdParams &p, int64_t *tile_base, int *queue, cudaStream_t st) {
  fwd_enum_kernel<<<1, 1024, 0, st>>>(p, tile_base, queue);
  return cudaGetLastError();
}

}  // namespace jfa
