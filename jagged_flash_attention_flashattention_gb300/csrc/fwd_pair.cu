// fwd_pair.cu -- the jagged attention forward on CTA pairs (cta_group::2),
// jagged self-attention without a band, D = 128.
//
// Method as in fwd.cu ("TLX Block Attention", section 2, on packed
// sequences). Structure: "Desarrollo de Jagged Flash Attention para el
// modelo GEM", section "Optimización del proceso de Backward y dQ", last
// paragraph: the 2-CTA MMA of FA4, two CTAs of a cluster computing one
// product together to raise tensor-core utilisation.
//
// A tile is 512 query rows of one (sequence, head). Product x (x = 0, 1)
// covers rows [256x, 256x + 256): rank 0 holds rows [256x, 256x + 128) and
// rank 1 rows [256x + 128, 256x + 256), each in its own shared memory (Q)
// and tensor memory (S, P, O). Every product is one M = 256 MMA issued by
// rank 0, so each CTA loads only half of each K tile (64 keys) and half of
// each V tile (64 of the 128 columns) into its own shared memory (32 KB of
// loads per K/V step against 64 KB in the single-CTA kernel), and one
// instruction does the work of two. Measured against the single-CTA forward
// it is slower at the GEM and stress shapes (512-row tiles pad short
// sequences more, and every step waits on the other SM), so it is offered
// beside it rather than instead of it.
//
// Roles (384 threads in each CTA of the pair):
//   warp 0       TMA producer of this CTA's halves: Q rows, and through a
//                5-slot ring the K half (64 keys) of step j with the V half
//                (64 columns) of step j-1
//   warp 1       rank 0: MMA issuer for the pair; rank 1: forwards each
//                completed load of rank 1 to rank 0 (the products read both
//                CTAs' shared memory)
//   warp 2       tensor-memory allocation (with the peer's warp 2)
//   warps 2-3    clear the backward's dQ accumulator, as in fwd.cu
//   warps 4-7    softmax + correction + epilogue of this CTA's rows of product 0
//   warps 8-11   the same for product 1
// The softmax warps of both CTAs arrive on rank 0's barriers; rank 0's
// commits arrive on the barriers of both.
//
// Tensor memory of each CTA (512 columns): [0,128) S/P of product 0,
// [128,256) S/P of product 1, [256,384) O of product 0, [384,512) O of
// product 1.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103.cuh"

namespace jfa {
namespace {

using namespace dev;

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int QTILE = 128 * D * 2;   // 128 query rows (two 64-column boxes)
  static constexpr int KHALF = 64 * D * 2;    // 64 keys (two 64-column boxes of 8 KB)
  static constexpr int VHALF = 128 * 64 * 2;  // 128 keys x 64 columns
  static constexpr int SLOT = KHALF + VHALF;
  static constexpr int NSLOT = 5;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = 2 * QTILE;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * SLOT;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr uint32_t IDESC_QK = idesc_bf16(256, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16(256, D, 0, 1);
};

struct PairBars {
  uint64_t q_full[2], q_empty[2], s_full[2], o_full[2];
  uint64_t p_ready[2], o_free[2];  // rank 0: the softmax warps of both CTAs
  uint64_t peer_q[2];              // rank 0: rank 1's Q half of product x landed
  uint64_t slot_full[PairCfg::NSLOT], slot_empty[PairCfg::NSLOT], peer_slot[PairCfg::NSLOT];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PairBars) <= 512, "barrier area");

struct PairTile {
  int b, h, n_kv, kv_len;
  int prow0, prow1;  // rows of product 0 / 1 (both CTAs); 0: the product is skipped
  int nrow0, nrow1;  // this CTA's rows of product 0 / 1
  int q0;            // row of the tile's first query (tm_q, O)
  int kv0;           // first key row of the sequence (tm_khalf, tm_v)
  int64_t lse0;
};

__device__ __forceinline__ int64_t pair_off(const void *off, int idx64, int i) {
  return idx64 ? static_cast<const int64_t *>(off)[i] : (int64_t) static_cast<const int *>(off)[i];
}

// A tile outside the batch is empty, and sequence bounds are clamped to
// [0, T], whatever the tile list or the offsets hold.
__device__ __forceinline__ PairTile decode_pair(const FwdParams &p, int t, uint32_t rank) {
  PairTile d;
  d.b = p.tiles[3 * t];
  d.h = p.tiles[3 * t + 1];
  const int m = p.tiles[3 * t + 2];
  const bool in = d.b >= 0 && d.b < p.B && d.h >= 0 && d.h < p.H && m >= 0 && m < (1 << 21);
  const int64_t s0 = in ? min(max(pair_off(p.offsets, p.idx64, d.b), (int64_t)0), p.T) : 0;
  const int64_t e0 = in ? min(max(pair_off(p.offsets, p.idx64, d.b + 1), s0), p.T) : 0;
  const int L = (int)(e0 - s0);
  const int row0 = m * 512;
  d.prow0 = max(0, min(256, L - row0));
  d.prow1 = max(0, min(256, L - row0 - 256));
  d.nrow0 = max(0, min(128, L - row0 - 128 * (int)rank));
  d.nrow1 = max(0, min(128, L - row0 - 256 - 128 * (int)rank));
  d.n_kv = d.prow0 > 0 ? (L + 127) / 128 : 0;
  d.kv_len = L;
  d.q0 = (int)s0 + row0;
  d.kv0 = (int)s0;
  d.lse0 = (int64_t)d.h * p.Tq + s0 + row0;
  return d;
}

template <int NSLOT>
__device__ __forceinline__ void next_slot(int &slot, uint32_t &ph) {
  if (++slot == NSLOT) {
    slot = 0;
    ph ^= 1;
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    jfa_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using C = PairCfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  PairBars &bars = *reinterpret_cast<PairBars *>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)cluster_id_x();

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.q_full[x], 1);
      mbar_init(&bars.q_empty[x], 1);
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.o_full[x], 1);
      mbar_init(&bars.p_ready[x], 8);
      mbar_init(&bars.o_free[x], 8);
      mbar_init(&bars.peer_q[x], 1);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bars.slot_full[s], 1);
      mbar_init(&bars.slot_empty[s], 1);
      mbar_init(&bars.peer_slot[s], 1);
    }
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_khalf);
    prefetch_tmap(&p.tm_v);
  }
  if (warp == 2) tmem_alloc_pair(&bars.tmem_base, 512);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  const WaitCtl ctl{p.status, &bars.abort_flag, p.timeout_ns};
  const int tbeg = p.sm_ptr[pair];
  const int tend = p.sm_ptr[pair + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ArmedLoads armed;  // barriers 0-1 q_full, 2.. slot_full
      uint32_t qph = 0, sph = 0;
      int slot = 0;
      PairTile nxt{};
      if (tbeg < tend) nxt = decode_pair(p, tbeg, rank);
      for (int t = tbeg; t < tend; ++t) {
        const PairTile tl = nxt;
        if (t + 1 < tend) nxt = decode_pair(p, t + 1, rank);
        if (tl.n_kv == 0) continue;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if ((x ? tl.prow1 : tl.prow0) == 0) continue;
          if (!mbar_wait(&bars.q_empty[x], ((qph >> x) & 1) ^ 1, ctl, 1)) goto drain;
          qph ^= 1u << x;
          mbar_arrive_expect_tx(&bars.q_full[x], C::QTILE);
          armed.arm(x);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::OFF_Q + x * C::QTILE + c * 16384, &p.tm_q, &bars.q_full[x], c * 64,
                        tl.h, tl.q0 + 256 * x + 128 * (int)rank);
        }
        for (int j = 0; j <= tl.n_kv; ++j) {  // slot of step j: K_j half (j < n), V_{j-1} half (j > 0)
          if (!mbar_wait(&bars.slot_empty[slot], sph ^ 1, ctl, 2)) goto drain;
          const bool k_in = j < tl.n_kv, v_in = j > 0;
          mbar_arrive_expect_tx(&bars.slot_full[slot], (k_in ? C::KHALF : 0) + (v_in ? C::VHALF : 0));
          armed.arm(2 + slot);
          uint8_t *dst = smem + C::OFF_RING + slot * C::SLOT;
          if (k_in)
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(dst + c * 8192, &p.tm_khalf, &bars.slot_full[slot], c * 64, tl.h,
                          tl.kv0 + 128 * j + 64 * (int)rank);
          if (v_in)
            tma_load_3d(dst + C::KHALF, &p.tm_v, &bars.slot_full[slot], 64 * (int)rank, tl.h,
                        tl.kv0 + 128 * (j - 1));
          next_slot<C::NSLOT>(slot, sph);
        }
      }
    drain:  // every armed copy has landed before the CTA can exit
      armed.drain([&](int i) { return i < 2 ? &bars.q_full[i] : &bars.slot_full[i - 2]; }, p.timeout_ns);
    }
  }
  else if (warp == 2 || warp == 3) {
    // ----------------------------------- backward accumulator pre-clearing
    // As in fwd.cu: no waits, so the count block 0 records is true once the
    // kernel has finished.
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
  } else if (warp == 1 && rank == 1) {
    // ------------------------------------- rank 1: forward completed loads
    // Rank 0's products read rank 1's shared memory: each load of rank 1 is
    // passed on to rank 0 once it has landed, in the order rank 0 waits.
    if (lane == 0) {
      uint32_t qph = 0, sph = 0;
      int slot = 0;
      PairTile nxt{};
      if (tbeg < tend) nxt = decode_pair(p, tbeg, rank);
      for (int t = tbeg; t < tend; ++t) {
        const PairTile tl = nxt;
        if (t + 1 < tend) nxt = decode_pair(p, t + 1, rank);
        if (tl.n_kv == 0) continue;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if ((x ? tl.prow1 : tl.prow0) == 0) continue;
          if (!mbar_wait(&bars.q_full[x], (qph >> x) & 1, ctl, 5)) goto done;
          qph ^= 1u << x;
          mbar_arrive_cta(&bars.peer_q[x], 0);
        }
        for (int j = 0; j <= tl.n_kv; ++j) {
          if (!mbar_wait(&bars.slot_full[slot], sph, ctl, 6)) goto done;
          mbar_arrive_cta(&bars.peer_slot[slot], 0);
          next_slot<C::NSLOT>(slot, sph);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------- rank 0: the pair's MMAs
    if (lane == 0) {
      uint32_t qph = 0, pph = 0, oph = 0, sph = 0;
      int slot = 0;
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint32_t ring = smem_u32(smem + C::OFF_RING);
      const uint64_t k_desc = sdesc_sw128(ring, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(ring + C::KHALF, 16384, 1024);
      auto issue_qk = [&](int x, int kslot) {  // S_x = Q_x K^T: K rows [0,64) here, [64,128) in rank 1
        const uint64_t qd = q_desc + (uint64_t)(x * (C::QTILE >> 4));
        const uint64_t kd = k_desc + (uint64_t)(kslot * (C::SLOT >> 4));
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss_pair(tmem + x * 128, qd + ((((k >> 2) * 16384) + (k & 3) * 32) >> 4),
                      kd + ((((k >> 2) * 8192) + (k & 3) * 32) >> 4), C::IDESC_QK, k > 0);
      };
      auto issue_pv = [&](int x, int vslot, bool acc) {  // O_x += P_x V: V columns [0,64) here
        const uint64_t vd = v_desc + (uint64_t)(vslot * (C::SLOT >> 4));
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts_pair(tmem + 256 + x * 128, tmem + x * 128 + k * 8, vd + (k * 2048 >> 4), C::IDESC_PV,
                      (acc || k > 0) ? 1u : 0u);
      };
      auto wait_slot = [&](int s) -> bool {  // both CTAs' halves of the slot
        if (!mbar_wait(&bars.slot_full[s], sph, ctl, 11)) return false;
        return mbar_wait_cluster(&bars.peer_slot[s], sph, ctl, 12);
      };
      PairTile nxt{};
      if (tbeg < tend) nxt = decode_pair(p, tbeg, rank);
      for (int t = tbeg; t < tend; ++t) {
        const PairTile tl = nxt;
        if (t + 1 < tend) nxt = decode_pair(p, t + 1, rank);
        if (tl.n_kv == 0) continue;
        const uint32_t has = (tl.prow0 > 0 ? 1u : 0u) | (tl.prow1 > 0 ? 2u : 0u);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!(has >> x & 1)) continue;
          if (!mbar_wait(&bars.q_full[x], (qph >> x) & 1, ctl, 10)) goto done;
          if (!mbar_wait_cluster(&bars.peer_q[x], (qph >> x) & 1, ctl, 13)) goto done;
          qph ^= 1u << x;
        }
        // S_0 (slot of step 0: K_0 only).
        if (!wait_slot(slot)) goto done;
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!(has >> x & 1)) continue;
          issue_qk(x, slot);
          mma_commit_pair_both(&bars.s_full[x]);
          if (tl.n_kv == 1) mma_commit_pair_both(&bars.q_empty[x]);
        }
        mma_commit_pair_both(&bars.slot_empty[slot]);
        next_slot<C::NSLOT>(slot, sph);
        for (int j = 1; j <= tl.n_kv; ++j) {
          // One slot: V_{j-1}, and K_j unless this is the last step.
          const int ps = slot;
          if (!wait_slot(ps)) goto done;
          next_slot<C::NSLOT>(slot, sph);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!(has >> x & 1)) continue;
            if (!mbar_wait_cluster(&bars.p_ready[x], (pph >> x) & 1, ctl, 14)) goto done;
            pph ^= 1u << x;
            if (j == 1) {  // first PV of the tile overwrites O: both epilogues must be done with it
              if (!mbar_wait_cluster(&bars.o_free[x], ((oph >> x) & 1) ^ 1, ctl, 15)) goto done;
              oph ^= 1u << x;
            }
            tc_fence_after();
            issue_pv(x, ps, j > 1);
            if (j == tl.n_kv) mma_commit_pair_both(&bars.o_full[x]);
            if (j < tl.n_kv) {  // S_j = Q K_j^T
              issue_qk(x, ps);
              mma_commit_pair_both(&bars.s_full[x]);
              if (j == tl.n_kv - 1) mma_commit_pair_both(&bars.q_empty[x]);
            }
          }
          mma_commit_pair_both(&bars.slot_empty[ps]);
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax + epilogue
    // As in fwd.cu, for this CTA's 128 rows of product x; a CTA whose rows
    // of an issued product lie past the sequence end still takes part in
    // its barriers (its rows are neither computed nor stored).
    const int x = (warp - 4) >> 2;  // product
    const int wq = warp & 3;        // TMEM lane quarter
    const int r = wq * 32 + lane;   // row within this CTA's half
    const uint32_t tS = tmem + ((uint32_t)(wq * 32) << 16) + x * 128;
    const uint32_t tO = tmem + ((uint32_t)(wq * 32) << 16) + 256 + x * 128;
    const float sl2 = p.scale_log2;
    uint32_t sph = 0, oph = 0;
    __nv_bfloat16 *obase = static_cast<__nv_bfloat16 *>(p.o);
    auto arrive0 = [&](uint64_t *bar) {  // on rank 0's barrier
      if (rank == 0) mbar_arrive(bar); else mbar_arrive_cta(bar, 0);
    };
    PairTile nxt{};
    if (tbeg < tend) nxt = decode_pair(p, tbeg, rank);
    for (int t = tbeg; t < tend; ++t) {
      const PairTile tl = nxt;
      if (t + 1 < tend) nxt = decode_pair(p, t + 1, rank);
      if (tl.n_kv == 0 || (x ? tl.prow1 : tl.prow0) == 0) continue;
      const int nrows = x ? tl.nrow1 : tl.nrow0;
      const bool row_ok = r < nrows;
      const int64_t orow = tl.q0 + 256 * x + 128 * (int)rank + r;
      uint4 *optr = reinterpret_cast<uint4 *>(obase + (orow * p.H + tl.h) * D);
      const int vis_hi = tl.kv_len - 1;  // the last K/V tile is masked past the sequence end
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < tl.n_kv; ++j) {
        if (!mbar_wait(&bars.s_full[x], sph, ctl, 20 + x)) goto done;
        sph ^= 1;
        if (nrows > 0) {
          tc_fence_after();
          uint32_t s[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
          tmem_wait_ld();
          const int hi_rel = vis_hi - j * 128;
          if (hi_rel < 127) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c * 32 + i > hi_rel) s[c][i] = __float_as_uint(-INFINITY);
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
          if (j == 0) {
            m_run = m_tile;
          } else if (m_tile > m_run + 8.f) {
            alpha = ex2(m_run - m_tile);
            m_run = m_tile;
          }
          const float m_use = m_run == -INFINITY ? 0.f : m_run;
          float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(-m_use, -m_use);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 xx = fma2(make_float2(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])),
                                     sl2v, negm);
              const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
              sum2[i & 1] = add2(sum2[i & 1], pp);
              pk[i] = pack_bf16(pp.x, pp.y);
            }
            tmem_st16(tS + c * 16, pk);
          }
          l_run = l_run * alpha + ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y));
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
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
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive0(&bars.p_ready[x]);
      }
      // epilogue
      if (!mbar_wait(&bars.o_full[x], oph, ctl, 22 + x)) goto done;
      oph ^= 1;
      if (nrows > 0) {
        tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
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
          p.lse[tl.lse0 + 256 * x + 128 * (int)rank + r] =
              l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive0(&bars.o_free[x]);
    }
  }
done:
  if (rank == 0 && warp == 1 && lane == 0 && bars.abort_flag) {
    // Let any product still in flight finish before the tensor memory is freed.
    mma_commit_pair(&bars.drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars.drain, 0) && globaltimer() - t0 < p.timeout_ns) {
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's products or arrivals may touch it
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

int fwd_pair_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(384, 1, 1);
  cfg.gridDim = dim3(2, 1, 1);
  cfg.dynamicSmemBytes = PairCfg::SMEM;
  if (cudaFuncSetAttribute(jfa_fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairCfg::SMEM) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, jfa_fwd_pair_kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_fwd_pair(const FwdParams &p, int num_pairs, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(jfa_fwd_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM);
  if (e != cudaSuccess) return e;
  jfa_fwd_pair_kernel<<<2 * num_pairs, 384, PairCfg::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace jfa
