// bwd.cu -- persistent, warp-specialised attention backward for sm_103a,
// jagged self-attention and broadcast-Q.
//
// Method ("TLX Block Attention", sections 2 and 4): with P rebuilt from the
// stored log-sum-exp, P = exp(scale * Q K^T - LSE), and Di = rowsum(dO * O):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Di),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
// Structure ("Desarrollo de Jagged Flash Attention para el modelo GEM",
// "Cambios estructurales y gestión de memoria" and "Optimización del proceso
// de Backward y dQ"): warp-specialised roles including a dQ-reduction group,
// early release of the dQ tensor memory so the MMA warp can start the next
// product, and, for broadcast-Q, a double-buffered shared-memory staging of
// the dQ partials that are summed over the whole batch.
//
// A tile is 128 key rows of one (sequence, head). dK and dV for those rows
// stay in tensor memory while the kernel walks every 64-row query block of
// the sequence (or the dense Q for broadcast-Q); Q and dO blocks stream
// through a ring of shared-memory stages (3 deep at D = 128, 7 at D = 64).
// Per query block:
//   S^T  = K Q^T        (M=128 keys, N=64 queries, K=D)      -> TMEM
//   dP^T = V dO^T                                            -> TMEM
//   P^T, dS^T computed by the compute warps (one key row per thread, on
//   packed fp32 pairs; LSE and Di are staged negated so that each of P and
//   dS is one packed FMA / add per pair);
//   LSE and Di = rowsum(dO * O) of the block's 64 query rows are formed
//   inline by the dQ warps, two blocks ahead of their dQ reduction (O rows
//   read from global memory, dO from the stage, bf16 products accumulated
//   in fp32 by mixed-precision FMAs; no separate pass);
//   dV  += P^T dO       (A = P^T bf16 from TMEM)
//   dK  += dS^T Q       (A = dS^T bf16 from TMEM)
//   dQ^T = K^T dS^T     (both operands MN-major in shared memory)  -> TMEM
// The dQ group reads dQ^T out of TMEM (one head-dim lane per thread; two
// TMEM buffers, so the next block's dQ^T product does not wait for the
// reduction), releases the TMEM at once, stages its 64 x 32 fp32 box in
// an 8 KB shared-memory buffer (scaled here only for broadcast-Q; the
// jagged cast applies the scale once to the sum) and adds it with a single TMA
// reduce-add (fewer, larger reductions measured faster than 32-row ones)
// into an fp32 accumulator in global memory: a workspace accumulator that a
// light kernel casts to bf16 at the end (jagged), or the caller's fp32 dQ
// itself (broadcast-Q, where dQ is a sum over the whole batch). The jagged
// accumulator starts at zero: a forward pass with the same workspace clears
// it and records the cleared byte count in the status block; otherwise a
// clearing kernel does it first, and the cast resets the count.
// dK and dV leave TMEM once per tile; at D = 128 each 128-byte half row is
// stored by four lanes (a shuffle transpose within lane quads), so a store
// instruction writes eight whole lines.
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM owner,
// warps 4-7 and 12-15 compute + dK/dV epilogue (two warps per TMEM lane
// quarter, each on half of the query columns), warps 8-11 LSE/Di staging +
// dQ reduction.
// Tensor memory columns: dV [0,128) dK [128,256) S/P [256,320)
// dP/dS [320,384) dQ^T [384,512) (two buffers).
#include <cuda_bf16.h>

#include "band.h"
#include "kernels.h"
#include "sm103.cuh"

namespace jfa {
namespace {

using namespace dev;

template <int D>
struct BwdCfg {
  static constexpr int KV_TILE = 128 * D * 2;  // 128-row K or V tile
  static constexpr int QT = 64 * D * 2;        // 64-row Q or dO tile
  static constexpr int QCHUNK = 64 * 128;      // one 64-column box of a 64-row tile
  static constexpr int NSTAGE = D == 128 ? 3 : 7;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_TILE;
  static constexpr int OFF_ZERO = 2 * KV_TILE;  // D = 64: zero rows padding K^T to M = 128
  static constexpr int ZERO_BYTES = D == 64 ? 16384 : 0;
  static constexpr int OFF_STAGE = OFF_ZERO + ZERO_BYTES;  // NSTAGE x (Q, dO)
  static constexpr int OFF_DS = OFF_STAGE + NSTAGE * 2 * QT;  // 128x64 bf16 dS^T
  static constexpr int OFF_DQS = OFF_DS + 16384;               // dQ staging: 4 warps x 8 KB
  static constexpr int OFF_LSE = OFF_DQS + 32768;              // [NSTAGE][64] -LSE, log2 units
  static constexpr int OFF_DI = OFF_LSE + NSTAGE * 256;        // [NSTAGE][64] -Di
  static constexpr int OFF_BAR = OFF_DI + NSTAGE * 256;
  static constexpr int SMEM = OFF_BAR + 512;
  static constexpr uint32_t KT_LBO = D == 128 ? 16384 : (OFF_ZERO - OFF_K);
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 64, 0, 0);
  static constexpr uint32_t IDESC_G = idesc_bf16(128, D, 0, 1);   // dV, dK
  static constexpr uint32_t IDESC_Q = idesc_bf16(128, 64, 1, 1);  // dQ^T
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum : uint32_t { COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 320, COL_DQ = 384 };

struct BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t stage_full[8], stage_empty[8], aux_full[8];
  uint64_t s_full, dp_full, p_ready, ds_ready, ds_free;
  uint64_t dq_full[2], dq_free[2];  // dQ^T double-buffered in TMEM
  uint64_t dkdv_full, dkdv_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdTile {
  int b, h, nq, nkv;  // query blocks to walk; valid key rows in this tile
  int qb0;            // first query block walked (blocks of 64 rows)
  int kv_row0;        // first key row (tm_k / tm_v / dK / dV)
  int qdiag0;         // query index aligned with the tile's first key (band mask)
  int q_row0;         // first query row of the sequence in tm_q and in the dQ accumulator
  int o_row0;         // first row of the sequence in O / dO
  int Lq;             // query rows of the sequence
  int64_t lse0;       // LSE index of query row 0 (jagged: + h*Tq; bcast: (b*H+h)*Lq)
  int prow0;          // deterministic dQ: partial row of query row 0 for this key block
  int lst;            // block-sparse: the tile's first list entry
};

__device__ __forceinline__ int64_t load_off(const void *off, int idx64, int i) {
  return idx64 ? static_cast<const int64_t *>(off)[i] : (int64_t) static_cast<const int *>(off)[i];
}

// GEN: the band mask and the deterministic dQ store are compiled in
// (jfa_varlen_bwd); without them every key sees all of its sequence's queries.
template <bool BCAST, bool GEN>
__device__ __forceinline__ BwdTile decode_tile(const BwdParams &p, int t) {
  BwdTile d;
  d.b = p.tiles[3 * t];
  d.h = p.tiles[3 * t + 1];
  const int n = p.tiles[3 * t + 2];
  // A tile outside this batch (a schedule built for another one) is empty,
  // and sequence bounds are clamped to [0, T]: no row past the tensors is
  // read or written whatever the tile list or the offsets hold.
  const bool in = d.b >= 0 && d.b < p.B && d.h >= 0 && d.h < p.H && n >= 0 && n < (1 << 23);
  const int64_t s0 = in ? min(max(load_off(p.offsets, p.idx64, d.b), (int64_t)0), p.T) : 0;
  const int64_t e0 = in ? min(max(load_off(p.offsets, p.idx64, d.b + 1), s0), p.T) : 0;
  const int L = (int)(e0 - s0);
  int64_t qs = 0;
  if (BCAST) {
    d.Lq = in ? p.Lq : 0;
  } else {
    qs = in ? min(max(load_off(p.q_offsets, p.idx64, d.b), (int64_t)0), p.Tq) : 0;
    d.Lq = (int)(in ? min(max(load_off(p.q_offsets, p.idx64, d.b + 1), qs), p.Tq) - qs : 0);
  }
  d.nkv = min(128, L - n * 128);
  d.qdiag0 = n * 128 - (L - d.Lq);
  d.qb0 = 0;
  d.nq = 0;
  if (d.nkv > 0)
    bwd_query_blocks(n, d.Lq, L, GEN ? p.win_left : -1, GEN ? p.win_right : -1, &d.qb0, &d.nq);
  d.kv_row0 = (int)s0 + n * 128;
  d.prow0 = 0;
  if (BCAST) {
    d.q_row0 = 0;
    d.o_row0 = d.b * p.Lq;
    d.lse0 = ((int64_t)d.b * p.H + d.h) * p.Lq;
  } else {
    d.q_row0 = (int)qs;
    d.o_row0 = (int)qs;
    d.lse0 = (int64_t)d.h * p.Tq + qs;
    if (GEN && p.det && d.nq > 0) d.prow0 = (int)(p.det_base[d.b] + (int64_t)n * ((d.Lq + 63) / 64 * 64));
  }
  d.lst = 0;
  if (GEN && p.blk_ptr != nullptr) {  // block-sparse: the query blocks of the tile's list
    d.lst = p.blk_ptr[t];
    d.qb0 = 0;
    d.nq = d.nkv > 0 ? min(max(p.blk_ptr[t + 1] - d.lst, 0), (d.Lq + 63) / 64) : 0;
  }
  return d;
}

// Query block (of 64 rows, counted in the sequence) of the tile's i-th step:
// consecutive from qb0, or the i-th list entry (clamped to the sequence)
// with a block mask.
template <bool GEN>
__device__ __forceinline__ int query_block(const BwdParams &p, const BwdTile &tl, int i) {
  if (GEN && p.blk_ptr != nullptr)
    return min((int)((uint32_t)__ldg(p.blk_list + tl.lst + i) & 0xffffffu), max((tl.Lq + 63) / 64 - 1, 0));
  return tl.qb0 + i;
}

// Walks the (tile, query block) sequence of one CTA, skipping empty tiles.
template <bool BCAST, bool GEN>
struct BlockIter {
  int t, tend, i;
  bool valid;
  BwdTile tl;
  __device__ __forceinline__ void seek(const BwdParams &p) {
    valid = false;
    for (; t < tend; ++t) {
      tl = decode_tile<BCAST, GEN>(p, t);
      if (tl.nq > 0 && tl.nkv > 0) {
        valid = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void next(const BwdParams &p) {
    if (++i >= tl.nq) {
      i = 0;
      ++t;
      seek(p);
    }
  }
};

template <int D, bool BCAST, bool GEN>
__global__ void __launch_bounds__(512, 1) jfa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  BwdBars &bars = *reinterpret_cast<BwdBars *>(smem + C::OFF_BAR);
  float *lse_s = reinterpret_cast<float *>(smem + C::OFF_LSE);
  float *di_s = reinterpret_cast<float *>(smem + C::OFF_DI);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
    if (threadIdx.x == 0) p.status[0] = 6;
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    mbar_init(&bars.kv_empty, 1);
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&bars.stage_full[s], 1);
      mbar_init(&bars.stage_empty[s], 9);  // MMA commit + the eight compute warps
      mbar_init(&bars.aux_full[s], 4);     // LSE and Di of the block, from the dQ warps
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p_ready, 8);
    mbar_init(&bars.ds_ready, 8);
    mbar_init(&bars.ds_free, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.dq_full[x], 1);
      mbar_init(&bars.dq_free[x], 4);
    }
    mbar_init(&bars.dkdv_full, 1);
    mbar_init(&bars.dkdv_free, 8);
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (C::ZERO_BYTES > 0) {
    uint4 *z = reinterpret_cast<uint4 *>(smem + C::OFF_ZERO);
    for (int i = threadIdx.x; i < C::ZERO_BYTES / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_do);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_dqacc);
  }
  if (warp == 2) tmem_alloc(&bars.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  const WaitCtl ctl{p.status, &bars.abort_flag, p.timeout_ns};
  const int tbeg = p.sm_ptr[blockIdx.x];
  const int tend = p.sm_ptr[blockIdx.x + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ArmedLoads armed;  // barrier 0 kv_full, 1.. stage_full
      uint32_t kvph = 0, eph = 0;
      int qb = 0;
      // The next tile is decoded one tile ahead (its index loads are off the
      // critical path at the tile switch).
      BwdTile nxt{};
      if (tbeg < tend) nxt = decode_tile<BCAST, GEN>(p, tbeg);
      for (int t = tbeg; t < tend; ++t) {
        const BwdTile tl = nxt;
        if (t + 1 < tend) nxt = decode_tile<BCAST, GEN>(p, t + 1);
        if (tl.nq == 0 || tl.nkv <= 0) continue;
        // The tile's query blocks stream through the stages; block 0's stage
        // does not depend on the K/V buffer, so it is loaded before waiting
        // for the previous tile to release K and V (its slot frees about two
        // blocks before that tile ends) and arrives with them, not after.
        for (int i = 0; i < tl.nq; ++i, ++qb) {
          const int s = qb % C::NSTAGE;
          const int qr = query_block<GEN>(p, tl, i) * 64;  // first query row of the block in the sequence
          if (!mbar_wait(&bars.stage_empty[s], bit(eph, s) ^ 1, ctl, 2)) goto drain;
          eph ^= 1u << s;
          mbar_arrive_expect_tx(&bars.stage_full[s], 2 * C::QT);
          armed.arm(1 + s);
          uint8_t *st = smem + C::OFF_STAGE + s * 2 * C::QT;
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(st + c * C::QCHUNK, &p.tm_q, &bars.stage_full[s], c * 64, tl.h,
                        tl.q_row0 + qr);
            tma_load_3d(st + C::QT + c * C::QCHUNK, &p.tm_do, &bars.stage_full[s], c * 64, tl.h,
                        tl.o_row0 + qr);
          }
          if (i == 0) {  // then K and V, once the previous tile is done with them
            if (!mbar_wait(&bars.kv_empty, kvph ^ 1, ctl, 1)) goto drain;
            kvph ^= 1;
            mbar_arrive_expect_tx(&bars.kv_full, 2 * C::KV_TILE);
            armed.arm(0);
            for (int c = 0; c < D / 64; ++c) {
              tma_load_3d(smem + C::OFF_K + c * 16384, &p.tm_k, &bars.kv_full, c * 64, tl.h, tl.kv_row0);
              tma_load_3d(smem + C::OFF_V + c * 16384, &p.tm_v, &bars.kv_full, c * 64, tl.h, tl.kv_row0);
            }
          }
        }
      }
    drain:  // every armed copy has landed before the CTA can exit
      armed.drain([&](int i) { return i == 0 ? &bars.kv_full : &bars.stage_full[i - 1]; }, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kvph = 0, fph = 0, pph = 0, dsph = 0, dqfph = 0, dkdvph = 0;
      int qb = 0;
      const uint32_t k_a = smem_u32(smem + C::OFF_K);
      const uint32_t v_a = smem_u32(smem + C::OFF_V);
      const uint32_t st_a = smem_u32(smem + C::OFF_STAGE);
      const uint32_t ds_a = smem_u32(smem + C::OFF_DS);
      // Descriptors are built once per operand; k-steps add offset >> 4 to the
      // start-address field (keeps the single issuing thread cheap).
      const uint64_t k_kmaj = sdesc_sw128(k_a, 16, 1024), v_kmaj = sdesc_sw128(v_a, 16, 1024);
      const uint64_t st_kmaj = sdesc_sw128(st_a, 16, 1024);
      const uint64_t st_mn = sdesc_sw128(st_a, C::QCHUNK, 1024);
      const uint64_t kT_mn = sdesc_sw128(k_a, C::KT_LBO, 1024);
      const uint64_t ds_mn = sdesc_sw128(ds_a, 8192, 1024);
      // S^T (or dP^T) = X Y^T, X = K (or V) [128 x D], Y = Q (or dO) [64 x D], both K-major.
      auto issue_xyT = [&](uint32_t dcol, uint64_t xd, uint64_t yd) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tmem + dcol, xd + (((k >> 2) * 16384 + (k & 3) * 32) >> 4),
                 yd + (((k >> 2) * C::QCHUNK + (k & 3) * 32) >> 4), C::IDESC_S, k > 0);
      };
      // dV (or dK) += A-from-TMEM x Y, Y = dO (or Q) [64 x D] MN-major. The bf16
      // A operand of query columns [32h, 32h+32) sits at TMEM columns
      // [32h, 32h+16) of its region (each compute warp overwrites only its own
      // scores), so k-step k reads column (k / 2) * 32 + (k % 2) * 8.
      auto issue_grad = [&](uint32_t dcol, uint32_t acol, uint64_t yd, bool acc) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + dcol, tmem + acol + (k >> 1) * 32 + (k & 1) * 8, yd + (k * 2048 >> 4),
                 C::IDESC_G, (acc || k > 0) ? 1u : 0u);
      };
      // The next tile is decoded one tile ahead (its index loads are off the
      // critical path at the tile switch).
      BwdTile nxt{};
      if (tbeg < tend) nxt = decode_tile<BCAST, GEN>(p, tbeg);
      for (int t = tbeg; t < tend; ++t) {
        const BwdTile tl = nxt;
        if (t + 1 < tend) nxt = decode_tile<BCAST, GEN>(p, t + 1);
        if (tl.nq == 0 || tl.nkv <= 0) continue;
        if (!mbar_wait(&bars.kv_full, kvph, ctl, 10)) goto done;
        kvph ^= 1;
        for (int i = 0; i < tl.nq; ++i, ++qb) {
          const int s = qb % C::NSTAGE;
          const uint32_t q_off = (uint32_t)(s * 2 * C::QT) >> 4, do_off = q_off + (C::QT >> 4);
          if (i == 0) {
            if (!mbar_wait(&bars.stage_full[s], bit(fph, s), ctl, 11)) goto done;
            fph ^= 1u << s;
            tc_fence_after();
            issue_xyT(COL_S, k_kmaj, st_kmaj + q_off);
            mma_commit(&bars.s_full);
            issue_xyT(COL_DP, v_kmaj, st_kmaj + do_off);
            mma_commit(&bars.dp_full);
          }
          if (!mbar_wait(&bars.p_ready, pph, ctl, 12)) goto done;
          pph ^= 1;
          if (i == 0) {  // dK/dV accumulators must have been drained by the previous epilogue
            if (!mbar_wait(&bars.dkdv_free, dkdvph ^ 1, ctl, 13)) goto done;
            dkdvph ^= 1;
          }
          tc_fence_after();
          issue_grad(COL_DV, COL_S, st_mn + do_off, i > 0);
          const bool more = i + 1 < tl.nq;
          const int s2 = (qb + 1) % C::NSTAGE;
          const uint32_t q2_off = (uint32_t)(s2 * 2 * C::QT) >> 4;
          if (more) {
            if (!mbar_wait(&bars.stage_full[s2], bit(fph, s2), ctl, 14)) goto done;
            fph ^= 1u << s2;
            tc_fence_after();
            issue_xyT(COL_S, k_kmaj, st_kmaj + q2_off);
            mma_commit(&bars.s_full);
          }
          if (!mbar_wait(&bars.ds_ready, dsph, ctl, 15)) goto done;
          dsph ^= 1;
          tc_fence_after();
          issue_grad(COL_DK, COL_DP, st_mn + q_off, i > 0);
          mma_commit(&bars.stage_empty[s]);
          const int qbuf = qb & 1;
          if (!mbar_wait(&bars.dq_free[qbuf], bit(dqfph, qbuf) ^ 1, ctl, 16)) goto done;
          dqfph ^= 1u << qbuf;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss(tmem + COL_DQ + qbuf * 64, kT_mn + (k * 2048 >> 4), ds_mn + (k * 2048 >> 4),
                   C::IDESC_Q, k > 0);
          mma_commit(&bars.dq_full[qbuf]);
          mma_commit(&bars.ds_free);
          if (more) {
            issue_xyT(COL_DP, v_kmaj, st_kmaj + q2_off + (C::QT >> 4));
            mma_commit(&bars.dp_full);
          }
        }
        mma_commit(&bars.dkdv_full);
        mma_commit(&bars.kv_empty);
      }
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // ------------------------------------------ compute + dK/dV epilogue
    // Eight warps: two per TMEM lane quarter, each taking half of the block's
    // 64 query columns (and half of the head dimension in the epilogue), so
    // two warps per scheduler hide each other's TMEM / MUFU latency.
    const int wq = warp & 3;
    const int ch = warp >= 12 ? 1 : 0;  // column half
    const int r = wq * 32 + lane;       // key row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t aph = 0, sph = 0, dpph = 0, dsfph = 0, dkdvph = 0;
    int qb = 0;
    // The next tile is decoded one tile ahead (its index loads are off the
    // critical path at the tile switch).
    BwdTile nxt{};
    if (tbeg < tend) nxt = decode_tile<BCAST, GEN>(p, tbeg);
    for (int t = tbeg; t < tend; ++t) {
      const BwdTile tl = nxt;
      if (t + 1 < tend) nxt = decode_tile<BCAST, GEN>(p, t + 1);
      if (tl.nkv <= 0) continue;
      const bool kv_ok = r < tl.nkv;
      if (tl.nq == 0) {  // keys that no query sees (band mask, or no queries): dK = dV = 0
        if (kv_ok) {
          const int64_t grow = (int64_t)(tl.kv_row0 + r) * p.H + tl.h;
          uint4 *dvp = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dv) + grow * D);
          uint4 *dkp = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dk) + grow * D);
          for (int c = ch * (D / 16); c < (ch + 1) * (D / 16); ++c) {
            dvp[c] = make_uint4(0, 0, 0, 0);
            dkp[c] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      const bool warp_ok = __all_sync(0xffffffffu, kv_ok);  // uniform: no per-element masking
      // Queries that see this thread's key (band mask; every query without one).
      const int kq = tl.qdiag0 + r;
      const int vq_lo =
          (!GEN || p.win_right < 0) ? 0 : (int)max((int64_t)kq - p.win_right, (int64_t)-1);
      const int vq_hi = (!GEN || p.win_left < 0) ? (1 << 30)  // (rows past Lq already have P = 0)
                                       : (int)min((int64_t)kq + p.win_left, (int64_t)1 << 30);
      for (int i = 0; i < tl.nq; ++i, ++qb) {
        const int s = qb % C::NSTAGE;
        if (!mbar_wait(&bars.aux_full[s], bit(aph, s), ctl, 20)) goto done;
        aph ^= 1u << s;
        // P^T: this thread's key row against 32 of the block's query columns.
        if (!mbar_wait(&bars.s_full, sph, ctl, 21)) goto done;
        sph ^= 1;
        tc_fence_after();
        float pr[32];
        {
          const float4 *l4 = reinterpret_cast<const float4 *>(lse_s + s * 64 + ch * 32);
          uint32_t a[32];
          tmem_ld32(tmem + lane_off + COL_S + ch * 32, a);
          tmem_wait_ld();
          // (the staged LSE is negated: x = S * scale * log2e - LSE in one packed FMA)
          const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 lv = l4[c];
            const float2 x0 = fma2(make_float2(__uint_as_float(a[c * 4]), __uint_as_float(a[c * 4 + 1])), sl2v,
                                   make_float2(lv.x, lv.y));
            const float2 x1 = fma2(make_float2(__uint_as_float(a[c * 4 + 2]), __uint_as_float(a[c * 4 + 3])),
                                   sl2v, make_float2(lv.z, lv.w));
            pr[c * 4] = ex2(x0.x);
            pr[c * 4 + 1] = ex2(x0.y);
            pr[c * 4 + 2] = ex2(x1.x);
            pr[c * 4 + 3] = ex2(x1.y);
          }
          if (!warp_ok) {  // key rows past the sequence (last tile only) have P = 0
#pragma unroll
            for (int i = 0; i < 32; ++i) pr[i] = kv_ok ? pr[i] : 0.f;
          }
          if constexpr (GEN) {  // band edges: P = 0 for the queries of these 32 columns that cannot see this key
            // (a block mask has no band: vq_lo = 0, vq_hi = 2^30, and nothing
            // is masked whatever the block, so its position is not looked up)
            const int cb = (tl.qb0 + i) * 64 + ch * 32;
            const int lo_rel = vq_lo - cb, hi_rel = vq_hi - cb;
            if (__any_sync(0xffffffffu, lo_rel > 0 || hi_rel < 31)) {
#pragma unroll
              for (int c = 0; c < 32; ++c) pr[c] = (c < lo_rel || c > hi_rel) ? 0.f : pr[c];
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(pr[2 * c], pr[2 * c + 1]);
          // P over this warp's own score columns only (the other half may not be read yet)
          tmem_st16(tmem + lane_off + COL_S + ch * 32, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_ready);
        // dS^T = P^T * (dP^T - Di)
        if (!mbar_wait(&bars.dp_full, dpph, ctl, 22)) goto done;
        dpph ^= 1;
        tc_fence_after();
        {
          const float4 *d4 = reinterpret_cast<const float4 *>(di_s + s * 64 + ch * 32);
          uint32_t a[32];
          tmem_ld32(tmem + lane_off + COL_DP + ch * 32, a);
          tmem_wait_ld();
          // (the staged Di is negated: dS = P * (dP + (-Di)) in two packed ops per pair)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 dv = d4[c];
            const float2 t0 = add2(make_float2(__uint_as_float(a[c * 4]), __uint_as_float(a[c * 4 + 1])),
                                   make_float2(dv.x, dv.y));
            const float2 t1 = add2(make_float2(__uint_as_float(a[c * 4 + 2]), __uint_as_float(a[c * 4 + 3])),
                                   make_float2(dv.z, dv.w));
            const float2 r0 = mul2(make_float2(pr[c * 4], pr[c * 4 + 1]), t0);
            const float2 r1 = mul2(make_float2(pr[c * 4 + 2], pr[c * 4 + 3]), t1);
            pr[c * 4] = r0.x;
            pr[c * 4 + 1] = r0.y;
            pr[c * 4 + 2] = r1.x;
            pr[c * 4 + 3] = r1.y;
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(pr[2 * c], pr[2 * c + 1]);
          tmem_st16(tmem + lane_off + COL_DP + ch * 32, pk);
          // dS^T into shared memory (MN-major operand of the dQ^T product).
          if (!mbar_wait(&bars.ds_free, dsfph ^ 1, ctl, 23)) goto done;
          dsfph ^= 1;
          uint8_t *row = smem + C::OFF_DS + r * 128;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(row + (((ch * 4 + j) ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          fence_async_smem();
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars.ds_ready);
          mbar_arrive(&bars.stage_empty[s]);  // done with this stage's LSE / Di
        }
      }
      // dK, dV epilogue for this tile's key rows (this warp's half of D).
      if (!mbar_wait(&bars.dkdv_full, dkdvph, ctl, 24)) goto done;
      dkdvph ^= 1;
      tc_fence_after();
      {
        const int64_t grow = (int64_t)(tl.kv_row0 + r) * p.H + tl.h;
        uint4 *dvp = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dv) + grow * D);
        uint4 *dkp = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dk) + grow * D);
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const float mul = which ? p.scale : 1.f;
          uint4 *dst = which ? dkp : dvp;
          // This warp's half of D: both 32-column chunks in flight at once.
          uint32_t v[D / 64][32];
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc)
            tmem_ld32(tmem + lane_off + (which ? COL_DK : COL_DV) + (ch * (D / 64) + cc) * 32, v[cc]);
          tmem_wait_ld();
          if constexpr (D == 128) {  // 64 columns = one 128-byte line per row: four lanes to a row
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              w[e] = pack_bf16_mul(v[0][2 * e], v[0][2 * e + 1], make_float2(mul, mul));
              w[16 + e] = pack_bf16_mul(v[1][2 * e], v[1][2 * e + 1], make_float2(mul, mul));
            }
            const int grp = wq * 32 + (lane & ~3);
            __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(which ? p.dk : p.dv);
            store_rows_by_quads(
                w, lane,
                [&](int k) {
                  return (void *)(outp + ((int64_t)(tl.kv_row0 + grp + k) * p.H + tl.h) * D + ch * 64);
                },
                [&](int k) { return grp + k < tl.nkv; });
          } else if (kv_ok) {
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                pk[e] = pack_bf16_mul(v[cc][2 * e], v[cc][2 * e + 1], make_float2(mul, mul));
              const int c = ch * (D / 64) + cc;
              st_global_v8(dst + c * 4, pk);
              st_global_v8(dst + c * 4 + 2, pk + 8);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.dkdv_free);
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------------------------- LSE / Di staging and dQ reduction
    // Per query block, ahead of the compute warps: LSE and Di = rowsum(dO * O)
    // of the block's 64 rows (two threads per row, O read from global memory
    // one block ahead into registers, dO from the stage). Then the dQ^T of
    // the block two before this one: drain it from its TMEM buffer, release
    // the buffer, and TMA reduce-add it.
    constexpr int ND = D / 2;  // head-dim elements per thread for Di
    constexpr int NV = ND / 8;
    const int wq = warp & 3;
    // Two threads per row, the row's halves eight lanes apart: the eight lanes
    // of a quarter-warp read eight different rows of the swizzled dO tile, so
    // their 16-byte chunks fall in eight different bank groups.
    const int row = wq * 16 + (lane & 7) + ((lane >> 4) << 3);
    const int half = (lane >> 3) & 1;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    float *stg = reinterpret_cast<float *>(smem + C::OFF_DQS + wq * 8192);
    const __nv_bfloat16 *obase = static_cast<const __nv_bfloat16 *>(p.o);
    uint32_t fph = 0, dqph = 0;
    int qb = 0;
    uint4 o_r[NV];
    float lse_r = INFINITY;
    bool row_ok = false;
    auto prefetch = [&](const BlockIter<BCAST, GEN> &it) {
      const int qrow = query_block<GEN>(p, it.tl, it.i) * 64 + row;
      row_ok = qrow < it.tl.Lq;
      if (row_ok) {
        lse_r = p.lse[it.tl.lse0 + qrow];
        const uint4 *src = reinterpret_cast<const uint4 *>(
            obase + ((int64_t)(it.tl.o_row0 + qrow) * p.H + it.tl.h) * D + half * ND);
#pragma unroll
        for (int j = 0; j < NV; ++j) o_r[j] = __ldg(src + j);
      }
    };
    // One pending dQ reduction: head, first query row in the accumulator (rows
    // past the sequence carry zeros: P = 0 there).
    struct DqJob {
      int h, row0;
      int prow;  // deterministic: partial row of the block's first query row
    };
    auto reduce_dq = [&](const DqJob &jb, int qbr) -> bool {
      const int qbuf = qbr & 1;
      if (!mbar_wait(&bars.dq_full[qbuf], bit(dqph, qbuf), ctl, 30)) return false;
      dqph ^= 1u << qbuf;
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(tmem + lane_off + COL_DQ + qbuf * 64, v[0]);
      tmem_ld32(tmem + lane_off + COL_DQ + qbuf * 64 + 32, v[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.dq_free[qbuf]);  // TMEM released before the reduction
      if (wq * 32 >= D) return true;               // D = 64: lanes 64..127 are padding
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      if constexpr (BCAST) {  // the caller's fp32 dQ is the accumulator: scale each partial
        const float2 sc2 = make_float2(p.scale, p.scale);
#pragma unroll
        for (int qc = 0; qc < 2; ++qc)
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 x = mul2(make_float2(__uint_as_float(v[qc][j]), __uint_as_float(v[qc][j + 1])), sc2);
            stg[(qc * 32 + j) * 32 + lane] = x.x;
            stg[(qc * 32 + j + 1) * 32 + lane] = x.y;
          }
      } else {  // jagged: the cast to bf16 applies the scale once, to the sum
#pragma unroll
        for (int qc = 0; qc < 2; ++qc)
#pragma unroll
          for (int j = 0; j < 32; ++j) stg[(qc * 32 + j) * 32 + lane] = __uint_as_float(v[qc][j]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (GEN && p.det)  // deterministic: this key block's own partial, summed in order later
          tma_store_3d(&p.tm_dqpart, stg, wq * 32, jb.h, jb.prow);
        else
          tma_reduce_add_3d(&p.tm_dqacc, stg, wq * 32, jb.h, jb.row0);
        bulk_commit();
      }
      return true;
    };
    BlockIter<BCAST, GEN> cur;
    cur.t = tbeg;
    cur.tend = tend;
    cur.i = 0;
    cur.seek(p);
    if (cur.valid) prefetch(cur);
    // Two blocks in flight between LSE/Di staging and the dQ reduction, so the
    // staging of block n runs ahead of the reduction of block n - 2.
    bool have0 = false, have1 = false;
    DqJob job0{0, 0, 0}, job1{0, 0, 0};
    while (cur.valid) {
      const int s = qb % C::NSTAGE;
      if (!mbar_wait(&bars.stage_full[s], bit(fph, s), ctl, 31)) goto done;
      fph ^= 1u << s;
      {
        float2 di2 = make_float2(0.f, 0.f);
        if (row_ok) {
          const uint8_t *drow = smem + C::OFF_STAGE + s * 2 * C::QT + C::QT +
                                ((half * ND) / 64) * C::QCHUNK + row * 128;
          const int j0 = ((half * ND) % 64) / 8;
#pragma unroll
          for (int j = 0; j < NV; ++j) {
            const uint4 dv = *reinterpret_cast<const uint4 *>(drow + (((j0 + j) ^ (row & 7)) << 4));
            di2 = fma_bf16x2_f32(o_r[j].x, dv.x, di2);
            di2 = fma_bf16x2_f32(o_r[j].y, dv.y, di2);
            di2 = fma_bf16x2_f32(o_r[j].z, dv.z, di2);
            di2 = fma_bf16x2_f32(o_r[j].w, dv.w, di2);
          }
        }
        float di = di2.x + di2.y;
        di += __shfl_xor_sync(0xffffffffu, di, 8);
        if (half == 0) {  // negated; a row that saw no key (LSE = -inf) gets P = 0
          lse_s[s * 64 + row] = row_ok && lse_r > -INFINITY ? -lse_r * 1.4426950408889634f : -INFINITY;
          di_s[s * 64 + row] = row_ok ? -di : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.aux_full[s]);
      DqJob jnew;  // this block's reduction, run two blocks from now
      {
        const int qr = query_block<GEN>(p, cur.tl, cur.i) * 64;
        jnew = DqJob{cur.tl.h, cur.tl.q_row0 + qr, cur.tl.prow0 + qr};
      }
      cur.next(p);  // advanced in place (one tile's state live, not two)
      if (cur.valid) prefetch(cur);
      if (have0 && !reduce_dq(job0, qb - 2)) goto done;
      job0 = job1;
      have0 = have1;
      job1 = jnew;
      have1 = true;
      ++qb;
    }
    if (have0 && !reduce_dq(job0, qb - 2)) goto done;
    if (have1 && !reduce_dq(job1, qb - 1)) goto done;
    if (lane == 0) bulk_wait<0>();
  }
done:
  if (warp == 1 && lane == 0 && bars.abort_flag) {
    mma_commit(&bars.drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars.drain, 0) && globaltimer() - t0 < p.timeout_ns) {
    }
  }
  if (warp >= 8 && warp < 12 && lane == 0) bulk_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BCAST, bool GEN>
cudaError_t launch_t(const BwdParams &p, int num_sms, cudaStream_t st) {
  auto kern = jfa_bwd_kernel<D, BCAST, GEN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, 512, BwdCfg<D>::SMEM, st>>>(p);
  return cudaGetLastError();
}

// Clearing of the fp32 accumulator, skipped when a forward pass with this
// workspace has already zeroed at least n16 units.
__global__ void acc_clear_kernel(float *acc, int64_t n16, const uint32_t *status) {
  const uint64_t zeroed =
      *reinterpret_cast<const volatile uint64_t *>(reinterpret_cast<const uint8_t *>(status) + kAccZeroedOff);
  if (zeroed >= (uint64_t)n16 * 16) return;
  uint4 *base = reinterpret_cast<uint4 *>(acc);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    base[i] = make_uint4(0, 0, 0, 0);
}

// scale * fp32 [rows, H, D] -> bf16 [rows, H, D]; 8 elements per thread.
__global__ void dq_convert_kernel(const float4 *__restrict__ acc, uint4 *__restrict__ dq, int64_t n8,
                                  float scale, uint32_t *status) {
  if (blockIdx.x == 0 && threadIdx.x == 0)  // the accumulator is dirty until cleared again
    *reinterpret_cast<volatile uint64_t *>(reinterpret_cast<uint8_t *>(status) + kAccZeroedOff) = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    dq[i] = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                       pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
  }
}

// Positions (row - first row of its sequence) of rows [r0, r0 + n) into
// pos[] in shared memory: thread 0 finds the first row's sequence by binary
// search of the offsets and walks forward (offsets clamped to [0, T]).
constexpr int kRopeChunk = 32;  // rows per block step of the rotary row kernels

__device__ __forceinline__ void chunk_positions(const void *off, int idx64, int64_t B, int64_t T,
                                                int64_t r0, int n, int *pos) {
  if (threadIdx.x == 0) {
    auto at = [&](int64_t b) { return min(max(load_off(off, idx64, (int)b), (int64_t)0), T); };
    int64_t lo = 0, hi = B;  // the last b with offsets[b] <= r0
    while (hi - lo > 1) {
      const int64_t mid = (lo + hi) >> 1;
      if (at(mid) <= r0) lo = mid; else hi = mid;
    }
    int64_t b = lo, s = at(b), e = at(b + 1);
    for (int i = 0; i < n; ++i) {
      const int64_t r = r0 + i;
      while (e <= r && b + 1 < B) {
        ++b;
        s = e;
        e = at(b + 1);
      }
      pos[i] = (int)(r - s);
    }
  }
  __syncthreads();
}

// As dq_convert_kernel, and each row's dQ rotated back (the transposed
// rotation) at the row's position in its sequence; the same row of dK (bf16,
// written by the backward kernel with respect to the rotated k) is rotated
// back in place in the same pass. Item = 4 pairs (i, i + D/2) of one (row,
// head).
template <int D>
__global__ void __launch_bounds__(256) dq_convert_rope_kernel(
    const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, __nv_bfloat16 *__restrict__ dk,
    int64_t rows, int H, float scale, const void *offsets, int idx64, int64_t B, int64_t T,
    const float *cos_t, const float *sin_t, int64_t rope_L, uint32_t *status) {
  __shared__ int pos_s[kRopeChunk];
  if (blockIdx.x == 0 && threadIdx.x == 0)
    *reinterpret_cast<volatile uint64_t *>(reinterpret_cast<uint8_t *>(status) + kAccZeroedOff) = 0;
  constexpr int NQ = D / 8;  // 4-pair groups per (row, head)
  const int per_row = H * NQ;
  for (int64_t r0 = (int64_t)blockIdx.x * kRopeChunk; r0 < rows; r0 += (int64_t)gridDim.x * kRopeChunk) {
    const int n = (int)min((int64_t)kRopeChunk, rows - r0);
    chunk_positions(offsets, idx64, B, T, r0, n, pos_s);
    for (int it = threadIdx.x; it < n * per_row; it += blockDim.x) {
      const int rr = it / per_row, g = it % NQ;
      const int64_t rh = (r0 + rr) * H + (it % per_row) / NQ;
      const int64_t pos = min(max((int64_t)pos_s[rr], (int64_t)0), rope_L - 1);
      const float4 cf = __ldg(reinterpret_cast<const float4 *>(cos_t + pos * (D / 2)) + g);
      const float4 sf = __ldg(reinterpret_cast<const float4 *>(sin_t + pos * (D / 2)) + g);
      const float4 a = *reinterpret_cast<const float4 *>(acc + rh * D + 4 * g);
      const float4 b = *reinterpret_cast<const float4 *>(acc + rh * D + D / 2 + 4 * g);
      const float l0 = (a.x * cf.x + b.x * sf.x) * scale, l1 = (a.y * cf.y + b.y * sf.y) * scale;
      const float l2 = (a.z * cf.z + b.z * sf.z) * scale, l3 = (a.w * cf.w + b.w * sf.w) * scale;
      const float h0 = (b.x * cf.x - a.x * sf.x) * scale, h1 = (b.y * cf.y - a.y * sf.y) * scale;
      const float h2 = (b.z * cf.z - a.z * sf.z) * scale, h3 = (b.w * cf.w - a.w * sf.w) * scale;
      *reinterpret_cast<uint2 *>(dq + rh * D + 4 * g) = make_uint2(pack_bf16(l0, l1), pack_bf16(l2, l3));
      *reinterpret_cast<uint2 *>(dq + rh * D + D / 2 + 4 * g) =
          make_uint2(pack_bf16(h0, h1), pack_bf16(h2, h3));
      uint2 *kl = reinterpret_cast<uint2 *>(dk + rh * D + 4 * g);
      uint2 *kh = reinterpret_cast<uint2 *>(dk + rh * D + D / 2 + 4 * g);
      const uint2 ka = *kl, kb = *kh;
      const float2 a01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ka.x));
      const float2 a23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ka.y));
      const float2 b01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kb.x));
      const float2 b23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kb.y));
      *kl = make_uint2(pack_bf16(a01.x * cf.x + b01.x * sf.x, a01.y * cf.y + b01.y * sf.y),
                       pack_bf16(a23.x * cf.z + b23.x * sf.z, a23.y * cf.w + b23.y * sf.w));
      *kh = make_uint2(pack_bf16(b01.x * cf.x - a01.x * sf.x, b01.y * cf.y - a01.y * sf.y),
                       pack_bf16(b23.x * cf.z - a23.x * sf.z, b23.y * cf.w - a23.y * sf.w));
    }
    __syncthreads();  // pos_s is rewritten for the next chunk
  }
}

// x_rot = x rotated at each row's position in its sequence (rotary "rotate
// half"): item = 8 pairs (i, i + D/2) of one (row, head), in fp32, rounded
// to bf16.
template <int D>
__global__ void __launch_bounds__(256) rope_rows_kernel(
    const __nv_bfloat16 *__restrict__ x, __nv_bfloat16 *__restrict__ y, int64_t rows, int H,
    const void *offsets, int idx64, int64_t B, int64_t T, const float *cos_t, const float *sin_t,
    int64_t rope_L, int64_t dense_L) {
  __shared__ int pos_s[kRopeChunk];
  constexpr int NQ = D / 16;  // 8-pair groups per (row, head)
  const int per_row = H * NQ;
  for (int64_t r0 = (int64_t)blockIdx.x * kRopeChunk; r0 < rows; r0 += (int64_t)gridDim.x * kRopeChunk) {
    const int n = (int)min((int64_t)kRopeChunk, rows - r0);
    if (dense_L > 0) {  // dense sequences of dense_L rows: position = row mod dense_L
      if (threadIdx.x < n) pos_s[threadIdx.x] = (int)((r0 + threadIdx.x) % dense_L);
      __syncthreads();
    } else {
      chunk_positions(offsets, idx64, B, T, r0, n, pos_s);
    }
    for (int it = threadIdx.x; it < n * per_row; it += blockDim.x) {
      const int rr = it / per_row, g = it % NQ;
      const int64_t rh = (r0 + rr) * H + (it % per_row) / NQ;
      const int64_t pos = min(max((int64_t)pos_s[rr], (int64_t)0), rope_L - 1);
      const float4 *cp = reinterpret_cast<const float4 *>(cos_t + pos * (D / 2) + 8 * g);
      const float4 *sp = reinterpret_cast<const float4 *>(sin_t + pos * (D / 2) + 8 * g);
      const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0v = __ldg(sp), s1v = __ldg(sp + 1);
      const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float sn[8] = {s0v.x, s0v.y, s0v.z, s0v.w, s1v.x, s1v.y, s1v.z, s1v.w};
      const uint4 a = *reinterpret_cast<const uint4 *>(x + rh * D + 8 * g);
      const uint4 b = *reinterpret_cast<const uint4 *>(x + rh * D + D / 2 + 8 * g);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      uint32_t ow[4], hw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xl = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&aw[e]));
        const float2 xh = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bw[e]));
        ow[e] = pack_bf16(xl.x * c[2 * e] - xh.x * sn[2 * e], xl.y * c[2 * e + 1] - xh.y * sn[2 * e + 1]);
        hw[e] = pack_bf16(xh.x * c[2 * e] + xl.x * sn[2 * e], xh.y * c[2 * e + 1] + xl.y * sn[2 * e + 1]);
      }
      *reinterpret_cast<uint4 *>(y + rh * D + 8 * g) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      *reinterpret_cast<uint4 *>(y + rh * D + D / 2 + 8 * g) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    __syncthreads();  // pos_s is rewritten for the next chunk
  }
}

// Sequence bounds exactly as decode_tile reads them (clamped to the tensors).
__device__ __forceinline__ void seq_bounds(const BwdParams &p, int64_t b, int64_t *qs, int64_t *Lq,
                                           int64_t *Lk) {
  const int64_t s0 = min(max(load_off(p.offsets, p.idx64, (int)b), (int64_t)0), p.T);
  const int64_t e0 = min(max(load_off(p.offsets, p.idx64, (int)b + 1), s0), p.T);
  *qs = min(max(load_off(p.q_offsets, p.idx64, (int)b), (int64_t)0), p.Tq);
  *Lq = min(max(load_off(p.q_offsets, p.idx64, (int)b + 1), *qs), p.Tq) - *qs;
  *Lk = e0 - s0;
}

// First partial row of key block n of sequence b (deterministic dQ).
__device__ __forceinline__ int64_t det_base_row(const BwdParams &p, int64_t b, int n,
                                                int64_t lqpad) {
  return p.det_base[b] + (int64_t)n * lqpad;
}

// Deterministic dQ layout (one CTA of 1024 threads): per sequence, the
// partial rows (ceil(Lk / 128) key blocks x Lq rounded up to 64) and the
// 64-row query blocks, as exclusive prefix sums over the batch.
__global__ void __launch_bounds__(1024) det_layout_kernel(const BwdParams p, int64_t *det_base,
                                                          int64_t *qb_base) {
  __shared__ int64_t s_rows[1024], s_qb[1024];
  const int t = threadIdx.x;
  const int64_t chunk = (p.B + 1023) / 1024;
  const int64_t b0 = min(p.B, (int64_t)t * chunk), b1 = min(p.B, b0 + chunk);
  int64_t rows = 0, qbs = 0;
  for (int64_t b = b0; b < b1; ++b) {
    int64_t qs, Lq, Lk;
    seq_bounds(p, b, &qs, &Lq, &Lk);
    rows += (Lk + 127) / 128 * ((Lq + 63) / 64 * 64);
    qbs += (Lq + 63) / 64;
  }
  s_rows[t] = rows;
  s_qb[t] = qbs;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan
    const int64_t a = t >= off ? s_rows[t - off] : 0, q = t >= off ? s_qb[t - off] : 0;
    __syncthreads();
    s_rows[t] += a;
    s_qb[t] += q;
    __syncthreads();
  }
  int64_t br = s_rows[t] - rows, bq = s_qb[t] - qbs;
  for (int64_t b = b0; b < b1; ++b) {
    int64_t qs, Lq, Lk;
    seq_bounds(p, b, &qs, &Lq, &Lk);
    det_base[b] = br;
    qb_base[b] = bq;
    br += (Lk + 127) / 128 * ((Lq + 63) / 64 * 64);
    bq += (Lq + 63) / 64;
  }
  if (t == 1023) {
    det_base[p.B] = s_rows[1023];
    qb_base[p.B] = s_qb[1023];
    if (s_rows[1023] > p.det_rows) atomicCAS(p.status, 0u, 3u);  // JFA_ERR_WORKSPACE
  }
}

// Deterministic dQ: one 64-row query block per iteration of the grid-stride
// loop; its rows sum, in key-block order, the partials of the key blocks that
// walked that query block (a contiguous range of key blocks, since the band's
// query range grows with the key block), scale, and store bf16.
template <int D>
__global__ void __launch_bounds__(256, 4) det_cast_kernel(const BwdParams p, const float *part,
                                                       const int64_t *qb_base, __nv_bfloat16 *dq) {
  __shared__ int s_na, s_nb;
  __shared__ int64_t s_b;
  const int64_t total = qb_base[p.B];
  const int HD8 = p.H * D / 8;
  for (int64_t g = blockIdx.x; g < total; g += gridDim.x) {
    if (threadIdx.x == 0) {  // the sequence of block g: the last b with qb_base[b] <= g
      int64_t lo = 0, hi = p.B;
      while (hi - lo > 1) {
        const int64_t mid = (lo + hi) / 2;
        if (qb_base[mid] <= g) lo = mid; else hi = mid;
      }
      s_b = lo;
      s_na = 1 << 30;
      s_nb = -1;
    }
    __syncthreads();
    const int64_t b = s_b;
    const int qb = (int)(g - qb_base[b]);
    int64_t qs, Lq, Lk;
    seq_bounds(p, b, &qs, &Lq, &Lk);
    const int nkt = (int)((Lk + 127) / 128);
    for (int n = threadIdx.x; n < nkt; n += blockDim.x) {
      int qb0, nq;
      bwd_query_blocks(n, Lq, Lk, p.win_left, p.win_right, &qb0, &nq);
      if (qb >= qb0 && qb < qb0 + nq) {
        atomicMin(&s_na, n);
        atomicMax(&s_nb, n);
      }
    }
    __syncthreads();
    const int na = s_na, nb = s_nb;
    const int64_t lqpad = (Lq + 63) / 64 * 64;
    const int rows = (int)min((int64_t)64, Lq - (int64_t)qb * 64);
    for (int e = threadIdx.x; e < rows * HD8; e += blockDim.x) {
      const int row = e / HD8, rem = e - row * HD8;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int n = na; n <= nb; ++n) {
        const int64_t prow = det_base_row(p, b, n, lqpad) + (int64_t)qb * 64 + row;
        if (prow >= p.det_rows) continue;  // (only with a workspace too small: reported)
        const float4 *src = reinterpret_cast<const float4 *>(part + prow * p.H * D) + rem * 2;
        const float4 x = src[0], y = src[1];
        acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
        acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
      }
      const float sc = p.scale;
      reinterpret_cast<uint4 *>(dq + (qs + (int64_t)qb * 64 + row) * p.H * D)[rem] =
          make_uint4(pack_bf16(acc[0] * sc, acc[1] * sc), pack_bf16(acc[2] * sc, acc[3] * sc),
                     pack_bf16(acc[4] * sc, acc[5] * sc), pack_bf16(acc[6] * sc, acc[7] * sc));
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_det_layout(const BwdParams &p, int64_t *det_base, int64_t *qb_base,
                              cudaStream_t st) {
  det_layout_kernel<<<1, 1024, 0, st>>>(p, det_base, qb_base);
  return cudaGetLastError();
}

cudaError_t launch_det_cast(const BwdParams &p, const float *part, const int64_t *qb_base,
                            void *dq, int D, int num_sms, cudaStream_t st) {
  auto *out = static_cast<__nv_bfloat16 *>(dq);
  if (D == 128)
    det_cast_kernel<128><<<num_sms * 8, 256, 0, st>>>(p, part, qb_base, out);
  else
    det_cast_kernel<64><<<num_sms * 8, 256, 0, st>>>(p, part, qb_base, out);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdParams &p, int D, int num_sms, cudaStream_t st) {
  const bool bcast = p.Lq > 0;
  const bool gen = !bcast && (p.win_left >= 0 || p.win_right >= 0 || p.det || p.blk_ptr != nullptr);
  if (D == 128) {
    if (bcast) return launch_t<128, true, false>(p, num_sms, st);
    return gen ? launch_t<128, false, true>(p, num_sms, st) : launch_t<128, false, false>(p, num_sms, st);
  }
  if (bcast) return launch_t<64, true, false>(p, num_sms, st);
  return gen ? launch_t<64, false, true>(p, num_sms, st) : launch_t<64, false, false>(p, num_sms, st);
}

static int grid_for(int64_t n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + 255) / 256;
  return (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
}

cudaError_t launch_acc_clear(float *acc, int64_t n16, const uint32_t *status, cudaStream_t st) {
  if (n16 == 0) return cudaSuccess;
  acc_clear_kernel<<<grid_for(n16), 256, 0, st>>>(acc, n16, status);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert_rope(const BwdParams &p, const float *acc, void *dq, int64_t rows,
                                   int D, cudaStream_t st) {
  auto *dkp = static_cast<__nv_bfloat16 *>(p.dk);
  const int64_t n = (rows + kRopeChunk - 1) / kRopeChunk * 256;  // one 256-thread block per chunk
  auto *out = static_cast<__nv_bfloat16 *>(dq);
  if (D == 128)
    dq_convert_rope_kernel<128><<<grid_for(n), 256, 0, st>>>(acc, out, dkp, rows, p.H, p.scale, p.offsets,
                                                             p.idx64, p.B, p.T, p.cos_t, p.sin_t,
                                                             p.rope_L, p.status);
  else
    dq_convert_rope_kernel<64><<<grid_for(n), 256, 0, st>>>(acc, out, dkp, rows, p.H, p.scale, p.offsets,
                                                            p.idx64, p.B, p.T, p.cos_t, p.sin_t,
                                                            p.rope_L, p.status);
  return cudaGetLastError();
}

cudaError_t launch_rope_rows(const void *x, void *y, int64_t rows, int H, int D, const void *offsets,
                             int idx64, int64_t B, const float *cos_t, const float *sin_t,
                             int64_t rope_L, int64_t dense_L, cudaStream_t st) {
  const int64_t n = (rows + kRopeChunk - 1) / kRopeChunk * 256;  // one 256-thread block per chunk
  const auto *xi = static_cast<const __nv_bfloat16 *>(x);
  auto *yo = static_cast<__nv_bfloat16 *>(y);
  if (D == 128)
    rope_rows_kernel<128><<<grid_for(n), 256, 0, st>>>(xi, yo, rows, H, offsets, idx64, B, rows,
                                                       cos_t, sin_t, rope_L, dense_L);
  else
    rope_rows_kernel<64><<<grid_for(n), 256, 0, st>>>(xi, yo, rows, H, offsets, idx64, B, rows,
                                                      cos_t, sin_t, rope_L, dense_L);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float *acc, void *dq, int64_t rows, int H, int D, float scale,
                              uint32_t *status, cudaStream_t st) {
  const int64_t n8 = rows * H * D / 8;
  dq_convert_kernel<<<grid_for(n8), 256, 0, st>>>(reinterpret_cast<const float4 *>(acc),
                                                  static_cast<uint4 *>(dq), n8, scale, status);
  return cudaGetLastError();
}

}  // namespace jfa
