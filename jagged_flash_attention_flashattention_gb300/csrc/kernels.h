// kernels.h -- parameter blocks and launchers of the device kernels
// (internal to libjfa; the public interface is include/jfa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace jfa {

// Forward kernel (jagged and broadcast-Q). Tiles are 256 query rows: two
// 128-row halves A and B that share every K/V tile.
struct FwdParams {
  CUtensorMap tm_q;  // bf16 [rows, H, D] viewed as {D, H, rows}, box {64, 1, 128}, 128B swizzle
  CUtensorMap tm_k;  // bf16 [Tk, H, D], same box
  CUtensorMap tm_v;
  CUtensorMap tm_khalf;   // CTA-pair forward: K viewed with 64-row boxes (one pair half of a K tile)
  const void *offsets;    // device [B+1]: K/V sequence bounds
  const void *q_offsets;  // device [B+1]: query sequence bounds (jagged; may equal offsets)
  int idx64;              // offsets are int64
  const int32_t *sm_ptr;
  const int32_t *tiles;
  void *o;      // bf16
  float *lse;   // fp32
  int64_t B;    // sequences: tiles naming b >= B are skipped
  int64_t T;    // packed K/V length; K/V bounds read from the offsets are clamped to [0, T]
  int64_t Tq;   // packed query length (jagged: LSE row stride; query bounds clamped to it)
  int win_left, win_right;  // band mask (band.h); -1 = unbounded
  int H;
  int Lq;       // broadcast-Q: dense query length; 0 for jagged self-attention
  float scale_log2;  // scale * log2(e)
  uint32_t *status;
  uint64_t timeout_ns;
  // Jagged only, when the workspace also holds the backward's fp32 dQ
  // accumulator: the two otherwise idle warps zero it (acc_n16 units of 16
  // bytes, split evenly over the CTAs) and block 0 records acc_n16 * 16 in the
  // status block, so the backward that follows skips its own clearing pass.
  float *acc_zero;
  int64_t acc_n16;
  // Dynamic tile scheduling (jagged, no band): dyn = 1 takes tiles from the
  // list `tiles` (n_tiles entries, in order), dyn = 2 from the device
  // enumeration tile_base[B+1] (tiles before sequence b, H * ceil(L_b / 256)
  // each, head-major within a sequence); CTAs claim the next tile with an
  // atomic add on *queue, which starts at zero.
  int dyn;
  int *queue;
  const int64_t *tile_base;
  int64_t n_tiles;
  // Block-sparse masks (masked / cross instantiation, no band): tile i of the
  // list walks the key blocks blk_list[blk_ptr[i] .. blk_ptr[i + 1]) (block |
  // half-0 bit << 29 | half-1 bit << 30); blk_meta[i] = first / end step of
  // each half. Null: no block mask.
  const int32_t *blk_ptr;
  const int32_t *blk_list;
  const int4 *blk_meta;
};

// Block-sparse list entries: key block in the low bits, one bit per query half.
constexpr uint32_t kBlkIndex = (1u << 29) - 1;
constexpr int kBlkSeesShift = 29;

// Byte offset, in the status block, of the uint64 count of accumulator bytes
// known to be zero (written by the forward kernel, reset by the dQ cast).
constexpr size_t kAccZeroedOff = 128;

cudaError_t launch_fwd(const FwdParams &p, int D, int num_sms, cudaStream_t st);

// CTA-pair forward (jagged self-attention, D = 128, no band): clusters of two
// CTAs, one per pair slot of the schedule (tiles of 512 query rows); grid =
// 2 * num_pairs.
cudaError_t launch_fwd_pair(const FwdParams &p, int num_pairs, cudaStream_t st);
// Clusters of two that can be resident at once (0 if the pair kernel cannot run).
int fwd_pair_max_clusters();

// Device enumeration of the forward tiles for dynamic scheduling: writes
// tile_base[0..B] from the device offsets (clamped like the kernels) and
// zeroes *queue. One CTA.
cudaError_t launch_fwd_enum(const FwdParams &p, int64_t *tile_base, int *queue, cudaStream_t st);

// Backward kernel (jagged and broadcast-Q). Tiles are 128 key rows; the
// kernel walks the sequence's query rows in blocks of 64.
struct BwdParams {
  CUtensorMap tm_q;   // bf16 query rows, box {64, 1, 64}
  CUtensorMap tm_do;  // bf16 dO rows (same row space as O), box {64, 1, 64}
  CUtensorMap tm_k;   // bf16 [Tk, H, D], box {64, 1, 128}
  CUtensorMap tm_v;
  CUtensorMap tm_dqacc;  // fp32 [rows, H, D] as {D, H, rows}, box {32, 1, 64}, no swizzle
  CUtensorMap tm_dqpart;  // deterministic dQ: fp32 partials [rows, H, D], box {32, 1, 64}
  const void *offsets;    // K/V sequence bounds
  const void *q_offsets;  // query sequence bounds (jagged; may equal offsets)
  int idx64;
  const int32_t *sm_ptr;
  const int32_t *tiles;
  const float *lse;
  const void *o;  // bf16 O rows (read directly for Di)
  void *dk;  // bf16 [Tk, H, D]
  void *dv;
  int64_t B;   // sequences: tiles naming b >= B are skipped
  int64_t T;   // packed K/V length; K/V bounds are clamped to [0, T]
  int64_t Tq;  // packed query length (jagged); query bounds are clamped to [0, Tq]
  int win_left, win_right;  // band mask (band.h); -1 = unbounded
  // Deterministic dQ: each key block stores its dQ partial of each query block
  // (no atomics) at row det_base[b] + n * round_up(Lq, 64) + 64 * qb of the
  // partial buffer (det_rows rows); a separate pass sums them in key-block order.
  int det;
  const int64_t *det_base;
  int64_t det_rows;
  int H;
  int Lq;  // broadcast-Q: dense query length; 0 for jagged
  float scale;
  float scale_log2;
  uint32_t *status;
  uint64_t timeout_ns;
  // Rotary (jagged self-attention, no band): fp32 tables [rope_L, D/2]; q and
  // k are the rotated rows, and the closing cast rotates dQ and dK back by the
  // transposed rotation at each row's position in its sequence. Null: no
  // rotary.
  const float *cos_t;
  const float *sin_t;
  int64_t rope_L;
  // Block-sparse masks (masked / cross instantiation, no band, no
  // deterministic dQ): tile i walks the 64-row query blocks
  // blk_list[blk_ptr[i] .. blk_ptr[i + 1]). Null: no block mask.
  const int32_t *blk_ptr;
  const int32_t *blk_list;
};

cudaError_t launch_bwd(const BwdParams &p, int D, int num_sms, cudaStream_t st);
// x_rot = x [rows, H, D] bf16 rotated at each row's position in its sequence
// (offsets [B+1], or, dense_L > 0, sequences of dense_L rows each and no
// offsets; positions clamped to [0, rope_L)).
cudaError_t launch_rope_rows(const void *x, void *y, int64_t rows, int H, int D, const void *offsets,
                             int idx64, int64_t B, const float *cos_t, const float *sin_t,
                             int64_t rope_L, int64_t dense_L, cudaStream_t st);
// The cast of launch_dq_convert with each row rotated back (p.cos_t, p.sin_t),
// and the same rows of dK (p.dk, bf16) rotated back in place.
cudaError_t launch_dq_convert_rope(const BwdParams &p, const float *acc, void *dq, int64_t rows,
                                   int D, cudaStream_t st);

// Zeroes the fp32 dQ accumulator (n16 units of 16 bytes) unless the status
// block already records at least that many zero bytes.
cudaError_t launch_acc_clear(float *acc, int64_t n16, const uint32_t *status, cudaStream_t st);

// scale * fp32 [rows, H, D] -> bf16 [rows, H, D] (the jagged accumulator
// holds unscaled dS K sums); also resets the status block's
// zero-accumulator count (the accumulator is dirty from here on).
cudaError_t launch_dq_convert(const float *acc, void *dq, int64_t rows, int H, int D, float scale,
                              uint32_t *status, cudaStream_t st);

// Deterministic dQ layout: det_base[b] (partial rows before sequence b,
// [B+1]) and qb_base[b] (64-row query blocks before sequence b, [B+1]) from
// the device offsets; if the partial rows exceed det_rows, status word 0 is
// set to JFA_ERR_WORKSPACE.
cudaError_t launch_det_layout(const BwdParams &p, int64_t *det_base, int64_t *qb_base,
                              cudaStream_t st);

// Deterministic dQ: dq[row] = bf16(scale * sum over the key blocks that walk
// the row's query block, in key-block order, of their partials).
cudaError_t launch_det_cast(const BwdParams &p, const float *part, const int64_t *qb_base,
                            void *dq, int D, int num_sms, cudaStream_t st);

// Block-diagonal kernels: [B, L, H, D], 64-token blocks, 128-row work units.
struct BlockdiagParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // {D, H, B*L}, box {64, 1, 128}
  void *o;   // forward output
  void *dq;  // backward outputs
  void *dk;
  void *dv;
  int64_t rows;  // B * L
  int64_t L;     // tokens per sequence (a row's position is row % L)
  // Rotary variant: fp32 tables [L, D/2]. The forward rotates q and k rows by
  // them before the products; the backward reads rotated q and k and rotates
  // dQ, dK back.
  const float *cos_t;
  const float *sin_t;
  int H;
  float scale;
  float scale_log2;
  uint32_t *status;
  uint64_t timeout_ns;
};

cudaError_t launch_blockdiag_fwd(const BlockdiagParams &p, int D, int num_sms, cudaStream_t st);
cudaError_t launch_blockdiag_bwd(const BlockdiagParams &p, int D, int num_sms, cudaStream_t st);
// (p.cos_t != nullptr selects the rotary variant of either kernel.)

}  // namespace jfa
