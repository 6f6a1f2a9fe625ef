/*
 * jfa.h -- C ABI of libjfa: Jagged Flash Attention for GB300 (sm_103a).
 *
 * Exact softmax attention, forward and backward, over packed bf16 Q/K/V
 * whose sequence boundaries are given by an offsets tensor, so that no
 * padding token is ever materialised ("Desarrollo de Jagged Flash Attention
 * para el modelo GEM", first section: FlashAttention applied directly to the
 * packed Q, K, V plus an offsets tensor). Two special cases are provided:
 * broadcast-Q (one dense Q shared by every jagged K/V sequence, dQ summed
 * over the batch; same article, "Optimización del proceso de Backward y dQ")
 * and fixed 64-token block-diagonal attention ("TLX Block Attention",
 * sections 1-2).
 *
 * Common conventions
 * ------------------
 * - Every pointer is owned by the caller. The library allocates and frees
 *   no memory. Device buffers must be device-resident (cudaMalloc, or a
 *   framework allocator) and 16-byte aligned; host buffers are plain host
 *   memory.
 * - Packed tensors are bf16, contiguous, laid out [T, H, D] (token, head,
 *   dim). D must be 64 or 128. H >= 1. T < 2^31.
 * - offsets: device array of B+1 integers (int32 or int64, chosen by
 *   jfa_index_t), offsets[0] = 0, non-decreasing, offsets[B] = T. The
 *   kernels read it on the device; the scheduler reads a host copy.
 * - scale: the softmax scale applied to Q K^T (normally 1/sqrt(D)).
 * - LSE (log-sum-exp of the scaled scores, natural log) is fp32.
 * - All calls that take a stream are asynchronous on that stream. Argument
 *   errors are detected on the host and returned before anything is
 *   launched. Launch failures return JFA_ERR_CUDA. A kernel whose bounded
 *   waits expire writes a code into the status word at the start of its
 *   workspace and exits; jfa_check_status() synchronises the stream and
 *   reports it as JFA_ERR_TIMEOUT.
 * - A more detailed message for the last error of the calling thread is
 *   available from jfa_last_error().
 * - Work tiles: the forward kernels take tiles of 256 query rows (two
 *   128-row halves sharing K/V), the backward kernels tiles of 128 key rows.
 *   The tile lists come from jfa_sched_build() with the tile_rows reported
 *   by jfa_tile_rows().
 */
#ifndef JFA_H_
#define JFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *jfa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1, /* bad pointer, size, layout or offsets */
  JFA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D not in {64,128}) */
  JFA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than jfa_workspace_size() */
  JFA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  JFA_ERR_TIMEOUT = 5      /* a kernel's bounded wait expired (see jfa_check_status) */
} jfa_status;

typedef enum { JFA_I32 = 0, JFA_I64 = 1 } jfa_index_t;

typedef enum {
  JFA_OP_FWD = 0,
  JFA_OP_BWD = 1,
  JFA_OP_BCASTQ_FWD = 2,
  JFA_OP_BCASTQ_BWD = 3,
  JFA_OP_BLOCKDIAG_FWD = 4,
  JFA_OP_BLOCKDIAG_BWD = 5,
  JFA_OP_FWD_PAIR = 6 /* jfa_fwd_pair: 512-row tiles, D = 128 */
} jfa_op;

/* Human-readable name of a status code (static string). */
const char *jfa_status_str(jfa_status s);

/* Detail message of the last non-OK status returned on this thread
 * (static thread-local buffer; empty string when none). */
const char *jfa_last_error(void);

/* ------------------------------------------------------------------------
 * Host tile scheduler.
 *
 * "Desarrollo de Jagged Flash Attention para el modelo GEM", section
 * "Optimizaciones específicas para el flujo de trabajo de GEM": tiles are
 * sorted on the host by their K/V workload, largest first, and dealt to the
 * SMs in a zigzag (boustrophedon) order: even passes fill SMs left to
 * right, odd passes right to left.
 *
 * A tile is (b, h, m): sequence b, head h, row block m of tile_rows rows.
 * Sequence b has ceil(rows_b / tile_rows) row blocks, with rows_b =
 * fixed_rows if fixed_rows > 0, else its length offsets[b+1]-offsets[b].
 * Its work is fixed_work if fixed_work > 0, else its length. The sort is
 * stable (ties keep the order b, h, m). Sorted position i goes to pass
 * p = i / num_sms and SM (i % num_sms) on even p, num_sms-1-(i % num_sms)
 * on odd p. With zigzag = 0 the unsorted tiles are dealt round-robin
 * (SM i % num_sms), the naive order kept for comparison.
 *
 * Output is CSR: sm_ptr[num_sms+1] (sm_ptr[0] = 0) and tiles[3*n_tiles]
 * holding (b, h, m) int32 triples, each SM's tiles in dealt order. Both
 * are host buffers owned by the caller.
 * ---------------------------------------------------------------------- */

/* Number of tiles jfa_sched_build() will emit. host_offsets: host array of
 * B+1 entries. Returns JFA_ERR_INVALID_ARG for bad offsets or sizes. */
jfa_status jfa_sched_size(int64_t B, int H, int tile_rows, const void *host_offsets,
                          jfa_index_t idx, int64_t fixed_rows, int64_t *n_tiles);

jfa_status jfa_sched_build(int64_t B, int H, int tile_rows, int num_sms,
                           const void *host_offsets, jfa_index_t idx, int64_t fixed_rows,
                           int64_t fixed_work, int zigzag, int32_t *sm_ptr, int32_t *tiles);

/* Scheduler for jfa_varlen_fwd / jfa_varlen_bwd (op = JFA_OP_FWD or
 * JFA_OP_BWD): separate query and key/value offsets (host arrays of B+1
 * entries; host_q_offsets NULL means the same as host_kv_offsets) and the
 * band mask (window_left, window_right) of jfa_varlen_fwd. Forward tiles
 * are 256 query rows of one (sequence, head); their work is the length of
 * the key range those rows can see. Backward tiles are 128 keys; their work
 * is the length of the query range that can see them. Tiles with no work
 * are still emitted (their rows get O = 0, or their keys dK = dV = 0). Sort,
 * tie order and deal are those of jfa_sched_build; without a window and with
 * equal offsets the output equals jfa_sched_build's for the same op. */
jfa_status jfa_sched_size_varlen(int64_t B, int H, jfa_op op, const void *host_q_offsets,
                                 const void *host_kv_offsets, jfa_index_t idx, int64_t *n_tiles);

jfa_status jfa_sched_build_varlen(int64_t B, int H, jfa_op op, int num_sms,
                                  const void *host_q_offsets, const void *host_kv_offsets,
                                  jfa_index_t idx, int window_left, int window_right, int zigzag,
                                  int32_t *sm_ptr, int32_t *tiles);

/* Scheduler for jfa_sparse_fwd / jfa_sparse_bwd: block-sparse attention
 * with separate query and key/value offsets. host_masks holds, for each
 * sequence b in order, a row-major [ceil(Lq_b / 128), ceil(Lk_b / 128)]
 * byte array (non-zero: the 128 queries of that block row see the 128 keys
 * of that block column), concatenated; n_mask = its total length, which must
 * equal the sum of those sizes (JFA_ERR_INVALID_ARG otherwise).
 *
 * Forward (op = JFA_OP_FWD): tiles of 256 query rows (query blocks 2m and
 * 2m + 1, the tile's two 128-row halves). Tile i walks list entries
 * list[list_ptr[i] .. list_ptr[i + 1]): the key blocks that either half sees,
 * in increasing order, each encoded as (key block) | (half 0 sees it) << 29
 * | (half 1 sees it) << 30; meta[4 i .. 4 i + 3] = first step and one past
 * the last step (indices into the tile's entries) that half 0, then half 1,
 * sees ((0, 0) for a half that sees none). Work (the sort key) = the keys in
 * the listed blocks.
 *
 * Backward (op = JFA_OP_BWD): tiles of one 128-key block; entries are the
 * 64-row query blocks whose 128-row block sees the key block, increasing;
 * work = the query rows in them; meta is not written (may be NULL).
 *
 * Sort, tie order and deal are those of jfa_sched_build; lists follow the
 * dealt order of `tiles`. Sizes: sm_ptr [num_sms + 1], tiles [3 n_tiles],
 * list_ptr [n_tiles + 1], list [n_entries], meta [4 n_tiles], all host
 * int32 buffers owned by the caller. */
jfa_status jfa_sched_size_sparse(int64_t B, int H, jfa_op op, const void *host_q_offsets,
                                 const void *host_kv_offsets, jfa_index_t idx,
                                 const uint8_t *host_masks, int64_t n_mask, int64_t *n_tiles,
                                 int64_t *n_entries);

jfa_status jfa_sched_build_sparse(int64_t B, int H, jfa_op op, int num_sms,
                                  const void *host_q_offsets, const void *host_kv_offsets,
                                  jfa_index_t idx, const uint8_t *host_masks, int64_t n_mask,
                                  int zigzag, int32_t *sm_ptr, int32_t *tiles, int32_t *list_ptr,
                                  int32_t *list, int32_t *meta);

/* Rows per tile that the kernels of `op` expect from the scheduler. */
jfa_status jfa_tile_rows(jfa_op op, int D, int *tile_rows);

/* Number of SMs of the current device (the persistent grid size). */
jfa_status jfa_num_sms(int *num_sms);

/* ------------------------------------------------------------------------
 * Workspace.
 *
 * Every kernel call takes a device workspace that starts with a 256-byte
 * status block. jfa_bwd also keeps an fp32 dQ accumulator there ([T, H, D])
 * that must start at zero. When jfa_fwd is given a workspace of at least
 * jfa_workspace_size(JFA_OP_BWD, T, H, D) bytes, its kernel clears that
 * accumulator on otherwise idle warps and records the cleared size in the
 * status block; jfa_bwd then skips its own clearing pass, and clears the
 * accumulator itself in every other case (no forward, a forward of a smaller
 * batch, a second backward). Calls that share a workspace must be ordered on
 * one stream. `n` is T for JFA_OP_FWD / JFA_OP_BWD and is ignored for the
 * other ops.
 * ---------------------------------------------------------------------- */
size_t jfa_workspace_size(jfa_op op, int64_t n, int H, int D);

/* Clears the status block (asynchronous on `stream`). */
jfa_status jfa_workspace_init(void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* Synchronises `stream`, reads the status block: JFA_OK, or
 * JFA_ERR_TIMEOUT if a kernel gave up waiting (the block is then cleared so
 * the workspace can be reused). */
jfa_status jfa_check_status(void *workspace, jfa_stream_t stream);

/* Diagnostic of the failure path above (no counterpart in the pages): one
 * thread waits, with the same bounded wait as every kernel, on an mbarrier
 * phase that nothing completes. After `timeout_ns` (1 us .. 1 s) it gives up,
 * writes JFA_ERR_TIMEOUT with wait site 99 into the workspace status block
 * and returns, so jfa_check_status() then reports JFA_ERR_TIMEOUT and clears
 * the block. Nothing faults and the context stays usable. Asynchronous on
 * `stream`; returns JFA_ERR_WORKSPACE for a missing or too-small workspace
 * (fewer than 256 bytes) and JFA_ERR_INVALID_ARG for a limit out of range. */
jfa_status jfa_selftest_wait_timeout(void *workspace, size_t ws_bytes, uint64_t timeout_ns,
                                     jfa_stream_t stream);

/* ------------------------------------------------------------------------
 * Jagged forward: for each sequence b and head h,
 *   O = softmax(scale * Q K^T) V,  LSE_i = ln sum_j exp(scale * q_i . k_j)
 * ("TLX Block Attention", section 2: the standard FlashAttention loop with
 * running max, correction factor and final normalisation, storing
 * L = m + log(l) for the backward pass).
 *
 * q, k, v: device bf16 [T, H, D]. offsets: device [B+1]. d_sm_ptr,
 * d_tiles: device copies of jfa_sched_build() output for
 * tile_rows = jfa_tile_rows(JFA_OP_FWD). num_sms: length of d_sm_ptr - 1
 * (the grid size). o: device bf16 [T, H, D]. lse: device fp32 [H, T].
 * workspace: >= jfa_workspace_size(JFA_OP_FWD, ...); a workspace sized for
 * JFA_OP_BWD also gets its dQ accumulator cleared for the backward (see
 * Workspace above).
 * ---------------------------------------------------------------------- */
jfa_status jfa_fwd(const void *q, const void *k, const void *v, const void *offsets,
                   jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                   const int32_t *d_sm_ptr, const int32_t *d_tiles, int num_sms, void *o,
                   float *lse, void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* Rotary embeddings for the jagged kernels ("TLX Block Attention", section 1:
 * rotary embeddings fused into the attention backward's epilogue; the same
 * "rotate half" reading as blockdiag_rotary_fwd, with each row's position
 * counted from the start of its sequence). cos_t, sin_t: device fp32
 * [rope_L, D/2]; a position past rope_L - 1 uses row rope_L - 1 (the binding
 * refuses sequences longer than rope_L).
 *
 * jfa_rope: x_rot[r] = x[r] rotated at position r - offsets[b] of its
 * sequence b (device bf16 [T, H, D]; x_rot may be x itself). The rotary
 * forward of the layer: jfa_fwd then runs on the rotated q and k.
 *
 * jfa_rotary_bwd: jfa_bwd given the rotated q_rot, k_rot (and v, o, lse,
 * dout as for jfa_bwd), whose dq, dk are the gradients with respect to the
 * unrotated q, k: the backward's closing cast (which reads the fp32 dQ
 * accumulator anyway) rotates dQ back (the transposed rotation) and, in the
 * same pass, the rows of dK. Jagged self-attention without a band; the
 * workspace, tiles and errors are those of jfa_bwd. */
jfa_status jfa_rope(const void *x, const void *offsets, jfa_index_t idx, int64_t B, int64_t T,
                    int H, int D, const float *cos_t, const float *sin_t, int64_t rope_L,
                    void *x_rot, jfa_stream_t stream);

jfa_status jfa_rotary_bwd(const void *q_rot, const void *k_rot, const void *v, const void *o,
                          const float *lse, const void *dout, const void *offsets,
                          jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                          const float *cos_t, const float *sin_t, int64_t rope_L,
                          const int32_t *d_sm_ptr, const int32_t *d_tiles, int num_sms, void *dq,
                          void *dk, void *dv, void *workspace, size_t ws_bytes,
                          jfa_stream_t stream);

/* Jagged forward on CTA pairs ("Desarrollo de Jagged Flash Attention para
 * el modelo GEM", "Optimización del proceso de Backward y dQ": the 2-CTA MMA
 * of FA4, to raise tensor-core utilisation). Same inputs, outputs and
 * workspace as jfa_fwd (including the clearing of the backward's dQ
 * accumulator), for jagged self-attention at D = 128 (other D:
 * JFA_ERR_UNSUPPORTED). Two CTAs of a cluster compute each product together
 * (M = 256 rows, each CTA loading half of every K and V tile); a tile is 512
 * query rows of one (sequence, head). Tiles: jfa_sched_build() with
 * tile_rows = jfa_tile_rows(JFA_OP_FWD_PAIR) = 512 and num_sms = num_pairs
 * (normally jfa_num_pairs()); the grid is 2 * num_pairs CTAs. */
jfa_status jfa_fwd_pair(const void *q, const void *k, const void *v, const void *offsets,
                        jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                        const int32_t *d_sm_ptr, const int32_t *d_tiles, int num_pairs, void *o,
                        float *lse, void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* Number of two-CTA clusters of jfa_fwd_pair that fit on the current device
 * at once (at most half its SMs). */
jfa_status jfa_num_pairs(int *num_pairs);

/* Jagged forward with device-side dynamic tile scheduling ("A TLX nagyobb
 * kontrollt ad a Triton fölött": Cluster Launch Control, i.e. running CTAs
 * taking work at run time, among the primitives the pages name; reading
 * used: persistent CTAs claim forward tiles one at a time from a global
 * atomic counter, instead of walking a fixed per-SM list). Same inputs and
 * outputs as jfa_fwd, without a band mask. d_tiles NULL: the tiles are
 * enumerated on the device from the device offsets (sequence by sequence,
 * head-major, 256 query rows each), so neither host offsets nor a host
 * schedule are needed; otherwise d_tiles holds n_tiles (b, h, m) int32
 * triples claimed in that order (e.g. jfa_sched_build with num_sms = 1,
 * which lists the tiles longest first: greedy LPT). num_ctas: persistent
 * CTAs (normally jfa_num_sms()). workspace >=
 * jfa_fwd_dynamic_workspace_size(B) bytes (the status block, the claim
 * counter and the device tile table); it is not the backward's workspace
 * and clears no dQ accumulator. */
jfa_status jfa_fwd_dynamic(const void *q, const void *k, const void *v, const void *offsets,
                           jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                           const int32_t *d_tiles, int64_t n_tiles, int num_ctas, void *o,
                           float *lse, void *workspace, size_t ws_bytes, jfa_stream_t stream);

size_t jfa_fwd_dynamic_workspace_size(int64_t B);

/* Jagged backward: given dO (device bf16 [T, H, D]) and the forward's O and
 * LSE, writes dQ, dK, dV (device bf16 [T, H, D]):
 *   P = exp(scale * Q K^T - LSE), dV = P^T dO, dP = dO V^T,
 *   Di = rowsum(dO * O) (computed inside the kernel, no separate pass),
 *   dS = P * (dP - Di), dQ = scale * dS K, dK = scale * dS^T Q
 * ("TLX Block Attention", sections 2 and 4; "Desarrollo de Jagged Flash
 * Attention ...", "Cambios estructurales ...": a warp dedicated to the dQ
 * reduction). Tiles: jfa_sched_build() with tile_rows =
 * jfa_tile_rows(JFA_OP_BWD) over key blocks. workspace >=
 * jfa_workspace_size(JFA_OP_BWD, T, H, D). */
jfa_status jfa_bwd(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dout, const void *offsets, jfa_index_t idx,
                   int64_t B, int64_t T, int H, int D, float scale, const int32_t *d_sm_ptr,
                   const int32_t *d_tiles, int num_sms, void *dq, void *dk, void *dv,
                   void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* ------------------------------------------------------------------------
 * Masked and cross (varlen) attention.
 *
 * "Desarrollo de Jagged Flash Attention para el modelo GEM", section
 * "Impacto en el desarrollo de modelos generativos": causal, sliding-window
 * and block-sparse masks as the extensions of the jagged kernels, built on
 * the masked last K/V block of "Optimización del proceso de Backward y dQ".
 * The pages give no formula; the band mask used is the usual one. In
 * sequence b (Lq = query rows, Lk = keys, shift = Lk - Lq) query i sees key
 * j iff
 *   (window_left  < 0 || j >= i + shift - window_left) &&
 *   (window_right < 0 || j <= i + shift + window_right),
 * so (-1, -1) is no mask, (-1, 0) causal, (w - 1, 0) a causal window of w
 * keys, with the diagonal aligned to the last query and the last key
 * (bottom-right). A query that sees no key gets O = 0, LSE = -inf and
 * contributes no gradient; keys that no query sees get dK = dV = 0.
 *
 * Queries and keys have separate offsets (jagged cross attention; pass the
 * same array twice for self-attention): q, o, dout, dq are [Tq, H, D] bf16
 * with q_offsets [B+1], k, v, dk, dv are [Tk, H, D] bf16 with kv_offsets
 * [B+1], LSE is fp32 [H, Tq]. Tiles: jfa_sched_build_varlen with the same
 * offsets and window.
 * ---------------------------------------------------------------------- */
jfa_status jfa_varlen_fwd(const void *q, const void *k, const void *v, const void *q_offsets,
                          const void *kv_offsets, jfa_index_t idx, int64_t B, int64_t Tq,
                          int64_t Tk, int H, int D, float scale, int window_left,
                          int window_right, const int32_t *d_sm_ptr, const int32_t *d_tiles,
                          int num_sms, void *o, float *lse, void *workspace, size_t ws_bytes,
                          jfa_stream_t stream);

/* Backward of jfa_varlen_fwd. deterministic = 0: dQ is summed in an fp32
 * accumulator by TMA reduce-adds from every key block, so the order of the
 * additions, and the last bits of dQ, can change from run to run (as in
 * jfa_bwd). deterministic = 1: every key block stores its own fp32 partial
 * of each query block it walks, and a closing pass sums a query block's
 * partials in key-block order, so dQ is bit-identical across runs (reading
 * of "Optimización del proceso de Backward y dQ": per-block fp32 partials and
 * an ordered final sum); it needs a larger workspace and one more pass over
 * the partials. workspace >= jfa_varlen_workspace_size(...) for the same
 * offsets and mode; a workspace too small for the device offsets is reported
 * by jfa_check_status as JFA_ERR_WORKSPACE (dQ is then wrong, and nothing is
 * written outside the workspace and the outputs). */
jfa_status jfa_varlen_bwd(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, const void *q_offsets,
                          const void *kv_offsets, jfa_index_t idx, int64_t B, int64_t Tq,
                          int64_t Tk, int H, int D, float scale, int window_left,
                          int window_right, int deterministic, const int32_t *d_sm_ptr,
                          const int32_t *d_tiles, int num_sms, void *dq, void *dk, void *dv,
                          void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* Workspace bytes of jfa_varlen_bwd (and enough for jfa_varlen_fwd) from
 * host copies of the offsets (host_q_offsets NULL = host_kv_offsets):
 * non-deterministic, the 256-byte status block and an fp32 [Tq, H, D] dQ
 * accumulator; deterministic, the status block, two [B+1] int64 tables and
 * sum over b of ceil(Lk_b / 128) * round_up(Lq_b, 64) fp32 partial rows of
 * H * D. The forward clears the accumulator when given a non-deterministic
 * workspace of this size, as jfa_fwd does. */
jfa_status jfa_varlen_workspace_size(int64_t B, const void *host_q_offsets,
                                     const void *host_kv_offsets, jfa_index_t idx, int H, int D,
                                     int deterministic, size_t *bytes);

/* ------------------------------------------------------------------------
 * Block-sparse attention.
 *
 * The third mask family that "Desarrollo de Jagged Flash Attention para el
 * modelo GEM", section "Impacto en el desarrollo de modelos generativos",
 * names for the jagged kernels. The pages give no mask format; the reading
 * used: one mask of 128 x 128 blocks per sequence, blocks counted from the
 * first query and the first key of the sequence, so query i sees key j iff
 * mask_b[i / 128][j / 128] != 0 (the last block row and column cover the
 * ragged tails). A query that sees no key gets O = 0, LSE = -inf and
 * contributes no gradient; keys that no query sees get dK = dV = 0.
 *
 * Layouts as for jfa_varlen_fwd / jfa_varlen_bwd (q, o, dout, dq [Tq, H, D],
 * k, v, dk, dv [Tk, H, D] bf16, LSE fp32 [H, Tq], q_offsets and kv_offsets
 * [B+1]). The mask enters only through the schedule: d_sm_ptr, d_tiles,
 * d_list_ptr, d_list (and, forward, d_meta) are device copies of
 * jfa_sched_build_sparse's output for the same offsets, masks and op. The
 * kernels clamp every listed block to its sequence: a list of another batch
 * gives wrong numbers but touches no memory outside the tensors. The
 * backward sums dQ in the fp32 accumulator of jfa_varlen_bwd's
 * non-deterministic workspace (jfa_varlen_workspace_size with
 * deterministic = 0); there is no deterministic mode here.
 * ---------------------------------------------------------------------- */
jfa_status jfa_sparse_fwd(const void *q, const void *k, const void *v, const void *q_offsets,
                          const void *kv_offsets, jfa_index_t idx, int64_t B, int64_t Tq,
                          int64_t Tk, int H, int D, float scale, const int32_t *d_sm_ptr,
                          const int32_t *d_tiles, const int32_t *d_list_ptr,
                          const int32_t *d_list, const int32_t *d_meta, int num_sms, void *o,
                          float *lse, void *workspace, size_t ws_bytes, jfa_stream_t stream);

jfa_status jfa_sparse_bwd(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, const void *q_offsets,
                          const void *kv_offsets, jfa_index_t idx, int64_t B, int64_t Tq,
                          int64_t Tk, int H, int D, float scale, const int32_t *d_sm_ptr,
                          const int32_t *d_tiles, const int32_t *d_list_ptr,
                          const int32_t *d_list, int num_sms, void *dq, void *dk, void *dv,
                          void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* jfa_bwd without a workspace argument. The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory when
 * they call, such as a plug-in inside a framework that owns all device memory
 * through its own pool, or a latency-critical path that may not call
 * cudaMalloc (which can synchronise the device). Inputs and outputs are as
 * for jfa_bwd and are still the caller's; the scratch jfa_bwd would keep in
 * its workspace (a 256-byte status block and an fp32 [T, H, D] dQ
 * accumulator) lives instead in one static device array of 64 MiB per
 * device, which stays allocated until the process exits on every device
 * that has loaded it. Limit: T * H * D <= 16,777,152; larger problems return
 * JFA_ERR_WORKSPACE with a message and launch nothing. The library
 * allocates and frees nothing here. Each call looks up the array's device
 * address with the calling thread's current device (a host-side query, so a
 * cudaDeviceReset, which reloads the array, is handled); the first call on a
 * device may also load the module that holds the array, so make that first
 * call before any stream capture. Every call on a device shares the one array
 * (each call clears what must start at zero), so calls whose work overlaps
 * on the GPU, e.g. on two streams, race and give wrong results: serialise
 * them. A kernel timeout is recorded in the array's status block and stays
 * there, through later calls, until jfa_noalloc_check_status() reads it. */
jfa_status jfa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dout, const void *offsets,
                           jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                           const int32_t *d_sm_ptr, const int32_t *d_tiles, int num_sms,
                           void *dq, void *dk, void *dv, jfa_stream_t stream);

/* Status of jfa_bwd_noalloc on the current device (no counterpart in the
 * paper either): synchronises `stream`, reads the static array's status
 * block and returns JFA_ERR_TIMEOUT, clearing the block, if a kernel of any
 * jfa_bwd_noalloc call since the last check gave up waiting; JFA_OK
 * otherwise. Allocates nothing. */
jfa_status jfa_noalloc_check_status(jfa_stream_t stream);

/* Broadcast-Q forward: q device bf16 [Lq, H, D] is shared by every
 * sequence of k, v (device bf16 [Tk, H, D], boundaries kv_offsets [B+1]).
 * o: device bf16 [B, Lq, H, D]; lse: device fp32 [B, H, Lq]. A sequence of
 * length 0 gets O = 0 and LSE = -inf. Tiles: jfa_sched_build() with
 * tile_rows = jfa_tile_rows(JFA_OP_BCASTQ_FWD), fixed_rows = Lq.
 * B * Lq must stay below 2^31 - 256 (rows of O are 32-bit indices in the
 * kernels); larger batches return JFA_ERR_INVALID_ARG and launch nothing. */
jfa_status jfa_bcastq_fwd(const void *q, const void *k, const void *v, const void *kv_offsets,
                          jfa_index_t idx, int64_t B, int64_t Lq, int64_t Tk, int H, int D,
                          float scale, const int32_t *d_sm_ptr, const int32_t *d_tiles,
                          int num_sms, void *o, float *lse, void *workspace, size_t ws_bytes,
                          jfa_stream_t stream);

/* Broadcast-Q backward: dout device bf16 [B, Lq, H, D]; writes
 * dq = sum over b of each sequence's dQ (device fp32 [Lq, H, D]) and dk,
 * dv (device bf16 [Tk, H, D]). The per-sequence dQ partials are summed in
 * fp32 through a double-buffered shared-memory staging area ("Optimización
 * del proceso de Backward y dQ") straight into dq, which is therefore fp32:
 * a sum over the whole batch grows with B and a bf16 result would lose more
 * than the accumulation itself. The call clears dq first. Tiles: tile_rows =
 * jfa_tile_rows(JFA_OP_BCASTQ_BWD) over key blocks, fixed_work = Lq. Same
 * B * Lq limit as jfa_bcastq_fwd. */
jfa_status jfa_bcastq_bwd(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, const void *kv_offsets,
                          jfa_index_t idx, int64_t B, int64_t Lq, int64_t Tk, int H, int D,
                          float scale, const int32_t *d_sm_ptr, const int32_t *d_tiles,
                          int num_sms, float *dq, void *dk, void *dv, void *workspace,
                          size_t ws_bytes, jfa_stream_t stream);

/* Block-diagonal forward ("TLX Block Attention", sections 1-2): q, k, v
 * device bf16 [B, L, H, D], L a multiple of 64; each 64-token block attends
 * only within itself. One score tile per block, no online correction and
 * no LSE. o: device bf16 [B, L, H, D]. */
jfa_status blockdiag_fwd(const void *q, const void *k, const void *v, int64_t B, int64_t L,
                         int H, int D, float scale, void *o, void *workspace, size_t ws_bytes,
                         jfa_stream_t stream);

/* Block-diagonal backward ("TLX Block Attention", section 4): recomputes
 * S and P from Q and K (no LSE, no O), Di = rowsum(P * dP) (equal to
 * rowsum(dO * O) since O = P V), then dQ, dK, dV (device bf16 [B, L, H, D]). */
jfa_status blockdiag_bwd(const void *q, const void *k, const void *v, const void *dout,
                         int64_t B, int64_t L, int H, int D, float scale, void *dq, void *dk,
                         void *dv, void *workspace, size_t ws_bytes, jfa_stream_t stream);

/* Block-diagonal attention with rotary embeddings fused in ("TLX Block
 * Attention", section 1: block attention with rotary embeddings, whose
 * combined attention-and-rotary backward the page reports about 3.5 times
 * faster than FA2 when the rotary is fused into the attention epilogue). The
 * page does not write the rotation out; the reading used is the "rotate
 * half" form: cos_t, sin_t are device fp32 tables [L, D/2] indexed by a
 * token's position in its sequence (row index mod L), and each row x of q
 * and k is rotated,
 *   x_r[i] = x[i] cos[i] - x[i + D/2] sin[i],
 *   x_r[i + D/2] = x[i + D/2] cos[i] + x[i] sin[i],   i < D/2.
 * Forward: o = block-diagonal attention of (q_r, k_r, v), the rotated rows
 * rounded to bf16 like a separate rotary pass writing bf16. When q_rot and
 * k_rot (device bf16 [B, L, H, D], 16-byte aligned) are given, the rotated
 * rows are written there, as a rotary layer's output saved for its backward:
 * a rotary pass writes them and the plain forward runs on them (faster than
 * rotating inside the forward's two-stage pipeline). Both NULL writes
 * nothing and needs no scratch: q and k are rotated in shared memory inside
 * the forward on their way to the products. The two give the same o bit for
 * bit. One NULL is JFA_ERR_INVALID_ARG.
 * Backward (the rotary backward fused into the attention epilogue): takes the
 * rotated q_rot, k_rot (as written by the forward), v and dout; dq, dk are
 * the gradients with respect to the unrotated q, k (the gradients of q_rot,
 * k_rot rotated back by the transposed rotation in the epilogue); dv as for
 * blockdiag_bwd. Other arguments and errors as for blockdiag_fwd /
 * blockdiag_bwd; NULL or misaligned tables return JFA_ERR_INVALID_ARG. */
jfa_status blockdiag_rotary_fwd(const void *q, const void *k, const void *v, const float *cos_t,
                                const float *sin_t, int64_t B, int64_t L, int H, int D,
                                float scale, void *o, void *q_rot, void *k_rot, void *workspace,
                                size_t ws_bytes, jfa_stream_t stream);

jfa_status blockdiag_rotary_bwd(const void *q_rot, const void *k_rot, const void *v,
                                const void *dout, const float *cos_t, const float *sin_t,
                                int64_t B, int64_t L, int H, int D, float scale, void *dq,
                                void *dk, void *dv, void *workspace, size_t ws_bytes,
                                jfa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* JFA_H_ */
