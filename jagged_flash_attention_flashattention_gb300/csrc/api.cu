// api.cu -- the extern "C" entry points of libjfa (declared in include/jfa.h):
// argument checks, TMA descriptor encoding and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "host_common.h"
#include "jfa.h"
#include "kernels.h"

using namespace jfa;

namespace {

constexpr uint64_t kTimeoutNs = 4ull * 1000 * 1000 * 1000;  // bounded waits give up after 4 s

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 [rows, H, D] as a 3-D tensor {D, H, rows}; box {64, 1, box_rows}, 128-byte swizzle.
jfa_status map_rows_bf16(CUtensorMap *m, const void *base, int64_t rows, int H, int D,
                         int box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return fail(JFA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (rows < 1) rows = 1;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(JFA_ERR_CUDA, "tensor map encode failed (%d)", (int)r);
  return JFA_OK;
}

// fp32 [rows, H, D] as {D, H, rows}; box {32, 1, 64}, no swizzle.
jfa_status map_acc_f32(CUtensorMap *m, void *base, int64_t rows, int H, int D) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return fail(JFA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (rows < 1) rows = 1;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  cuuint32_t box[3] = {32, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(JFA_ERR_CUDA, "tensor map encode failed (%d)", (int)r);
  return JFA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

jfa_status need_ptr(const void *p, const char *name) {
  if (!p) return fail(JFA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(JFA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return JFA_OK;
}

#define JFA_TRY(x)                    \
  do {                                \
    jfa_status _s = (x);              \
    if (_s != JFA_OK) return _s;      \
  } while (0)

jfa_status check_dims(int64_t B, int64_t T, int H, int D) {
  if (D != 64 && D != 128) return fail(JFA_ERR_UNSUPPORTED, "D = %d (supported: 64, 128)", D);
  if (H < 1) return fail(JFA_ERR_INVALID_ARG, "H = %d < 1", H);
  if (B < 0 || T < 0) return fail(JFA_ERR_INVALID_ARG, "negative size");
  if (T >= (int64_t(1) << 31) - 256) return fail(JFA_ERR_INVALID_ARG, "T too large");
  return JFA_OK;
}

jfa_status check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(JFA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return fail(JFA_ERR_WORKSPACE, "workspace not 16-byte aligned");
  if (ws_bytes < need)
    return fail(JFA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, need);
  return JFA_OK;
}

jfa_status check_sched(const int32_t *sm_ptr, const int32_t *tiles, int num_sms) {
  if (num_sms < 1) return fail(JFA_ERR_INVALID_ARG, "num_sms = %d < 1", num_sms);
  if (!sm_ptr) return fail(JFA_ERR_INVALID_ARG, "sm_ptr is NULL");
  if (!tiles) return fail(JFA_ERR_INVALID_ARG, "tiles is NULL");
  return JFA_OK;
}

jfa_status cuda_status(cudaError_t e, const char *what) {
  if (e != cudaSuccess) return fail(JFA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return JFA_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Dynamic tile scheduling: the claim counter sits in the status block, the
// device tile table ([B+1] int64) right after it.
constexpr size_t kDynQueueOff = 192;
size_t dyn_workspace_bytes(int64_t B) {
  return kStatusBytes + round_up((size_t)(B + 1) * sizeof(int64_t), 256);
}

}  // namespace

// ------------------------------------------------------------------ misc

extern "C" jfa_status jfa_tile_rows(jfa_op op, int D, int *tile_rows) {
  if (!tile_rows) return fail(JFA_ERR_INVALID_ARG, "tile_rows is NULL");
  if (D != 64 && D != 128) return fail(JFA_ERR_UNSUPPORTED, "D = %d", D);
  switch (op) {
    case JFA_OP_FWD:
    case JFA_OP_BCASTQ_FWD: *tile_rows = 256; return JFA_OK;
    case JFA_OP_BWD:
    case JFA_OP_BCASTQ_BWD: *tile_rows = 128; return JFA_OK;
    case JFA_OP_BLOCKDIAG_FWD:
    case JFA_OP_BLOCKDIAG_BWD: *tile_rows = 128; return JFA_OK;
    case JFA_OP_FWD_PAIR:
      if (D != 128) return fail(JFA_ERR_UNSUPPORTED, "the CTA-pair forward takes D = 128");
      *tile_rows = 512;
      return JFA_OK;
  }
  return fail(JFA_ERR_INVALID_ARG, "unknown op %d", (int)op);
}

extern "C" jfa_status jfa_num_sms(int *num_sms) {
  if (!num_sms) return fail(JFA_ERR_INVALID_ARG, "num_sms is NULL");
  int dev = 0;
  JFA_TRY(cuda_status(cudaGetDevice(&dev), "cudaGetDevice"));
  JFA_TRY(cuda_status(cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev),
                      "cudaDeviceGetAttribute"));
  return JFA_OK;
}

extern "C" size_t jfa_workspace_size(jfa_op op, int64_t n, int H, int D) {
  if (n < 0 || H < 1 || D < 1) return kStatusBytes;
  if (op == JFA_OP_BWD) return kStatusBytes + round_up((size_t)n * H * D * sizeof(float), 256);
  return kStatusBytes;
}

extern "C" jfa_status jfa_workspace_init(void *workspace, size_t ws_bytes, jfa_stream_t stream) {
  JFA_TRY(check_ws(workspace, ws_bytes, kStatusBytes));
  return cuda_status(cudaMemsetAsync(workspace, 0, kStatusBytes, (cudaStream_t)stream),
                     "cudaMemsetAsync");
}

jfa_status jfa::read_status_block(void *status, void *stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint32_t st[4] = {0, 0, 0, 0};
  JFA_TRY(cuda_status(cudaMemcpyAsync(st, status, sizeof(st), cudaMemcpyDeviceToHost, stream),
                      "cudaMemcpyAsync"));
  JFA_TRY(cuda_status(cudaStreamSynchronize(stream), "cudaStreamSynchronize"));
  if (st[0] != 0) {
    // The whole block is cleared; a zero count of cleared accumulator bytes
    // only makes the next backward clear its accumulator itself.
    cudaMemsetAsync(status, 0, kStatusBytes, stream);
    cudaStreamSynchronize(stream);
    if (st[0] == JFA_ERR_TIMEOUT)
      return fail(JFA_ERR_TIMEOUT, "kernel wait site %u in block %u gave up", st[1], st[2]);
    if (st[0] == JFA_ERR_WORKSPACE)
      return fail(JFA_ERR_WORKSPACE,
                  "the deterministic dQ partials need more rows than the workspace holds "
                  "(size it with jfa_varlen_workspace_size for the same offsets)");
    return fail(JFA_ERR_CUDA, "a kernel reported device status %u", st[0]);
  }
  return JFA_OK;
}

extern "C" jfa_status jfa_check_status(void *workspace, jfa_stream_t stream) {
  JFA_TRY(check_ws(workspace, kStatusBytes, kStatusBytes));
  return read_status_block(workspace, stream);
}

// ------------------------------------------------------------------ forward

namespace {

jfa_status check_window(int left, int right) {
  if (left < -1 || right < -1)
    return fail(JFA_ERR_INVALID_ARG, "window (%d, %d): bounds must be >= -1", left, right);
  return JFA_OK;
}

// Shared by every forward entry point. kv_offsets bound the K/V sequences;
// q_offsets the query sequences (jagged, may equal kv_offsets), or NULL with
// Lq > 0 for broadcast-Q (one dense Q of Lq rows); q_rows = rows of q.
jfa_status fwd_common(const void *q, const void *k, const void *v, const void *kv_offsets,
                      const void *q_offsets, jfa_index_t idx, int64_t B, int64_t q_rows,
                      int64_t Tk, int64_t Lq, int H, int D, float scale, int win_left,
                      int win_right, const int32_t *sm_ptr, const int32_t *tiles, int num_sms,
                      void *o, float *lse, void *ws, size_t ws_bytes, cudaStream_t st,
                      int dyn = 0, int64_t n_dyn_tiles = 0, bool pair = false,
                      const int32_t *blk_ptr = nullptr, const int32_t *blk_list = nullptr,
                      const int32_t *blk_meta = nullptr) {
  JFA_TRY(check_dims(B, Tk, H, D));
  JFA_TRY(check_dims(B, q_rows, H, D));
  JFA_TRY(check_window(win_left, win_right));
  if (idx != JFA_I32 && idx != JFA_I64) return fail(JFA_ERR_INVALID_ARG, "bad index type");
  if (!(scale > 0.f)) return fail(JFA_ERR_INVALID_ARG, "scale must be > 0");
  JFA_TRY(check_ws(ws, ws_bytes, kStatusBytes));
  if (num_sms < 1) return fail(JFA_ERR_INVALID_ARG, "num_sms = %d < 1", num_sms);
  JFA_TRY(need_ptr(kv_offsets, "kv_offsets"));
  if (Lq == 0) JFA_TRY(need_ptr(q_offsets, "q_offsets"));
  if (pair && (D != 128 || Lq != 0 || win_left >= 0 || win_right >= 0 || dyn != 0))
    return fail(JFA_ERR_UNSUPPORTED, "the CTA-pair forward takes jagged self-attention at D = 128 only");
  if (dyn == 2 && ws_bytes < dyn_workspace_bytes(B))
    return fail(JFA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, dyn_workspace_bytes(B));
  if (B == 0 || q_rows == 0) return JFA_OK;
  if (dyn == 0) JFA_TRY(check_sched(sm_ptr, tiles, num_sms));
  if (dyn == 1 && n_dyn_tiles > 0 && !tiles) return fail(JFA_ERR_INVALID_ARG, "tiles is NULL");
  if (blk_ptr || blk_list || blk_meta) {
    if (!blk_ptr || !blk_list || !blk_meta)
      return fail(JFA_ERR_INVALID_ARG, "list_ptr, list and meta must all be given");
    if (Lq != 0 || dyn != 0 || pair || win_left >= 0 || win_right >= 0)
      return fail(JFA_ERR_UNSUPPORTED, "block masks: jagged layouts without a band");
  }
  JFA_TRY(need_ptr(q, "q"));
  JFA_TRY(need_ptr(o, "o"));
  JFA_TRY(need_ptr(lse, "lse"));
  if (Tk > 0) {
    JFA_TRY(need_ptr(k, "k"));
    JFA_TRY(need_ptr(v, "v"));
  } else {
    k = v = q;  // never read: every K/V sequence is empty
  }
  FwdParams p;
  memset(&p, 0, sizeof(p));
  JFA_TRY(map_rows_bf16(&p.tm_q, q, q_rows, H, D, 128));
  JFA_TRY(map_rows_bf16(&p.tm_k, k, Tk > 0 ? Tk : q_rows, H, D, 128));
  JFA_TRY(map_rows_bf16(&p.tm_v, v, Tk > 0 ? Tk : q_rows, H, D, 128));
  if (pair) JFA_TRY(map_rows_bf16(&p.tm_khalf, k, Tk > 0 ? Tk : q_rows, H, D, 64));
  p.offsets = kv_offsets;
  p.q_offsets = Lq > 0 ? kv_offsets : q_offsets;
  p.idx64 = idx == JFA_I64;
  p.sm_ptr = sm_ptr;
  p.tiles = tiles;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.T = Tk;
  p.Tq = q_rows;
  p.win_left = win_left;
  p.win_right = win_right;
  p.H = H;
  p.Lq = (int)Lq;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = static_cast<uint32_t *>(ws);
  p.timeout_ns = kTimeoutNs;
  p.blk_ptr = blk_ptr;
  p.blk_list = blk_list;
  p.blk_meta = reinterpret_cast<const int4 *>(blk_meta);
  // A workspace sized for the jagged backward: clear its dQ accumulator here,
  // on the forward kernel's idle warps, instead of in a pass of its own.
  const size_t acc_bytes = (size_t)q_rows * H * D * sizeof(float);
  if (dyn) {  // the workspace holds the claim counter (and the tile table), no accumulator
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    p.dyn = dyn;
    p.queue = reinterpret_cast<int *>(wsb + kDynQueueOff);
    p.n_tiles = n_dyn_tiles;
    if (dyn == 2) {
      p.tile_base = reinterpret_cast<int64_t *>(wsb + kStatusBytes);
      JFA_TRY(cuda_status(launch_fwd_enum(p, const_cast<int64_t *>(p.tile_base), p.queue, st),
                          "tile enumeration"));
    } else {
      JFA_TRY(cuda_status(cudaMemsetAsync(p.queue, 0, sizeof(int), st), "cudaMemsetAsync"));
    }
  } else if (Lq == 0 && ws_bytes >= kStatusBytes + round_up(acc_bytes, 256)) {
    p.acc_zero = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kStatusBytes);
    p.acc_n16 = (int64_t)(acc_bytes / 16);
  }
  if (pair) return cuda_status(launch_fwd_pair(p, num_sms, st), "pair fwd launch");
  return cuda_status(launch_fwd(p, D, num_sms, st), "fwd launch");
}

}  // namespace

extern "C" jfa_status jfa_fwd(const void *q, const void *k, const void *v, const void *offsets,
                              jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                              const int32_t *d_sm_ptr, const int32_t *d_tiles, int num_sms,
                              void *o, float *lse, void *workspace, size_t ws_bytes,
                              jfa_stream_t stream) {
  return fwd_common(q, k, v, offsets, offsets, idx, B, T, T, 0, H, D, scale, -1, -1, d_sm_ptr,
                    d_tiles, num_sms, o, lse, workspace, ws_bytes, (cudaStream_t)stream);
}

extern "C" jfa_status jfa_fwd_pair(const void *q, const void *k, const void *v,
                                   const void *offsets, jfa_index_t idx, int64_t B, int64_t T, int H,
                                   int D, float scale, const int32_t *d_sm_ptr,
                                   const int32_t *d_tiles, int num_pairs, void *o, float *lse,
                                   void *workspace, size_t ws_bytes, jfa_stream_t stream) {
  return fwd_common(q, k, v, offsets, offsets, idx, B, T, T, 0, H, D, scale, -1, -1, d_sm_ptr,
                    d_tiles, num_pairs, o, lse, workspace, ws_bytes, (cudaStream_t)stream, 0, 0,
                    true);
}

extern "C" jfa_status jfa_num_pairs(int *num_pairs) {
  if (!num_pairs) return fail(JFA_ERR_INVALID_ARG, "num_pairs is NULL");
  const int n = fwd_pair_max_clusters();
  if (n < 1) return fail(JFA_ERR_UNSUPPORTED, "no cluster of two CTAs of the pair forward fits");
  *num_pairs = n;
  return JFA_OK;
}

extern "C" jfa_status jfa_fwd_dynamic(const void *q, const void *k, const void *v,
                                      const void *offsets, jfa_index_t idx, int64_t B, int64_t T,
                                      int H, int D, float scale, const int32_t *d_tiles,
                                      int64_t n_tiles, int num_ctas, void *o, float *lse,
                                      void *workspace, size_t ws_bytes, jfa_stream_t stream) {
  if (n_tiles < 0 || n_tiles >= (int64_t(1) << 31) / 3) return fail(JFA_ERR_INVALID_ARG, "bad n_tiles");
  return fwd_common(q, k, v, offsets, offsets, idx, B, T, T, 0, H, D, scale, -1, -1, nullptr,
                    d_tiles, num_ctas, o, lse, workspace, ws_bytes, (cudaStream_t)stream,
                    d_tiles ? 1 : 2, n_tiles);
}

extern "C" size_t jfa_fwd_dynamic_workspace_size(int64_t B) {
  return B < 0 ? kStatusBytes : dyn_workspace_bytes(B);
}

extern "C" jfa_status jfa_varlen_fwd(const void *q, const void *k, const void *v,
                                     const void *q_offsets, const void *kv_offsets,
                                     jfa_index_t idx, int64_t B, int64_t Tq, int64_t Tk, int H,
                                     int D, float scale, int window_left, int window_right,
                                     const int32_t *d_sm_ptr, const int32_t *d_tiles,
                                     int num_sms, void *o, float *lse, void *workspace,
                                     size_t ws_bytes, jfa_stream_t stream) {
  return fwd_common(q, k, v, kv_offsets, q_offsets, idx, B, Tq, Tk, 0, H, D, scale, window_left,
                    window_right, d_sm_ptr, d_tiles, num_sms, o, lse, workspace, ws_bytes,
                    (cudaStream_t)stream);
}

extern "C" jfa_status jfa_bcastq_fwd(const void *q, const void *k, const void *v,
                                     const void *kv_offsets, jfa_index_t idx, int64_t B,
                                     int64_t Lq, int64_t Tk, int H, int D, float scale,
                                     const int32_t *d_sm_ptr, const int32_t *d_tiles,
                                     int num_sms, void *o, float *lse, void *workspace,
                                     size_t ws_bytes, jfa_stream_t stream) {
  if (Lq < 0 || Lq >= (1 << 30)) return fail(JFA_ERR_INVALID_ARG, "bad Lq");
  if (B > 0 && Lq >= ((int64_t(1) << 31) - 256) / B)  // O rows are addressed with 32-bit indices
    return fail(JFA_ERR_INVALID_ARG, "B * Lq too large");
  if (Lq == 0) return JFA_OK;
  return fwd_common(q, k, v, kv_offsets, nullptr, idx, B, Lq, Tk, Lq, H, D, scale, -1, -1,
                    d_sm_ptr, d_tiles, num_sms, o, lse, workspace, ws_bytes, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ backward

namespace {

jfa_status launch_status(cudaError_t e, const char *what) {
  if (e == cudaErrorNotSupported) return fail(JFA_ERR_UNSUPPORTED, "%s: not built", what);
  return cuda_status(e, what);
}

// Bytes of the deterministic workspace header: the status block, then the
// per-sequence partial-row and query-block prefix sums ([B+1] int64 each).
size_t det_header_bytes(int64_t B) {
  return kStatusBytes + round_up(2 * (size_t)(B + 1) * sizeof(int64_t), 256);
}

// Shared by every backward entry point (see fwd_common for the offsets).
jfa_status bwd_common(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, const void *kv_offsets,
                      const void *q_offsets, jfa_index_t idx, int64_t B, int64_t q_rows,
                      int64_t Tk, int64_t Lq, int H, int D, float scale, int win_left,
                      int win_right, int det, const int32_t *sm_ptr, const int32_t *tiles,
                      int num_sms, void *dq, void *dk, void *dv, void *ws, size_t ws_bytes,
                      cudaStream_t st, const float *cos_t = nullptr, const float *sin_t = nullptr,
                      int64_t rope_L = 0, const int32_t *blk_ptr = nullptr,
                      const int32_t *blk_list = nullptr) {
  JFA_TRY(check_dims(B, Tk, H, D));
  JFA_TRY(check_dims(B, q_rows, H, D));
  if (cos_t || sin_t) {
    JFA_TRY(need_ptr(cos_t, "cos"));
    JFA_TRY(need_ptr(sin_t, "sin"));
    if (rope_L < 1) return fail(JFA_ERR_INVALID_ARG, "rotary tables have %lld rows", (long long)rope_L);
    if (Lq != 0 || det || win_left >= 0 || win_right >= 0)
      return fail(JFA_ERR_UNSUPPORTED, "rotary backward: jagged self-attention without a band");
  }
  JFA_TRY(check_window(win_left, win_right));
  if (blk_ptr || blk_list) {
    if (!blk_ptr || !blk_list) return fail(JFA_ERR_INVALID_ARG, "list_ptr and list must both be given");
    if (Lq != 0 || det || win_left >= 0 || win_right >= 0 || cos_t)
      return fail(JFA_ERR_UNSUPPORTED, "block masks: jagged layouts without a band or deterministic dQ");
  }
  if (idx != JFA_I32 && idx != JFA_I64) return fail(JFA_ERR_INVALID_ARG, "bad index type");
  if (!(scale > 0.f)) return fail(JFA_ERR_INVALID_ARG, "scale must be > 0");
  if (det && Lq > 0) return fail(JFA_ERR_UNSUPPORTED, "deterministic dQ is for the jagged layouts");
  const int64_t acc_rows = Lq > 0 ? Lq : q_rows;
  // Jagged: fp32 accumulator in the workspace, cast to bf16 at the end (or,
  // deterministic, per-key-block partials summed in order by the cast).
  // Broadcast-Q: the caller's fp32 dq is the accumulator itself.
  const size_t need =
      det ? det_header_bytes(B)
          : kStatusBytes + (Lq > 0 ? 0 : round_up((size_t)acc_rows * H * D * sizeof(float), 256));
  JFA_TRY(check_ws(ws, ws_bytes, need));
  if (num_sms < 1) return fail(JFA_ERR_INVALID_ARG, "num_sms = %d < 1", num_sms);
  JFA_TRY(need_ptr(kv_offsets, "kv_offsets"));
  if (Lq == 0) JFA_TRY(need_ptr(q_offsets, "q_offsets"));
  if (B == 0 || (q_rows == 0 && Tk == 0)) return JFA_OK;
  if (Tk > 0) {
    JFA_TRY(need_ptr(k, "k"));
    JFA_TRY(need_ptr(v, "v"));
    JFA_TRY(need_ptr(dk, "dk"));
    JFA_TRY(need_ptr(dv, "dv"));
  } else {
    k = v = q;
  }
  if (q_rows == 0) {  // keys that no query sees: dK = dV = 0
    const size_t kv_bytes = (size_t)Tk * H * D * 2;
    JFA_TRY(cuda_status(cudaMemsetAsync(dk, 0, kv_bytes, st), "cudaMemsetAsync"));
    return cuda_status(cudaMemsetAsync(dv, 0, kv_bytes, st), "cudaMemsetAsync");
  }
  JFA_TRY(check_sched(sm_ptr, tiles, num_sms));
  JFA_TRY(need_ptr(q, "q"));
  JFA_TRY(need_ptr(o, "o"));
  JFA_TRY(need_ptr(lse, "lse"));
  JFA_TRY(need_ptr(dout, "dout"));
  JFA_TRY(need_ptr(dq, "dq"));
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  float *acc = Lq > 0 ? static_cast<float *>(dq) : reinterpret_cast<float *>(wsb + kStatusBytes);
  BwdParams p;
  memset(&p, 0, sizeof(p));
  const int64_t o_rows = Lq > 0 ? B * Lq : q_rows;
  JFA_TRY(map_rows_bf16(&p.tm_q, q, acc_rows, H, D, 64));
  JFA_TRY(map_rows_bf16(&p.tm_do, dout, o_rows, H, D, 64));
  JFA_TRY(map_rows_bf16(&p.tm_k, k, Tk > 0 ? Tk : 1, H, D, 128));
  JFA_TRY(map_rows_bf16(&p.tm_v, v, Tk > 0 ? Tk : 1, H, D, 128));
  float *part = nullptr;
  int64_t *det_base = nullptr, *qb_base = nullptr;
  if (det) {
    det_base = reinterpret_cast<int64_t *>(wsb + kStatusBytes);
    qb_base = det_base + (B + 1);
    part = reinterpret_cast<float *>(wsb + det_header_bytes(B));
    p.det = 1;
    p.det_base = det_base;
    // Partial rows are 32-bit TMA coordinates: at most 2^31 - 64 of them.
    p.det_rows = (int64_t)((ws_bytes - det_header_bytes(B)) / ((size_t)H * D * sizeof(float)));
    if (p.det_rows > (int64_t(1) << 31) - 64) p.det_rows = (int64_t(1) << 31) - 64;
    JFA_TRY(map_acc_f32(&p.tm_dqpart, part, p.det_rows > 0 ? p.det_rows : 1, H, D));
    JFA_TRY(map_acc_f32(&p.tm_dqacc, part, p.det_rows > 0 ? p.det_rows : 1, H, D));  // unused
  } else {
    JFA_TRY(map_acc_f32(&p.tm_dqacc, acc, acc_rows, H, D));
  }
  p.offsets = kv_offsets;
  p.q_offsets = Lq > 0 ? kv_offsets : q_offsets;
  p.idx64 = idx == JFA_I64;
  p.sm_ptr = sm_ptr;
  p.tiles = tiles;
  p.lse = lse;
  p.o = o;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.T = Tk;
  p.Tq = q_rows;
  p.win_left = win_left;
  p.win_right = win_right;
  p.H = H;
  p.Lq = (int)Lq;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = static_cast<uint32_t *>(ws);
  p.timeout_ns = kTimeoutNs;
  p.cos_t = cos_t;
  p.sin_t = sin_t;
  p.rope_L = rope_L;
  p.blk_ptr = blk_ptr;
  p.blk_list = blk_list;
  if (det) {
    JFA_TRY(launch_status(launch_det_layout(p, det_base, qb_base, st), "deterministic layout"));
    if (Tk > 0) JFA_TRY(launch_status(launch_bwd(p, D, num_sms, st), "bwd launch"));
    return launch_status(launch_det_cast(p, part, qb_base, dq, D, num_sms, st), "dq sum");
  }
  const size_t acc_bytes = (size_t)acc_rows * H * D * sizeof(float);
  if (Lq > 0)
    JFA_TRY(cuda_status(cudaMemsetAsync(acc, 0, acc_bytes, st), "cudaMemsetAsync"));
  else  // skipped on the device when a forward pass has already cleared it
    JFA_TRY(launch_status(launch_acc_clear(acc, (int64_t)(acc_bytes / 16), p.status, st),
                          "accumulator clear"));
  if (Tk > 0) JFA_TRY(launch_status(launch_bwd(p, D, num_sms, st), "bwd launch"));
  if (Lq > 0) return JFA_OK;
  if (cos_t) return launch_status(launch_dq_convert_rope(p, acc, dq, acc_rows, D, st), "dq convert");
  return launch_status(launch_dq_convert(acc, dq, acc_rows, H, D, scale, p.status, st), "dq convert");
}

}  // namespace

extern "C" jfa_status jfa_bwd(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dout, const void *offsets,
                              jfa_index_t idx, int64_t B, int64_t T, int H, int D, float scale,
                              const int32_t *d_sm_ptr, const int32_t *d_tiles, int num_sms,
                              void *dq, void *dk, void *dv, void *workspace, size_t ws_bytes,
                              jfa_stream_t stream) {
  return bwd_common(q, k, v, o, lse, dout, offsets, offsets, idx, B, T, T, 0, H, D, scale, -1, -1,
                    0, d_sm_ptr, d_tiles, num_sms, dq, dk, dv, workspace, ws_bytes,
                    (cudaStream_t)stream);
}

extern "C" jfa_status jfa_rotary_bwd(const void *q_rot, const void *k_rot, const void *v,
                                     const void *o, const float *lse, const void *dout,
                                     const void *offsets, jfa_index_t idx, int64_t B, int64_t T,
                                     int H, int D, float scale, const float *cos_t,
                                     const float *sin_t, int64_t rope_L, const int32_t *d_sm_ptr,
                                     const int32_t *d_tiles, int num_sms, void *dq, void *dk,
                                     void *dv, void *workspace, size_t ws_bytes,
                                     jfa_stream_t stream) {
  if (!cos_t || !sin_t) return fail(JFA_ERR_INVALID_ARG, "rotary tables are NULL");
  return bwd_common(q_rot, k_rot, v, o, lse, dout, offsets, offsets, idx, B, T, T, 0, H, D, scale,
                    -1, -1, 0, d_sm_ptr, d_tiles, num_sms, dq, dk, dv, workspace, ws_bytes,
                    (cudaStream_t)stream, cos_t, sin_t, rope_L);
}

extern "C" jfa_status jfa_rope(const void *x, const void *offsets, jfa_index_t idx, int64_t B,
                               int64_t T, int H, int D, const float *cos_t, const float *sin_t,
                               int64_t rope_L, void *x_rot, jfa_stream_t stream) {
  JFA_TRY(check_dims(B, T, H, D));
  if (idx != JFA_I32 && idx != JFA_I64) return fail(JFA_ERR_INVALID_ARG, "bad index type");
  if (rope_L < 1) return fail(JFA_ERR_INVALID_ARG, "rotary tables have %lld rows", (long long)rope_L);
  JFA_TRY(need_ptr(cos_t, "cos"));
  JFA_TRY(need_ptr(sin_t, "sin"));
  JFA_TRY(need_ptr(offsets, "offsets"));
  if (B == 0 || T == 0) return JFA_OK;
  JFA_TRY(need_ptr(x, "x"));
  JFA_TRY(need_ptr(x_rot, "x_rot"));
  return cuda_status(launch_rope_rows(x, x_rot, T, H, D, offsets, idx == JFA_I64, B, cos_t, sin_t,
                                      rope_L, 0, (cudaStream_t)stream),
                     "rope launch");
}

extern "C" jfa_status jfa_varlen_bwd(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dout, const void *q_offsets,
                                     const void *kv_offsets, jfa_index_t idx, int64_t B,
                                     int64_t Tq, int64_t Tk, int H, int D, float scale,
                                     int window_left, int window_right, int deterministic,
                                     const int32_t *d_sm_ptr, const int32_t *d_tiles,
                                     int num_sms, void *dq, void *dk, void *dv, void *workspace,
                                     size_t ws_bytes, jfa_stream_t stream) {
  return bwd_common(q, k, v, o, lse, dout, kv_offsets, q_offsets, idx, B, Tq, Tk, 0, H, D, scale,
                    window_left, window_right, deterministic ? 1 : 0, d_sm_ptr, d_tiles, num_sms,
                    dq, dk, dv, workspace, ws_bytes, (cudaStream_t)stream);
}

extern "C" jfa_status jfa_sparse_fwd(const void *q, const void *k, const void *v,
                                     const void *q_offsets, const void *kv_offsets,
                                     jfa_index_t idx, int64_t B, int64_t Tq, int64_t Tk, int H,
                                     int D, float scale, const int32_t *d_sm_ptr,
                                     const int32_t *d_tiles, const int32_t *d_list_ptr,
                                     const int32_t *d_list, const int32_t *d_meta, int num_sms,
                                     void *o, float *lse, void *workspace, size_t ws_bytes,
                                     jfa_stream_t stream) {
  JFA_TRY(need_ptr(d_list_ptr, "list_ptr"));
  JFA_TRY(need_ptr(d_list, "list"));
  JFA_TRY(need_ptr(d_meta, "meta"));
  return fwd_common(q, k, v, kv_offsets, q_offsets, idx, B, Tq, Tk, 0, H, D, scale, -1, -1,
                    d_sm_ptr, d_tiles, num_sms, o, lse, workspace, ws_bytes, (cudaStream_t)stream,
                    0, 0, false, d_list_ptr, d_list, d_meta);
}

extern "C" jfa_status jfa_sparse_bwd(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dout, const void *q_offsets,
                                     const void *kv_offsets, jfa_index_t idx, int64_t B,
                                     int64_t Tq, int64_t Tk, int H, int D, float scale,
                                     const int32_t *d_sm_ptr, const int32_t *d_tiles,
                                     const int32_t *d_list_ptr, const int32_t *d_list,
                                     int num_sms, void *dq, void *dk, void *dv, void *workspace,
                                     size_t ws_bytes, jfa_stream_t stream) {
  JFA_TRY(need_ptr(d_list_ptr, "list_ptr"));
  JFA_TRY(need_ptr(d_list, "list"));
  return bwd_common(q, k, v, o, lse, dout, kv_offsets, q_offsets, idx, B, Tq, Tk, 0, H, D, scale,
                    -1, -1, 0, d_sm_ptr, d_tiles, num_sms, dq, dk, dv, workspace, ws_bytes,
                    (cudaStream_t)stream, nullptr, nullptr, 0, d_list_ptr, d_list);
}

extern "C" jfa_status jfa_varlen_workspace_size(int64_t B, const void *host_q_offsets,
                                                const void *host_kv_offsets, jfa_index_t idx,
                                                int H, int D, int deterministic, size_t *bytes) {
  if (!bytes) return fail(JFA_ERR_INVALID_ARG, "bytes is NULL");
  if (H < 1 || D < 1) return fail(JFA_ERR_INVALID_ARG, "bad H or D");
  if (!host_q_offsets) host_q_offsets = host_kv_offsets;
  JFA_TRY(check_host_offsets(host_kv_offsets, idx, B, -1));
  JFA_TRY(check_host_offsets(host_q_offsets, idx, B, -1));
  const int64_t Tq = offset_at(host_q_offsets, idx, B);
  if (!deterministic) {
    *bytes = kStatusBytes + round_up((size_t)Tq * H * D * sizeof(float), 256);
    return JFA_OK;
  }
  size_t rows = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t Lq = offset_at(host_q_offsets, idx, b + 1) - offset_at(host_q_offsets, idx, b);
    const int64_t Lk = offset_at(host_kv_offsets, idx, b + 1) - offset_at(host_kv_offsets, idx, b);
    rows += (size_t)((Lk + 127) / 128) * (size_t)((Lq + 63) / 64 * 64);
  }
  *bytes = det_header_bytes(B) + rows * H * D * sizeof(float);
  return JFA_OK;
}

extern "C" jfa_status jfa_bcastq_bwd(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dout, const void *kv_offsets,
                                     jfa_index_t idx, int64_t B, int64_t Lq, int64_t Tk, int H,
                                     int D, float scale, const int32_t *d_sm_ptr,
                                     const int32_t *d_tiles, int num_sms, float *dq, void *dk,
                                     void *dv, void *workspace, size_t ws_bytes,
                                     jfa_stream_t stream) {
  if (Lq < 0 || Lq >= (1 << 30)) return fail(JFA_ERR_INVALID_ARG, "bad Lq");
  if (B > 0 && Lq >= ((int64_t(1) << 31) - 256) / B)  // O / dO rows use 32-bit indices
    return fail(JFA_ERR_INVALID_ARG, "B * Lq too large");
  if (Lq == 0) return JFA_OK;
  return bwd_common(q, k, v, o, lse, dout, kv_offsets, nullptr, idx, B, Lq, Tk, Lq, H, D, scale,
                    -1, -1, 0, d_sm_ptr, d_tiles, num_sms, dq, dk, dv, workspace, ws_bytes,
                    (cudaStream_t)stream);
}

// ------------------------------------------------------------ block-diagonal

namespace {

jfa_status blockdiag_common(const void *q, const void *k, const void *v, const void *dout,
                            int64_t B, int64_t L, int H, int D, float scale, void *o, void *dq,
                            void *dk, void *dv, void *ws, size_t ws_bytes, bool bwd,
                            cudaStream_t st, const float *cos_t = nullptr,
                            const float *sin_t = nullptr, bool rotary = false,
                            void *q_rot = nullptr, void *k_rot = nullptr) {
  JFA_TRY(check_dims(B, B * L, H, D));
  if (L < 0 || L % 64 != 0) return fail(JFA_ERR_INVALID_ARG, "L = %lld is not a multiple of 64", (long long)L);
  if (!(scale > 0.f)) return fail(JFA_ERR_INVALID_ARG, "scale must be > 0");
  JFA_TRY(check_ws(ws, ws_bytes, kStatusBytes));
  if (rotary) {
    JFA_TRY(need_ptr(cos_t, "cos"));
    JFA_TRY(need_ptr(sin_t, "sin"));
    if ((q_rot == nullptr) != (k_rot == nullptr))
      return fail(JFA_ERR_INVALID_ARG, "q_rot and k_rot must both be given or both be NULL");
    if (q_rot != nullptr) {
      JFA_TRY(need_ptr(q_rot, "q_rot"));
      JFA_TRY(need_ptr(k_rot, "k_rot"));
    }
  }
  if (B == 0 || L == 0) return JFA_OK;
  JFA_TRY(need_ptr(q, "q"));
  JFA_TRY(need_ptr(k, "k"));
  JFA_TRY(need_ptr(v, "v"));
  if (rotary && !bwd && q_rot != nullptr) {
    // The caller keeps the rotated rows: write them with the rotary pass
    // (HBM-bound, positions row mod L) and run the plain forward on them; the
    // same rotation and the same products as the fused forward (bit-identical),
    // off the fused kernel's two-stage pipeline. Without q_rot and k_rot the
    // fused forward rotates in shared memory and needs no scratch.
    JFA_TRY(cuda_status(launch_rope_rows(q, q_rot, B * L, H, D, nullptr, 0, B, cos_t, sin_t, L, L, st),
                        "rope launch"));
    JFA_TRY(cuda_status(launch_rope_rows(k, k_rot, B * L, H, D, nullptr, 0, B, cos_t, sin_t, L, L, st),
                        "rope launch"));
    return blockdiag_common(q_rot, k_rot, v, nullptr, B, L, H, D, scale, o, nullptr, nullptr,
                            nullptr, ws, ws_bytes, false, st);
  }
  BlockdiagParams p;
  memset(&p, 0, sizeof(p));
  const int64_t rows = B * L;
  JFA_TRY(map_rows_bf16(&p.tm_q, q, rows, H, D, 128));
  JFA_TRY(map_rows_bf16(&p.tm_k, k, rows, H, D, 128));
  JFA_TRY(map_rows_bf16(&p.tm_v, v, rows, H, D, 128));
  if (bwd) {
    JFA_TRY(need_ptr(dout, "dout"));
    JFA_TRY(need_ptr(dq, "dq"));
    JFA_TRY(need_ptr(dk, "dk"));
    JFA_TRY(need_ptr(dv, "dv"));
    JFA_TRY(map_rows_bf16(&p.tm_do, dout, rows, H, D, 128));
  } else {
    JFA_TRY(need_ptr(o, "o"));
  }
  p.o = o;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.rows = rows;
  p.L = L;
  p.cos_t = rotary ? cos_t : nullptr;
  p.sin_t = rotary ? sin_t : nullptr;
  p.H = H;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = static_cast<uint32_t *>(ws);
  p.timeout_ns = kTimeoutNs;
  int dev = 0, sms = 0;
  JFA_TRY(cuda_status(cudaGetDevice(&dev), "cudaGetDevice"));
  JFA_TRY(cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                      "cudaDeviceGetAttribute"));
  return launch_status(bwd ? launch_blockdiag_bwd(p, D, sms, st) : launch_blockdiag_fwd(p, D, sms, st),
                       bwd ? "blockdiag bwd launch" : "blockdiag fwd launch");
}

}  // namespace

extern "C" jfa_status blockdiag_fwd(const void *q, const void *k, const void *v, int64_t B,
                                    int64_t L, int H, int D, float scale, void *o,
                                    void *workspace, size_t ws_bytes, jfa_stream_t stream) {
  return blockdiag_common(q, k, v, nullptr, B, L, H, D, scale, o, nullptr, nullptr, nullptr,
                          workspace, ws_bytes, false, (cudaStream_t)stream);
}

extern "C" jfa_status blockdiag_bwd(const void *q, const void *k, const void *v,
                                    const void *dout, int64_t B, int64_t L, int H, int D,
                                    float scale, void *dq, void *dk, void *dv, void *workspace,
                                    size_t ws_bytes, jfa_stream_t stream) {
  return blockdiag_common(q, k, v, dout, B, L, H, D, scale, nullptr, dq, dk, dv, workspace,
                          ws_bytes, true, (cudaStream_t)stream);
}

extern "C" jfa_status blockdiag_rotary_fwd(const void *q, const void *k, const void *v,
                                           const float *cos_t, const float *sin_t, int64_t B,
                                           int64_t L, int H, int D, float scale, void *o,
                                           void *q_rot, void *k_rot, void *workspace,
                                           size_t ws_bytes, jfa_stream_t stream) {
  return blockdiag_common(q, k, v, nullptr, B, L, H, D, scale, o, nullptr, nullptr, nullptr,
                          workspace, ws_bytes, false, (cudaStream_t)stream, cos_t, sin_t, true,
                          q_rot, k_rot);
}

extern "C" jfa_status blockdiag_rotary_bwd(const void *q_rot, const void *k_rot, const void *v,
                                           const void *dout, const float *cos_t,
                                           const float *sin_t, int64_t B, int64_t L, int H, int D,
                                           float scale, void *dq, void *dk, void *dv,
                                           void *workspace, size_t ws_bytes, jfa_stream_t stream) {
  return blockdiag_common(q_rot, k_rot, v, dout, B, L, H, D, scale, nullptr, dq, dk, dv, workspace,
                          ws_bytes, true, (cudaStream_t)stream, cos_t, sin_t, true);
}
