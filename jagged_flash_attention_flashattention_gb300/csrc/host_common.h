// Host-side helpers shared by the C-ABI translation units: status strings,
// the thread-local detail message, offsets validation and the layout of the
// status block at the head of every workspace.
#pragma once
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "jfa.h"

namespace jfa {

// Bytes of the status block at the head of every workspace (and of the
// static scratch of jfa_bwd_noalloc): word 0 error code (0 = none), word 1
// wait site, word 2 block index; the uint64 at byte 128 counts accumulator
// bytes known to be zero.
constexpr size_t kStatusBytes = 256;

// Synchronises `stream` (a cudaStream_t), reads the status block at device
// address `status` and returns JFA_ERR_TIMEOUT if a kernel gave up waiting,
// after clearing the block's error words; JFA_OK otherwise.
jfa_status read_status_block(void *status, void *stream);

// Records a detail message for jfa_last_error() and returns `s`.
jfa_status fail(jfa_status s, const char *fmt, ...);

// Reads offsets[i] from a host array of int32 or int64.
inline int64_t offset_at(const void *off, jfa_index_t idx, int64_t i) {
  return idx == JFA_I32 ? (int64_t) static_cast<const int32_t *>(off)[i]
                        : static_cast<const int64_t *>(off)[i];
}

// Checks offsets[0] = 0, non-decreasing and (if T >= 0) offsets[B] = T.
jfa_status check_host_offsets(const void *off, jfa_index_t idx, int64_t B, int64_t T);

}  // namespace jfa
