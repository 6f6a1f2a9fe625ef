// Host-side helpers shared by the C-ABI translation units: status strings,
// the thread-local detail message and offsets validation.
#pragma once
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "jfa.h"

namespace jfa {

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
