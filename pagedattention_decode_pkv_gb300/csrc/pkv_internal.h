// Internal helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstdarg>
#include <cstddef>
#include <cstdint>

#include "../../include/pkv.h"

namespace pkv {

// Records the message for pkv_last_error_string() and returns `status`.
pkv_status set_error(pkv_status status, const char *fmt, ...);
pkv_status ok();

inline int64_t dtype_bytes(pkv_dtype t) { return t == PKV_F32 ? 4 : (t == PKV_F16 || t == PKV_BF16) ? 2 : 0; }
inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace pkv
