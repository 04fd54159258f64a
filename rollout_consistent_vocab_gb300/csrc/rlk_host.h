// rlk_host.h -- host-side helpers shared by the library's translation units:
// the per-thread error message and the argument checks.
#pragma once

#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "rlk_logp.h"

namespace rlk {

inline char* last_error_buf() {
  static thread_local char buf[512] = "";
  return buf;
}

inline rlk_status fail(rlk_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(last_error_buf(), 512, fmt, ap);
  va_end(ap);
  return s;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline rlk_status check_out(const void* p, const char* what, bool required) {
  if (!p) return required ? fail(RLK_EINVAL, "%s is NULL", what) : RLK_OK;
  if (!aligned(p, 4)) return fail(RLK_EALIGN, "%s is not 4-byte aligned", what);
  return RLK_OK;
}

// A per-row parameter array (checked for alignment) or a scalar (checked for its domain).
inline rlk_status check_tau(const float* arr, float scalar) {
  if (arr) return aligned(arr, 4) ? RLK_OK : fail(RLK_EALIGN, "temperature is not 4-byte aligned");
  if (!(scalar >= 0.0f && scalar <= 3.402823466e38f))
    return fail(RLK_EINVAL, "temperature %g must be finite and >= 0", (double)scalar);
  return RLK_OK;
}
inline rlk_status check_top_p(const float* arr, float scalar) {
  if (arr) return aligned(arr, 4) ? RLK_OK : fail(RLK_EALIGN, "top_p is not 4-byte aligned");
  if (!(scalar > 0.0f && scalar <= 1.0f)) return fail(RLK_EINVAL, "top_p %g must be in (0, 1]", (double)scalar);
  return RLK_OK;
}
inline rlk_status check_top_k(const int32_t* arr, int32_t scalar) {
  if (arr) return aligned(arr, 4) ? RLK_OK : fail(RLK_EALIGN, "top_k is not 4-byte aligned");
  if (!(scalar == -1 || (scalar >= 1 && scalar <= RLK_VOCAB_REAL)))
    return fail(RLK_EINVAL, "top_k %d must be -1 or 1..%d", scalar, RLK_VOCAB_REAL);
  return RLK_OK;
}

}  // namespace rlk
