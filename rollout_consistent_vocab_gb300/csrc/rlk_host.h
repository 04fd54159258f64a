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

// Logits buffer: base 16-byte aligned, rows a multiple of 8 elements apart.
inline rlk_status check_logits(const void* logits, int64_t T, int64_t stride, const char* what) {
  if (!logits) return fail(RLK_EINVAL, "%s is NULL", what);
  if (stride < RLK_VOCAB_PADDED) return fail(RLK_EINVAL, "%s row_stride %lld < %d", what, (long long)stride, RLK_VOCAB_PADDED);
  if (!aligned(logits, 16)) return fail(RLK_EALIGN, "%s base is not 16-byte aligned", what);
  if (stride % 8 != 0) return fail(RLK_EALIGN, "%s row_stride %lld is not a multiple of 8", what, (long long)stride);
  (void)T;
  return RLK_OK;
}

inline rlk_status check_args(const rlk_logp_args* a, bool restr, bool need_target = true) {
  if (!a) return fail(RLK_EINVAL, "args is NULL");
  if (a->T < 0) return fail(RLK_EINVAL, "T = %lld < 0", (long long)a->T);
  if (a->T >= (int64_t(1) << 28)) return fail(RLK_EINVAL, "T = %lld: at most 2^28 - 1 rows per call", (long long)a->T);
  if (a->vocab_real != RLK_VOCAB_REAL || a->vocab_padded != RLK_VOCAB_PADDED)
    return fail(RLK_EINVAL, "vocab sizes must be %d/%d, got %d/%d", RLK_VOCAB_REAL, RLK_VOCAB_PADDED, a->vocab_real, a->vocab_padded);
  if (a->T == 0) return RLK_OK;
  rlk_status s = check_logits(a->logits, a->T, a->row_stride, "logits");
  if (s != RLK_OK) return s;
  if (need_target) {
    if (!a->target) return fail(RLK_EINVAL, "target is NULL");
    if (!aligned(a->target, 4)) return fail(RLK_EALIGN, "target is not 4-byte aligned");
  }
  if ((s = check_tau(a->temperature, a->temperature_scalar)) != RLK_OK) return s;
  if (restr) {
    if ((s = check_top_p(a->top_p, a->top_p_scalar)) != RLK_OK) return s;
    if ((s = check_top_k(a->top_k, a->top_k_scalar)) != RLK_OK) return s;
  }
  if (a->err_count && !aligned(a->err_count, 4)) return fail(RLK_EALIGN, "err_count is not 4-byte aligned");
  return RLK_OK;
}

// Gradient buffer of a backward pass: [T, stride] bf16 or f32, base 16-byte
// aligned, rows a multiple of 16 bytes apart; and the upstream gradients.
inline rlk_status check_grad_args(const float* grad_full, const float* grad_restr, const void* grad,
                                  int64_t stride, int32_t dtype) {
  if (!grad_full && !grad_restr) return fail(RLK_EINVAL, "grad_full and grad_restr are both NULL");
  rlk_status s;
  if ((s = check_out(grad_full, "grad_full", false)) != RLK_OK) return s;
  if ((s = check_out(grad_restr, "grad_restr", false)) != RLK_OK) return s;
  if (dtype != RLK_GRAD_BF16 && dtype != RLK_GRAD_F32)
    return fail(RLK_EINVAL, "grad_dtype %d must be RLK_GRAD_BF16 or RLK_GRAD_F32", dtype);
  if (!grad) return fail(RLK_EINVAL, "grad_logits is NULL");
  if (stride < RLK_VOCAB_PADDED)
    return fail(RLK_EINVAL, "grad_row_stride %lld < %d", (long long)stride, RLK_VOCAB_PADDED);
  const int esize = dtype == RLK_GRAD_F32 ? 4 : 2;
  if (!aligned(grad, 16)) return fail(RLK_EALIGN, "grad_logits is not 16-byte aligned");
  if ((stride * esize) % 16 != 0)
    return fail(RLK_EALIGN, "grad_row_stride %lld is not a multiple of 16 bytes", (long long)stride);
  return RLK_OK;
}

// The sampler behind rlk_sample and rlk_sample_noalloc: `workspace` holds
// the 16-byte per-row records; `bits` (NULL: not kept) the per-row, per-shard
// chunk bitmaps that let rows whose support lies in the first candidate
// window be drawn from the marked chunks alone.
rlk_status sample_impl(const rlk_logp_args* args, unsigned long long seed,
                       const unsigned long long* counter, const uint32_t* uniform,
                       int32_t* out_token, float* out_restr, float* out_full,
                       int32_t* out_support, void* workspace, uint32_t* bits, void* stream);

}  // namespace rlk
