/*
 * rlk_norm.h -- C ABI of the deterministic gradient L2 norm for GB300
 * (sm_103a), part of librlk_logp.so.
 *
 * The operation ("H100 canonical CP backward validation", section "Change",
 * the paragraph on Megatron's L2 norm): the sum of the FP32 squares of the
 * gradient elements is gathered in integer bins keyed by exponent before the
 * distributed reduction, so that the sum -- and the norm that drives gradient
 * clipping -- does not depend on the order of the elements or on how they
 * are split across ranks.  The same page ("Timing and scope") times the norm
 * on 10M BF16-derived FP32 elements.
 *
 * Per element g (FP32, or BF16 / FP16 converted exactly to FP32):
 *   q = g * g in FP32, rounded to nearest even;
 *   q = M * 2^(E - 150) exactly, E the biased exponent field of q (a
 *   subnormal square counts as E = 1 with M its fraction).
 * The result is  S = sum over elements of q,  taken EXACTLY and rounded once
 * to float64 (nearest even), and  norm = sqrt(S)  correctly rounded in
 * float64.  A NaN square makes both NaN; otherwise an infinite square (g
 * infinite, or g*g above the FP32 range) makes both +inf.
 *
 * The bins: uint64_t[RLK_NORM_BINS] in device memory.
 *   bins[0]                   number of NaN squares
 *   bins[RLK_NORM_BINS - 1]   number of infinite squares
 *   bins[e], 1 <= e <= 382    an integer of weight 2^(e - 150)
 * The bins denote the exact value sum_e bins[e] 2^(e - 150); two bin vectors
 * add elementwise (integers, so in any order) to the bins of the union of
 * their elements.  That sum is the distributed reduction: an all-reduce
 * (SUM) of the 384 words across ranks, then rlk_sqnorm_finalize.  The kernel
 * may split the same exact value over the entries differently from one
 * launch to the next; the value, and so S and the norm, never change.
 * The bins stay exact while fewer than 2^38 elements in all have been
 * accumulated into them (every increment is below 2^24).
 *
 * Conventions: device pointers owned by the caller; nothing is allocated or
 * synchronised; work is enqueued on `stream` (a cudaStream_t as void*).
 * RLK_EINVAL for a null pointer (x may be NULL when n == 0), n < 0,
 * n > 2^36 or an unknown dtype; RLK_EALIGN for x not aligned to its element
 * size, or bins / out not 8-byte aligned; RLK_ECUDA for a launch failure.
 */
#ifndef RLK_NORM_H
#define RLK_NORM_H

#include <stdint.h>

#include "rlk_logp.h"

#ifdef __cplusplus
extern "C" {
#endif

#define RLK_NORM_BINS 384

typedef enum {
  RLK_DT_F32 = 0,
  RLK_DT_BF16 = 1,
  RLK_DT_F16 = 2
} rlk_dtype;

/* Add the squares of the n elements at x (dtype rlk_dtype) into bins
 * (device uint64_t[RLK_NORM_BINS], not cleared: zero it before the first
 * tensor).  n == 0 enqueues nothing. */
rlk_status rlk_sqnorm_accumulate(const void* x, int64_t n, int32_t dtype, uint64_t* bins,
                                 void* stream);

/* out[0] = the sum of squares S, out[1] = the norm (device double[2]). */
rlk_status rlk_sqnorm_finalize(const uint64_t* bins, double* out, void* stream);

/* One tensor end to end: clear bins, accumulate, finalize. */
rlk_status rlk_grad_norm(const void* x, int64_t n, int32_t dtype, uint64_t* bins, double* out,
                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RLK_NORM_H */
