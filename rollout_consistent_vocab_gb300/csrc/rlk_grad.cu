// rlk_grad.cu -- the backward pass from a saved per-row record.
//
// The forward (rlk_logp_pair_save) resolves each row and keeps 16 bytes per
// row: the maximum M, 1/Z, 1/Z_S and the support's lowest order key.  The
// gradient with respect to the logits is then an element-wise map of each
// row, so this pass is a pure stream: one CTA per (row, shard) pulls the
// shard's 38 KB with a bulk copy (TMA) into shared memory and writes the
// gradient with streaming stores, through the same coefficient and element
// code (rlk_device.cuh) as the single-pass backward, hence the same bits.
// The training side differentiates the very logprobs the rollout side
// scored ("H100 canonical CP backward validation"); nothing here depends on
// T or on where the row sits.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include "rlk_logp.h"
#include "rlk_device.cuh"
#include "rlk_host.h"

namespace rlk {

struct __align__(128) GradSmem {
  uint4 shard[SHARD_CHUNKS];
  unsigned long long bar_load;
};

struct GParams {
  const uint16_t* logits;
  int64_t stride;
  const int32_t* target;
  const float* tau_arr;
  float tau_s;
  const rlk_row_stats* stats;
  const float* g_full;
  const float* g_restr;
  char* grad;
  int64_t grad_stride;
  int grad_f32;
};

__global__ void __launch_bounds__(NTHR, CTAS_PER_SM) grad_kernel(const GParams P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GradSmem& S = *reinterpret_cast<GradSmem*>(smem_raw);
  const int64_t row = blockIdx.x / NSHARD;
  const int r = static_cast<int>(blockIdx.x % NSHARD);
  const int nchunks = (r == NSHARD - 1) ? LAST_CHUNKS : SHARD_CHUNKS;
  const bool f32 = P.grad_f32 != 0;
  char* const gshard = P.grad + (row * P.grad_stride + static_cast<int64_t>(r) * SW) * (f32 ? 4 : 2);

  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const int t = P.target[row];
  const rlk_row_stats st = P.stats[row];
  GradCoeffs m = grad_coeffs(st, tau, P.g_full ? P.g_full[row] : 0.0f,
                             P.g_restr ? P.g_restr[row] : 0.0f);
  if (m.mode != GRAD_VALUES) {          // zero or NaN rows need no logits
    write_grad_shard(nullptr, false, nchunks, r * SW, t, m, gshard, f32);
    return;
  }
  const uint32_t bar = smem_addr(&S.bar_load);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = static_cast<uint32_t>(nchunks) * 16u;
    mbar_arrive_expect_tx(bar, bytes);
    const uint64_t pol = evict_first_policy();
    const uint32_t piece = bytes / TMA_PIECES;
    const char* src = reinterpret_cast<const char*>(P.logits + row * P.stride + static_cast<int64_t>(r) * SW);
    const uint32_t dst = smem_addr(S.shard);
#pragma unroll
    for (int i = 0; i < TMA_PIECES; ++i) bulk_load(dst + i * piece, src + i * piece, piece, bar, pol);
  }
  __syncthreads();
  if (!mbar_wait_bounded(bar)) {
    mbar_wait_bounded(bar);             // give copies in flight a second bounded chance to land
    m = nan_coeffs();
  }
  write_grad_shard(S.shard, false, nchunks, r * SW, t, m, gshard, f32);
}

}  // namespace rlk

using namespace rlk;

extern "C" {

rlk_status rlk_logp_backward_saved(const rlk_logp_args* args, const rlk_row_stats* stats,
                                   const float* grad_full, const float* grad_restr,
                                   void* grad_logits, int64_t grad_row_stride, int32_t grad_dtype,
                                   void* stream) {
  rlk_status s = check_args(args, false);
  if (s != RLK_OK || args->T == 0) return s;
  if (!stats) return fail(RLK_EINVAL, "stats is NULL");
  if (!aligned(stats, 16)) return fail(RLK_EALIGN, "stats is not 16-byte aligned");
  if ((s = check_grad_args(grad_full, grad_restr, grad_logits, grad_row_stride, grad_dtype)) != RLK_OK)
    return s;
  GParams P;
  memset(&P, 0, sizeof(P));
  P.logits = static_cast<const uint16_t*>(args->logits);
  P.stride = args->row_stride;
  P.target = args->target;
  P.tau_arr = args->temperature;
  P.tau_s = args->temperature_scalar;
  P.stats = stats;
  P.g_full = grad_full;
  P.g_restr = grad_restr;
  P.grad = static_cast<char*>(grad_logits);
  P.grad_stride = grad_row_stride;
  P.grad_f32 = grad_dtype == RLK_GRAD_F32 ? 1 : 0;

  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(grad_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(GradSmem)));
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  grad_kernel<<<static_cast<unsigned>(args->T * NSHARD), NTHR, sizeof(GradSmem),
                static_cast<cudaStream_t>(stream)>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

}  // extern "C"
