// rlk_noalloc.cu -- the sampler for callers that cannot allocate device memory.
//
// rlk_sample needs 16 bytes of device scratch per row, which its caller
// normally provides.  Some callers have no way to provide it at call time:
// code whose device memory is owned by a framework allocator or by a fixed
// memory plan (an inference-engine plugin at enqueue time, a serving loop with
// a pre-reserved budget), where a cudaMalloc would bypass the plan, may
// synchronise the device and can fail in the middle of a run.  For them this
// file keeps the scratch in a fixed array in device memory that is part of
// the library itself: it costs RLK_SAMPLE_NOALLOC_MAX_ROWS x 16 bytes on every
// GPU that loads the library, for as long as the process runs, and nothing
// is allocated per call.

#include <cuda_runtime.h>
#include <stdint.h>

#include "rlk_logp.h"
#include "rlk_host.h"

namespace rlk {

// The draw's per-row records for up to RLK_SAMPLE_NOALLOC_MAX_ROWS rows.  In
// host code this name only stands for the array: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_sample_scratch[RLK_SAMPLE_NOALLOC_MAX_ROWS * 16];

// The scratch array's device address on the current device.  It is looked
// up on every call rather than cached: the lookup is a host-side table read
// (no stream work), and a cached address would go stale if the device's
// primary context were reset and the library's module loaded again.
rlk_status scratch_on_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_sample_scratch);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  *out = p;
  return RLK_OK;
}

}  // namespace rlk

using namespace rlk;

extern "C" {

rlk_status rlk_sample_noalloc(const rlk_logp_args* args, unsigned long long seed,
                              const unsigned long long* counter, const uint32_t* uniform,
                              int32_t* out_token, float* out_restr, float* out_full,
                              int32_t* out_support, void* stream) {
  if (args && args->T > RLK_SAMPLE_NOALLOC_MAX_ROWS)
    return fail(RLK_EINVAL, "T = %lld exceeds the %d rows of rlk_sample_noalloc's built-in scratch; "
                "split the batch or call rlk_sample with a workspace",
                (long long)args->T, RLK_SAMPLE_NOALLOC_MAX_ROWS);
  if (!args || args->T <= 0)                  // validation and the empty batch, as rlk_sample
    return sample_impl(args, seed, counter, uniform, out_token, out_restr, out_full, out_support,
                       nullptr, nullptr, stream);
  void* scratch = nullptr;
  rlk_status s = scratch_on_current_device(&scratch);
  if (s != RLK_OK) return s;
  // the records only: every row is drawn by re-reading its shards (no chunk bitmaps)
  return sample_impl(args, seed, counter, uniform, out_token, out_restr, out_full, out_support,
                     scratch, nullptr, stream);
}

}  // extern "C"
