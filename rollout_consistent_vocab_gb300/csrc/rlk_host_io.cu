// rlk_host_io.cu -- the rlk_logp_kl step on inputs that live in host memory.
//
// On a GB300 the logits that a host holds reach the GPU over the host link,
// about 30 times slower than the passes read HBM, so the step from host
// memory is bound by that link.  This entry point splits the rows into
// ranges: range c + 1 is copied in on a second stream while the passes over
// range c run, and each range's results go back on the compute stream, so
// the passes hide behind the copies.  Only the 151936 real columns of a row
// are copied (the passes never read the padded ones).  The passes are
// rlk_logp_kl itself, on the device copies of a range; a row's results do
// not depend on the rows around it ("H100 rollout context parallelism":
// the same token must score the same whatever the batch), so they are
// bit-identical to one rlk_logp_kl call over the whole batch.

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "rlk_logp.h"
#include "rlk_host.h"

namespace rlk {
namespace {

constexpr size_t LOGITS_ROW_BYTES = static_cast<size_t>(RLK_VOCAB_PADDED) * 2u;
constexpr size_t REAL_ROW_BYTES = static_cast<size_t>(RLK_VOCAB_REAL) * 2u;
static_assert(REAL_ROW_BYTES % 16 == 0, "a row's real columns are whole 16-byte pieces");

size_t round256(size_t v) { return (v + 255u) & ~static_cast<size_t>(255u); }

// The device workspace: both logits tensors at the padded row length, the
// targets, then the five outputs, each region 256-byte aligned.
struct Workspace {
  uint16_t* logits;
  uint16_t* ref;
  int32_t* target;
  float* full;
  float* restr;
  int32_t* support;
  float* full_ref;
  float* kl;
};

Workspace carve(void* base, int64_t T) {
  char* p = static_cast<char*>(base);
  const size_t tensor = static_cast<size_t>(T) * LOGITS_ROW_BYTES;   // a multiple of 256
  const size_t vec = round256(static_cast<size_t>(T) * 4u);
  Workspace w;
  w.logits = reinterpret_cast<uint16_t*>(p);
  w.ref = reinterpret_cast<uint16_t*>(p + tensor);
  char* q = p + 2 * tensor;
  w.target = reinterpret_cast<int32_t*>(q);
  w.full = reinterpret_cast<float*>(q + vec);
  w.restr = reinterpret_cast<float*>(q + 2 * vec);
  w.support = reinterpret_cast<int32_t*>(q + 3 * vec);
  w.full_ref = reinterpret_cast<float*>(q + 4 * vec);
  w.kl = reinterpret_cast<float*>(q + 5 * vec);
  return w;
}

rlk_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RLK_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The events of one call, released on every return path (an event still
// pending is released when it completes).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t add(cudaEvent_t* out) {
    cudaEvent_t e = nullptr;
    const cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r == cudaSuccess) {
      ev.push_back(e);
      *out = e;
    }
    return r;
  }
};

}  // namespace
}  // namespace rlk

using namespace rlk;

static_assert(RLK_LOGP_KL_HOST_WORKSPACE_BYTES(3) ==
                  3u * 2u * (size_t)RLK_VOCAB_PADDED * 2u + 6u * 256u,
              "the header's workspace size matches the carve");

extern "C" rlk_status rlk_logp_kl_host(const rlk_logp_args* policy, const void* ref_logits,
                                       int64_t ref_row_stride, float* out_full, float* out_restr,
                                       int32_t* out_support, float* out_full_ref, float* out_kl,
                                       void* workspace, int32_t chunks, void* stream,
                                       void* copy_stream) {
  // ---- every argument check before the first CUDA call
  if (!policy) return fail(RLK_EINVAL, "args is NULL");
  const int64_t T = policy->T;
  if (T < 0) return fail(RLK_EINVAL, "T = %lld < 0", (long long)T);
  if (T >= (int64_t(1) << 27))
    return fail(RLK_EINVAL, "T = %lld: at most 2^27 - 1 rows per rlk_logp_kl_host call", (long long)T);
  if (policy->vocab_real != RLK_VOCAB_REAL || policy->vocab_padded != RLK_VOCAB_PADDED)
    return fail(RLK_EINVAL, "vocab sizes must be %d/%d, got %d/%d", RLK_VOCAB_REAL, RLK_VOCAB_PADDED,
                policy->vocab_real, policy->vocab_padded);
  if (T == 0) return RLK_OK;
  if (!policy->logits) return fail(RLK_EINVAL, "logits is NULL");
  if (policy->row_stride < RLK_VOCAB_PADDED)
    return fail(RLK_EINVAL, "logits row_stride %lld < %d", (long long)policy->row_stride, RLK_VOCAB_PADDED);
  if (!policy->target) return fail(RLK_EINVAL, "target is NULL");
  if (!ref_logits) return fail(RLK_EINVAL, "ref_logits is NULL");
  if (ref_row_stride < RLK_VOCAB_PADDED)
    return fail(RLK_EINVAL, "ref_logits row_stride %lld < %d", (long long)ref_row_stride, RLK_VOCAB_PADDED);
  rlk_status s;
  if ((s = check_tau(policy->temperature, policy->temperature_scalar)) != RLK_OK) return s;
  if ((s = check_top_p(policy->top_p, policy->top_p_scalar)) != RLK_OK) return s;
  if ((s = check_top_k(policy->top_k, policy->top_k_scalar)) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  if ((s = check_out(out_full_ref, "out_full_ref", true)) != RLK_OK) return s;
  if ((s = check_out(out_kl, "out_kl", true)) != RLK_OK) return s;
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  if (!workspace) return fail(RLK_EINVAL, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(RLK_EALIGN, "workspace is not 256-byte aligned");
  if (chunks < 1) return fail(RLK_EINVAL, "chunks = %d < 1", chunks);

  // at most T ranges, and at most RLK_KL_HOST_MAX_CHUNKS (each range costs an event)
  int64_t nch = chunks < T ? chunks : T;
  if (nch > RLK_KL_HOST_MAX_CHUNKS) nch = RLK_KL_HOST_MAX_CHUNKS;
  const Workspace w = carve(workspace, T);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = copy_stream ? static_cast<cudaStream_t>(copy_stream) : st;
  const bool two = cs != st;
  const char* hx = static_cast<const char*>(policy->logits);
  const char* hr = static_cast<const char*>(ref_logits);
  const size_t hx_pitch = static_cast<size_t>(policy->row_stride) * 2u;
  const size_t hr_pitch = static_cast<size_t>(ref_row_stride) * 2u;

  Events events;
  cudaError_t e;
  if (two) {
    // the first copies wait for the work already queued on `stream` (an
    // earlier call's passes may still read this workspace)
    cudaEvent_t start;
    if ((e = events.add(&start)) != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
    if ((e = cudaEventRecord(start, st)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if ((e = cudaStreamWaitEvent(cs, start, 0)) != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t a = c * T / nch, b = (c + 1) * T / nch, rows = b - a;
    // ---- the range's inputs in, on the copy stream
    e = cudaMemcpy2DAsync(w.logits + a * RLK_VOCAB_PADDED, LOGITS_ROW_BYTES, hx + a * hx_pitch, hx_pitch,
                          REAL_ROW_BYTES, static_cast<size_t>(rows), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(w.ref + a * RLK_VOCAB_PADDED, LOGITS_ROW_BYTES, hr + a * hr_pitch, hr_pitch,
                            REAL_ROW_BYTES, static_cast<size_t>(rows), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(w.target + a, policy->target + a, static_cast<size_t>(rows) * 4u,
                          cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    if (two) {
      cudaEvent_t in;
      if ((e = events.add(&in)) != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
      if ((e = cudaEventRecord(in, cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
      if ((e = cudaStreamWaitEvent(st, in, 0)) != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    // ---- the passes over the range, on the compute stream
    rlk_logp_args d = *policy;
    d.logits = w.logits + a * RLK_VOCAB_PADDED;
    d.row_stride = RLK_VOCAB_PADDED;
    d.T = rows;
    d.target = w.target + a;
    d.temperature = policy->temperature ? policy->temperature + a : nullptr;
    d.top_p = policy->top_p ? policy->top_p + a : nullptr;
    d.top_k = policy->top_k ? policy->top_k + a : nullptr;
    s = rlk_logp_kl(&d, w.ref + a * RLK_VOCAB_PADDED, RLK_VOCAB_PADDED, w.full + a,
                    out_restr ? w.restr + a : nullptr, out_support ? w.support + a : nullptr,
                    w.full_ref + a, w.kl + a, st);
    if (s != RLK_OK) return s;
    // ---- its results out, behind the passes on the same stream
    const size_t nb = static_cast<size_t>(rows) * 4u;
    e = cudaMemcpyAsync(out_full + a, w.full + a, nb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && out_restr)
      e = cudaMemcpyAsync(out_restr + a, w.restr + a, nb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && out_support)
      e = cudaMemcpyAsync(out_support + a, w.support + a, nb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(out_full_ref + a, w.full_ref + a, nb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out_kl + a, w.kl + a, nb, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
  }
  return RLK_OK;
}
