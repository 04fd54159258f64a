// rlk_linear.cu -- full-vocabulary logprob straight from the LM head.
//
// The KL reference side needs only the full logprob of each row's target
// ("Configurable H100 consistency runs", KL-reference paragraph: the
// reference is scaled over the whole vocabulary), so the logits need never be
// stored: the LM head GEMM x = h . W^T runs on the 5th-generation tensor
// cores and its epilogue reduces every 128-row x 256-column tile of logits to
// one (max, sum-exp) pair per row, summaries of fixed column tiles combined in
// a fixed vocabulary order afterwards.
//
// linear_kernel: persistent, one CTA per SM over (128-row, 256-column)
// output tiles.
//   warp 0, one thread   TMA producer: A (h, 128 x 64 bf16) and B (W, 256 x 64
//                        bf16) tiles, 128-byte swizzle, into a 4-stage ring;
//   warp 1               TMEM allocation (512 columns: two fp32 accumulators);
//                        one thread issues tcgen05.mma (M 128, N 256, K 16,
//                        bf16 in, fp32 accumulate) and commits each stage
//                        back to the producer, then the tile to the epilogue;
//   warps 4-7            epilogue: each thread owns one row (TMEM lane), reads
//                        its 256 fp32 logits 32 columns at a time and keeps an
//                        online (max, sum-exp) over the real columns.
// merge_lin_kernel: one warp per row folds the row's 596 tile summaries in a
// fixed tree and forms full = (x_t - M) / tau - ln Z.
//
// Every logit is accumulated over K in the same order whatever the batch, and
// every reduction has a fixed shape, so a row's result does not depend on T.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "rlk_logp.h"
#include "rlk_device.cuh"
#include "rlk_host.h"

namespace rlk {

constexpr int LM = 128;                     // rows per tile (TMEM lanes)
constexpr int LN = 256;                     // vocabulary columns per tile
constexpr int LK = 64;                      // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int LSTAGES = 4;
constexpr int NTILE = VPAD / LN;            // 596 vocabulary tiles
constexpr uint32_t A_BYTES = LM * LK * 2;   // 16 KB
constexpr uint32_t B_BYTES = LN * LK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int LIN_THREADS = 256;
constexpr uint32_t LIN_SMEM = LSTAGES * STAGE_BYTES + 1024 + 256;
static_assert(VPAD % LN == 0, "vocabulary tiles");
static_assert(LIN_SMEM <= 232448, "shared memory of one CTA");

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both
// K-major, N = 256 (N >> 3 at bit 17), M = 128 (M >> 4 at bit 24).
constexpr uint32_t LIN_IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                               (static_cast<uint32_t>(LN >> 3) << 17) |
                               (static_cast<uint32_t>(LM >> 4) << 24);

struct LinArgs {
  int64_t T;
  int mt;                                   // row tiles
  int nk;                                   // K stages (H / 64)
  const int32_t* target;
  const float* tau_arr;
  float tau_s;
  float2* ws_ml;                            // [T][NTILE] (max, sum-exp) of each tile
  float* ws_xt;                             // [T] the target's logit
  int32_t* err;
};

// ------------------------------------------------------------ PTX

__device__ __forceinline__ bool mbar_wait_parity_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_timer();
  while (!mbar_try(bar, parity)) {
    if (global_timer() - t0 > TIMEOUT_NS) return false;
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] . B[smem]^T, one elected thread
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(LIN_IDESC) : "memory");
}
// arrive on a barrier once every tcgen05 operation this thread issued is done
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}
// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle
// layout: start address >> 4 (bits 0-13), leading byte offset 16 B (unused by
// swizzled K-major tiles), stride byte offset 1024 B = 8 rows x 128 B (bits
// 32-45), descriptor version 1 (bit 46), layout 128-byte swizzle (2 at bit 61).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
// 32 TMEM lanes x 32 columns of 32-bit values: thread i of the warp gets lane
// (base lane + i), columns col .. col + 31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ------------------------------------------------------------ kernels

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Persistent: one CTA per SM walks the tiles tile = blockIdx.x + i * gridDim.x
// (row tiles fastest, so the CTAs running at one time share a vocabulary tile
// and its weight is read from HBM once).  The TMA ring runs on across tiles;
// two TMEM accumulators (columns 0-255 and 256-511) let the MMA thread fill
// one while the epilogue warps drain the other.
__global__ void __launch_bounds__(LIN_THREADS, 1)
linear_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
              const LinArgs P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;              // 1024-byte aligned ring
  const uint32_t bars = base + LSTAGES * STAGE_BYTES;
  const uint32_t full0 = bars, empty0 = bars + 8 * LSTAGES;
  const uint32_t accf0 = bars + 16 * LSTAGES, acce0 = accf0 + 16;   // accumulator full / empty, x2
  const uint32_t slot = acce0 + 16;                           // TMEM address written by the allocation
  uint32_t* slot_ptr = reinterpret_cast<uint32_t*>(smem_raw + (slot - raw));
  uint32_t* flag_ptr = slot_ptr + 1;                          // a wait gave up
  const int ntiles = P.mt * NTILE;

  if (tid == 0) {
    for (int s = 0; s < LSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4);                            // one arrival per epilogue warp
    }
    *flag_ptr = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;

  if (warp == 0 && lane == 0) {
    // ---- producer: every K stage of every tile of this CTA through the ring
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < ntiles && !*flag_ptr; tile += gridDim.x) {
      const int m_tile = tile % P.mt, n_tile = tile / P.mt;
      for (int kb = 0; kb < P.nk; ++kb, ++it) {
        const uint32_t s = it % LSTAGES;
        if (it >= LSTAGES && !mbar_wait_parity_bounded(empty0 + 8 * s, ((it / LSTAGES) - 1) & 1)) {
          *flag_ptr = 1u;
          break;
        }
        const uint32_t a = base + s * STAGE_BYTES, b = a + A_BYTES;
        mbar_arrive_expect_tx(full0 + 8 * s, STAGE_BYTES);
        tma_load_2d(a, &tmap_a, kb * LK, m_tile * LM, full0 + 8 * s);
        tma_load_2d(b, &tmap_b, kb * LK, n_tile * LN, full0 + 8 * s);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: tile j accumulates in buffer j & 1
    uint32_t it = 0, j = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
      const uint32_t buf = j & 1;
      if (j >= 2 && !mbar_wait_parity_bounded(acce0 + 8 * buf, ((j >> 1) - 1) & 1)) *flag_ptr = 1u;
      tc_fence_after();
      const uint32_t d = tmem + buf * 256;
      for (int kb = 0; kb < P.nk; ++kb, ++it) {
        const uint32_t s = it % LSTAGES;
        if (!*flag_ptr && !mbar_wait_parity_bounded(full0 + 8 * s, (it / LSTAGES) & 1)) *flag_ptr = 1u;
        if (*flag_ptr) continue;                              // keep the phase count, issue nothing
        tc_fence_after();
        const uint32_t a = base + s * STAGE_BYTES, b = a + A_BYTES;
        const uint64_t ad = sw128_desc(a), bd = sw128_desc(b);
#pragma unroll
        for (int k = 0; k < LK / 16; ++k)                     // +32 bytes along K: +2 in the address field
          umma_bf16(d, ad + 2 * k, bd + 2 * k, (kb | k) != 0 ? 1u : 0u);
        umma_commit(empty0 + 8 * s);
      }
      umma_commit(accf0 + 8 * buf);
    }
  } else if (warp >= 4) {
    // ---- epilogue: thread = row of the tile (TMEM lane)
    const int ew = warp - 4;
    uint32_t j = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
      const int m_tile = tile % P.mt, n_tile = tile / P.mt;
      const uint32_t buf = j & 1;
      const bool ok = mbar_wait_parity_bounded(accf0 + 8 * buf, (j >> 1) & 1);
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(m_tile) * LM + ew * 32 + lane;
      const bool live = row < P.T;
      const float tau = live ? (P.tau_arr ? P.tau_arr[row] : P.tau_s) : 1.0f;
      const float c = __fdiv_rn(LOG2E, tau);
      const int tcol = live ? P.target[row] - n_tile * LN : -1;
      float m = -INFINITY, l = 0.0f, xt = __int_as_float(0x7fc00000);
      const uint32_t trow = tmem + buf * 256 + (static_cast<uint32_t>(ew * 32) << 16);
#pragma unroll 1
      for (int ch = 0; ch < LN / 32; ++ch) {
        float v[32];
        tmem_ld32(trow + ch * 32, v);                         // warp-collective: every lane takes part
        if (ch == LN / 32 - 1) {                              // the accumulator is read: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce0 + 8 * buf);
        }
        const int col0 = n_tile * LN + ch * 32;
        float cmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          if (col0 + jj < VREAL) cmax = fmaxf(cmax, v[jj]);
          if (tcol == ch * 32 + jj) xt = v[jj];
        }
        if (cmax > m) {
          l = l * ex2((m - cmax) * c);
          m = cmax;
        }
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)
          if (col0 + jj < VREAL) l += ex2((v[jj] - m) * c);
      }
      if (live) {
        const bool good = ok && *flag_ptr == 0u;
        P.ws_ml[row * NTILE + n_tile] = good ? make_float2(m, l) : make_float2(__int_as_float(0x7fc00000), 0.0f);
        if (tcol >= 0 && tcol < LN) P.ws_xt[row] = xt;
        if (!good && P.err && n_tile == 0) atomicAdd(P.err, 1);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per row: fold the row's tile summaries (lane q takes tiles q, q + 32,
// ... in order; then a max and a butterfly sum over the lanes: a fixed tree).
__global__ void __launch_bounds__(128) merge_lin_kernel(const LinArgs P, float* out_full) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (row >= P.T) return;
  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const int t = P.target[row];
  if (!(tau > 0.0f && tau <= 3.402823466e38f) || t < 0 || t >= VREAL) {
    if (lane == 0) {
      out_full[row] = __int_as_float(0x7fc00000);
      if (P.err) atomicAdd(P.err, 1);
    }
    return;
  }
  const float c = __fdiv_rn(LOG2E, tau);
  const float2* ml = P.ws_ml + row * NTILE;
  float mq = -INFINITY;
  for (int q = lane; q < NTILE; q += 32) mq = fmaxf(mq, ml[q].x);
  float zq = 0.0f;
  for (int q = lane; q < NTILE; q += 32) {
    const float2 v = ml[q];
    if (v.x > -INFINITY) zq = fmaf(v.y, ex2((v.x - mq) * c), zq);
  }
  float M = mq;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float z = (mq > -INFINITY) ? zq * ex2((mq - M) * c) : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z = z + __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) out_full[row] = __fdiv_rn(P.ws_xt[row] - M, tau) - logf(z);
}

// ------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

rlk_status encode_tiled(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                        int64_t row_stride, uint32_t box_rows) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                           cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
      return fail(RLK_ECUDA, "cuTensorMapEncodeTiled is not available");
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(LK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RLK_ECUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return RLK_OK;
}

}  // namespace rlk

using namespace rlk;

extern "C" {

rlk_status rlk_linear_logp(const void* hidden, int64_t T, int64_t H, int64_t hidden_stride,
                           const void* weight, int64_t weight_stride, const int32_t* target,
                           const float* temperature, float temperature_scalar, float* out_full,
                           void* workspace, int32_t* err_count, void* stream) {
  if (T < 0 || T >= (int64_t(1) << 24)) return fail(RLK_EINVAL, "T = %lld out of range [0, 2^24)", (long long)T);
  if (T == 0) return RLK_OK;
  if (H < LK || H % LK != 0 || H > (int64_t(1) << 20))
    return fail(RLK_EINVAL, "H = %lld must be a positive multiple of %d (at most 2^20)", (long long)H, LK);
  if (!hidden || !weight) return fail(RLK_EINVAL, "hidden or weight is NULL");
  if (!aligned(hidden, 16) || !aligned(weight, 16)) return fail(RLK_EALIGN, "hidden and weight must be 16-byte aligned");
  if (hidden_stride < H || weight_stride < H)
    return fail(RLK_EINVAL, "row strides must be >= H");
  if ((hidden_stride * 2) % 16 != 0 || (weight_stride * 2) % 16 != 0)
    return fail(RLK_EALIGN, "row strides must be multiples of 8 elements");
  rlk_status s;
  if ((s = check_out(target, "target", true)) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  if (temperature) {
    if (!aligned(temperature, 4)) return fail(RLK_EALIGN, "temperature is not 4-byte aligned");
  } else if (!(temperature_scalar > 0.0f && temperature_scalar <= 3.402823466e38f)) {
    return fail(RLK_EINVAL, "temperature %g must be finite and > 0", (double)temperature_scalar);
  }
  if (!workspace) return fail(RLK_EINVAL, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(RLK_EALIGN, "workspace is not 16-byte aligned");
  if (err_count && !aligned(err_count, 4)) return fail(RLK_EALIGN, "err_count is not 4-byte aligned");

  CUtensorMap ta, tb;
  if ((s = encode_tiled(&ta, hidden, static_cast<uint64_t>(H), static_cast<uint64_t>(T), hidden_stride, LM)) != RLK_OK)
    return s;
  if ((s = encode_tiled(&tb, weight, static_cast<uint64_t>(H), static_cast<uint64_t>(VPAD), weight_stride, LN)) != RLK_OK)
    return s;
  LinArgs P;
  memset(&P, 0, sizeof(P));
  P.T = T;
  P.mt = static_cast<int>((T + LM - 1) / LM);
  P.nk = static_cast<int>(H / LK);
  P.target = target;
  P.tau_arr = temperature;
  P.tau_s = temperature_scalar;
  P.ws_ml = static_cast<float2*>(workspace);
  P.ws_xt = reinterpret_cast<float*>(static_cast<char*>(workspace) + static_cast<size_t>(T) * NTILE * 8);
  P.err = err_count;

  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(LIN_SMEM));
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  const int64_t ntiles = static_cast<int64_t>(P.mt) * NTILE;
  const unsigned grid = static_cast<unsigned>(ntiles < sms ? ntiles : sms);   // one CTA per SM
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  linear_kernel<<<grid, LIN_THREADS, LIN_SMEM, st>>>(ta, tb, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  merge_lin_kernel<<<static_cast<unsigned>((T + 3) / 4), 128, 0, st>>>(P, out_full);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

}  // extern "C"
