// rlk_linear.cu -- full and restricted logprob straight from the LM head.
//
// The KL reference side needs only the full logprob of each row's target
// ("Configurable H100 consistency runs", KL-reference paragraph: the
// reference is scaled over the whole vocabulary), so the logits need never be
// stored: the LM head GEMM x = h . W^T runs on the 5th-generation tensor
// cores and its epilogue reduces every 128-row x 256-column tile of logits to
// one (max, sum-exp) pair per row, summaries of fixed column tiles combined in
// a fixed vocabulary order afterwards.
//
// linear_kernel<EPI>: persistent, one CTA per SM over (128-row, 256-column)
// output tiles.
//   warp 0, one thread   TMA producer: A (h, 128 x 64 bf16) and B (W, 256 x 64
//                        bf16) tiles, 128-byte swizzle, into a 4-stage ring;
//   warp 1               TMEM allocation (512 columns: two fp32 accumulators);
//                        one thread issues tcgen05.mma (M 128, N 256, K 16,
//                        bf16 in, fp32 accumulate) and commits each stage
//                        back to the producer, then the tile to the epilogue;
//   warps 4-7            epilogue: each thread owns one row (TMEM lane), reads
//                        its 256 fp32 logits 32 columns at a time and
//                        EPI_SUMMARY: keeps an online (max, sum-exp) over the
//                          real columns (EPI_SUMMARY_TOP8: and the 8 largest
//                          logits of the tile, for the restricted side);
//                        EPI_WINDOW: histograms and lists the logits whose
//                          order key lies in its row's current window (the
//                          restricted side below).
// merge_lin_kernel: one warp per row folds the row's 596 tile summaries in a
// fixed tree and forms full = (x_t - M) / tau - ln Z.
//
// The policy side keeps its top-k-then-top-p support (same paragraph), which
// needs the row's k-th largest logit and its nucleus threshold.  Without the
// logits in memory these are found by exact radix selection over the fp32
// order keys, each round recomputing the GEMM for the row tiles that still
// have an unresolved row (rlk_linear_logp_pair below).
//
// Every logit is accumulated over K in the same order whatever the batch, and
// every reduction has a fixed shape (or is an exact integer sum), so a row's
// results do not depend on T.

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

enum : int { EPI_SUMMARY = 0, EPI_WINDOW = 1, EPI_SUMMARY_TOP8 = 2 };
constexpr int TOPR = 8;                     // largest logits kept per (row, vocabulary tile)

// ---- restricted side: exact selection over fp32 order keys
constexpr int NB = 1024;                    // histogram buckets of a window
constexpr int LIST_CAP = 4096;              // keys listed per row and round
constexpr int PAIR_ROUNDS = 12;             // window rounds launched per call
constexpr uint32_t KEY_BOTTOM = 0x007FFFFFu;   // order key of -inf; smaller keys are NaN patterns
enum : uint32_t { WIN_IDLE = 0, WIN_KEY = 1, WIN_VALUE = 2 };
// mode bit: every logit of the window is already listed (from the first
// pass's per-tile top logits), so the next round needs no GEMM for the row
constexpr uint32_t WIN_LISTED = 0x100u;
constexpr uint32_t LIST_FAILED = 0x80000000u;   // listn bit: a histogram round lost a tile

// Order key of an fp32 value: unsigned order equals numeric order for
// non-NaN values; -0 shares the key of +0.
__device__ __forceinline__ uint32_t key32(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key32_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// Fixed-point mass exp((x - M) / tau) * 2^44 of one logit, rounded to the
// nearest integer; the histogram pass and the selection evaluate it with the
// same operations, so equal logits have equal masses.
__device__ __forceinline__ unsigned long long lmass(float x, float M, float c) {
  return fx_round(__fmul_rn(ex2(__fmul_rn(__fsub_rn(x, M), c)), FX_SCALE));
}

// A row's window for the next histogram round: the logits whose order key
// lies in [wlo, whi], bucketed either by key, (whi - key) >> shift, or
// linearly in value, min(NB - 1, floor((va - x) * vg)); bucket 0 is the top.
struct LinWin {
  uint32_t mode;                            // WIN_IDLE (resolved), WIN_KEY, WIN_VALUE
  uint32_t wlo, whi;
  uint32_t shift;
  float va, vg;
  float M, c;                               // row maximum, log2(e) / tau
};
static_assert(sizeof(LinWin) == 32, "LinWin layout");

__device__ __forceinline__ int value_bucket(float x, float va, float vg) {
  const float d = __fmul_rn(__fsub_rn(va, x), vg);
  return d < static_cast<float>(NB - 1) ? static_cast<int>(d) : NB - 1;
}
__device__ __forceinline__ int win_bucket(const LinWin& w, float x, uint32_t K) {
  return w.mode == WIN_KEY ? static_cast<int>((w.whi - K) >> w.shift) : value_bucket(x, w.va, w.vg);
}

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
  float* ws_top;                            // [T][NTILE][TOPR] EPI_SUMMARY_TOP8: descending
  // EPI_WINDOW rounds
  const uint32_t* np;                       // number of listed row tiles
  const int32_t* mlist;                     // row tiles with an unresolved row
  const LinWin* win;                        // [T]
  uint32_t* hcnt;                           // [T][NB] counts per bucket
  unsigned long long* hmass;                // [T][NB] fixed-point masses per bucket
  uint32_t* list;                           // [T][LIST_CAP] order keys in the window
  uint32_t* listn;                          // [T] keys in the window (may exceed LIST_CAP)
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
// one while the epilogue warps drain the other.  EPI_WINDOW walks only the row
// tiles listed in mlist[0 .. *np) (every vocabulary tile of each).
template <int EPI>
__global__ void __launch_bounds__(LIN_THREADS, 1)
linear_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
              const LinArgs P) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nm = EPI != EPI_WINDOW ? P.mt : static_cast<int>(*P.np);
  if (nm == 0) return;                                        // uniform: nothing allocated yet
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;              // 1024-byte aligned ring
  const uint32_t bars = base + LSTAGES * STAGE_BYTES;
  const uint32_t full0 = bars, empty0 = bars + 8 * LSTAGES;
  const uint32_t accf0 = bars + 16 * LSTAGES, acce0 = accf0 + 16;   // accumulator full / empty, x2
  const uint32_t slot = acce0 + 16;                           // TMEM address written by the allocation
  uint32_t* slot_ptr = reinterpret_cast<uint32_t*>(smem_raw + (slot - raw));
  uint32_t* flag_ptr = slot_ptr + 1;                          // a wait gave up
  const int ntiles = nm * NTILE;
  auto row_tile = [&](int tile) { return EPI != EPI_WINDOW ? tile % nm : P.mlist[tile % nm]; };

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
      const int m_tile = row_tile(tile), n_tile = tile / nm;
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
      const int m_tile = row_tile(tile), n_tile = tile / nm;
      const uint32_t buf = j & 1;
      const bool ok = mbar_wait_parity_bounded(accf0 + 8 * buf, (j >> 1) & 1);
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(m_tile) * LM + ew * 32 + lane;
      const bool live = row < P.T;
      const uint32_t trow = tmem + buf * 256 + (static_cast<uint32_t>(ew * 32) << 16);
      if constexpr (EPI != EPI_WINDOW) {
        const float tau = live ? (P.tau_arr ? P.tau_arr[row] : P.tau_s) : 1.0f;
        const float c = __fdiv_rn(LOG2E, tau);
        const int tcol = live ? P.target[row] - n_tile * LN : -1;
        float m = -INFINITY, l = 0.0f, xt = __int_as_float(0x7fc00000);
        float top[TOPR];                                      // descending; NaN never enters
#pragma unroll
        for (int q = 0; q < TOPR; ++q) top[q] = -INFINITY;
#pragma unroll 1
        for (int ch = 0; ch < LN / 32; ++ch) {
          float v[32];
          tmem_ld32(trow + ch * 32, v);                       // warp-collective: every lane takes part
          if (ch == LN / 32 - 1) {                            // the accumulator is read: hand it back
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
          if constexpr (EPI == EPI_SUMMARY_TOP8) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              if (col0 + jj < VREAL && v[jj] > top[TOPR - 1]) {
                top[TOPR - 1] = v[jj];
#pragma unroll
                for (int q = TOPR - 1; q > 0; --q) {        // one bubble step keeps the order
                  const float hi = fmaxf(top[q - 1], top[q]), lo = fminf(top[q - 1], top[q]);
                  top[q - 1] = hi;
                  top[q] = lo;
                }
              }
            }
          }
        }
        if (live) {
          const bool good = ok && *flag_ptr == 0u;
          P.ws_ml[row * NTILE + n_tile] = good ? make_float2(m, l) : make_float2(__int_as_float(0x7fc00000), 0.0f);
          if (tcol >= 0 && tcol < LN) P.ws_xt[row] = xt;
          if (!good && P.err && n_tile == 0) atomicAdd(P.err, 1);
          if constexpr (EPI == EPI_SUMMARY_TOP8) {
            float4* dst = reinterpret_cast<float4*>(P.ws_top + (row * NTILE + n_tile) * TOPR);
            dst[0] = make_float4(top[0], top[1], top[2], top[3]);
            dst[1] = make_float4(top[4], top[5], top[6], top[7]);
          }
        }
      } else {
        // histogram and list the logits of the row's window (exact integer
        // sums: the order in which tiles arrive does not matter)
        LinWin w;
        w.mode = WIN_IDLE;
        if (live) w = P.win[row];
        const bool want = w.mode != WIN_IDLE && !(w.mode & WIN_LISTED);
        const bool act = want && ok && *flag_ptr == 0u;
        uint32_t* cnt = P.hcnt + row * NB;
        unsigned long long* mass = P.hmass + row * NB;
        uint32_t* lst = P.list + row * LIST_CAP;
#pragma unroll 1
        for (int ch = 0; ch < LN / 32; ++ch) {
          float v[32];
          tmem_ld32(trow + ch * 32, v);
          if (ch == LN / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * buf);
          }
          if (!act) continue;
          const int col0 = n_tile * LN + ch * 32;
          uint32_t in = 0;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const uint32_t K = key32(v[jj]);
            if (col0 + jj < VREAL && K >= w.wlo && K <= w.whi) in |= 1u << jj;
          }
          if (!in) continue;
          uint32_t at = atomicAdd(P.listn + row, static_cast<uint32_t>(__popc(in)));
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            if (!((in >> jj) & 1u)) continue;
            const uint32_t K = key32(v[jj]);
            const int b = win_bucket(w, v[jj], K);
            atomicAdd(cnt + b, 1u);
            atomicAdd(mass + b, lmass(v[jj], w.M, w.c));
            if (at < LIST_CAP) lst[at] = K;
            ++at;
          }
        }
        // a wait gave up: the row's counts are incomplete; the selection fails it
        if (live && want && !act) atomicOr(P.listn + row, LIST_FAILED);
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

// Fold a row's tile summaries (lane q takes tiles q, q + 32, ... in order;
// then a max and a butterfly sum over the lanes: a fixed tree).  Every lane
// returns the row maximum M and Z = sum_j exp2((x_j - M) c).
__device__ __forceinline__ void lin_merge(const LinArgs& P, int64_t row, int lane, float c, float& M, float& z) {
  const float2* ml = P.ws_ml + row * NTILE;
  float mq = -INFINITY;
  for (int q = lane; q < NTILE; q += 32) mq = fmaxf(mq, ml[q].x);
  float zq = 0.0f;
  for (int q = lane; q < NTILE; q += 32) {
    const float2 v = ml[q];
    if (!(v.x == -INFINITY)) zq = fmaf(v.y, ex2((v.x - mq) * c), zq);   // a NaN summary poisons Z
  }
  M = mq;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  z = (mq > -INFINITY) ? zq * ex2((mq - M) * c) : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z = z + __shfl_xor_sync(0xffffffffu, z, o);
}

__device__ __forceinline__ bool tau_ok(float tau) { return tau > 0.0f && tau <= 3.402823466e38f; }

// One warp per row: full = (x_t - M) / tau - ln Z.
__global__ void __launch_bounds__(128) merge_lin_kernel(const LinArgs P, float* out_full) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (row >= P.T) return;
  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const int t = P.target[row];
  if (!tau_ok(tau) || t < 0 || t >= VREAL) {
    if (lane == 0) {
      out_full[row] = __int_as_float(0x7fc00000);
      if (P.err) atomicAdd(P.err, 1);
    }
    return;
  }
  const float c = __fdiv_rn(LOG2E, tau);
  float M, z;
  lin_merge(P, row, lane, c, M, z);
  if (lane == 0) out_full[row] = __fdiv_rn(P.ws_xt[row] - M, tau) - logf(z);
}

// ------------------------------------------------------------ restricted side
//
// The support S of a row is found without its logits in memory, by exact
// selection over the fp32 order keys (the same top-k-then-top-p definition
// as for stored logits, "Configurable H100 consistency runs", sampling-flags
// paragraph, on the GEMM's fp32 logits):
//   stage 0 (top-k on): the k-th largest key v_k; S_k = keys >= v_k, Z_k its
//     fixed-point mass;
//   stage 1 (top-p on): the nucleus key v*: the first key from the top at
//     which the mass of the keys above it is < T = ceil(p Z_k) and the mass
//     through it is >= T (v_k if never reached); S = keys >= v*.
// A search narrows a window of keys [wlo, whi] round by round.  Each round
// recomputes the GEMM for the row tiles that hold an unresolved row; its
// epilogue adds every in-window logit to the row's bucket (count, mass) and
// appends its key to the row's list.  pair_round_kernel then either resolves
// the row from the list (every in-window key listed: sorted, exact) or moves
// the window to the bucket where the count or mass target is crossed,
// carrying the counts and masses above it.  The first window of a search is
// bounded a priori: for top-k by the k-th largest of the logits the first
// pass kept (the 8 largest of every 256-column tile: k distinct tokens reach
// it), for top-p alone by the mass bound (a token of mass <= (1 - p) Z / V
// leaves at least p Z above it), halved for margin.  When every tile's 8th
// kept logit lies below that window, the kept logits hold the whole window:
// the row is listed from them and its first round needs no GEMM.

// Per-row selection state.
struct LinSel {
  unsigned long long carry_m;               // fixed-point mass of the keys above the window
  unsigned long long T;                     // nucleus target ceil(p Z_k) (stage 1)
  uint32_t carry_c;                         // keys above the window
  uint32_t stage;                           // 0: k-th largest key; 1: nucleus key
  int32_t k;                                // top-k (stage 0)
  float p;                                  // top-p; 1 = off
  uint32_t floor_key;                       // lowest key the nucleus may keep (v_k, or KEY_BOTTOM)
  uint32_t top_key;                         // key of the row maximum
  uint32_t kt;                              // key of the target's logit
  float d;                                  // (x_t - M) / tau
  uint32_t pad[4];
};
static_assert(sizeof(LinSel) == 64, "LinSel layout");

struct PairArgs {
  int64_t T;
  const float* top_p;
  float top_p_s;
  const int32_t* top_k;
  int32_t top_k_s;
  float* out_full;
  float* out_restr;
  int32_t* out_support;
  int32_t* err;
  LinWin* win;                              // [T]
  LinSel* sel;                              // [T]
  uint32_t* hcnt;                           // [T][NB]
  unsigned long long* hmass;                // [T][NB]
  uint32_t* list;                           // [T][LIST_CAP]
  uint32_t* listn;                          // [T]
  int32_t* rowlist;                         // [2][T] rows of a round (round parity)
  int32_t* mlist;                           // [2][row tiles] row tiles of a round needing the GEMM
  uint32_t* mflag;                          // [PAIR_ROUNDS][row tiles] a tile is listed for the round
  uint32_t* counters;                       // [PAIR_ROUNDS][2]: rows, row tiles listed per round
  int mt;
};

constexpr int RT = 256;                     // threads of pair_round_kernel
constexpr uint32_t ROUND_SMEM = LIST_CAP * 4 + LIST_CAP * 8;
static_assert(NB <= LIST_CAP, "bucket counts reuse the key array");

__device__ __forceinline__ void key_window(LinWin& w, uint32_t lo, uint32_t hi) {
  w.mode = WIN_KEY;
  w.wlo = lo;
  w.whi = hi;
  const uint32_t r = hi - lo;
  const int bits = r ? 32 - __clz(r) : 0;
  w.shift = bits > 10 ? static_cast<uint32_t>(bits - 10) : 0u;     // (whi - wlo) >> shift < NB = 2^10
}

// The first window of a search, [lo, top]: linear in value when the span is
// a usable float (buckets of equal width in logit), by key otherwise.
__device__ __forceinline__ void open_window(LinWin& w, uint32_t lo, uint32_t top) {
  const float span = __fsub_rn(w.M, key32_value(lo));
  const float vg = span > 0.0f ? __fdiv_rn(static_cast<float>(NB), span) : 0.0f;
  if (lo > KEY_BOTTOM && span >= 1e-30f && span <= 1e38f && vg > 0.0f && vg <= 1e38f) {
    w.mode = WIN_VALUE;
    w.wlo = lo;
    w.whi = top;
    w.shift = 0u;
    w.va = w.M;
    w.vg = vg;
  } else {
    key_window(w, lo, top);
  }
}

// Put an unresolved row on round r's list, and its row tile on the round's
// GEMM list unless the row's window is already listed (counters and flags
// are cleared before the first pass).
__device__ __forceinline__ void enqueue_row(const PairArgs& A, int r, int64_t row, bool gemm) {
  if (r >= PAIR_ROUNDS) return;
  A.rowlist[(r & 1) * A.T + atomicAdd(A.counters + 2 * r, 1u)] = static_cast<int32_t>(row);
  const int m = static_cast<int>(row / LM);
  if (gemm && atomicExch(A.mflag + r * A.mt + m, 1u) == 0u)
    A.mlist[(r & 1) * A.mt + atomicAdd(A.counters + 2 * r + 1, 1u)] = m;
}


// Inclusive prefix sums, in place, of n masses (and counts, if cc) in
// shared memory: each thread sums a contiguous run, then a block scan.
__device__ void block_prefix(unsigned long long* cm, uint32_t* cc, int n, unsigned long long* wm, uint32_t* wc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + RT - 1) / RT;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  unsigned long long sm = 0ull;
  uint32_t sc = 0u;
  for (int i = i0; i < i1; ++i) {
    sm += cm[i];
    if (cc) sc += cc[i];
  }
  unsigned long long im = sm;
  uint32_t ic = sc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long tm = __shfl_up_sync(0xffffffffu, im, o);
    const uint32_t tc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) {
      im += tm;
      ic += tc;
    }
  }
  if (lane == 31) {
    wm[warp] = im;
    wc[warp] = ic;
  }
  __syncthreads();
  unsigned long long bm = im - sm;
  uint32_t bc = ic - sc;
  for (int w = 0; w < warp; ++w) {
    bm += wm[w];
    bc += wc[w];
  }
  for (int i = i0; i < i1; ++i) {
    bm += cm[i];
    cm[i] = bm;
    if (cc) {
      bc += cc[i];
      cc[i] = bc;
    }
  }
  __syncthreads();
}

// Bitonic sort of n <= LIST_CAP keys into descending order (padded with 0,
// which sorts below every key of a real logit).
__device__ void sort_desc(uint32_t* keys, int n) {
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  for (int i = n + threadIdx.x; i < p2; i += RT) keys[i] = 0u;
  __syncthreads();
  for (int k = 2; k <= p2; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < p2; i += RT) {
        const int ix = i ^ j;
        if (ix > i) {
          const uint32_t a = keys[i], b = keys[ix];
          if (((i & k) == 0) ? a < b : a > b) {
            keys[i] = b;
            keys[ix] = a;
          }
        }
      }
      __syncthreads();
    }
}

// The window's contents in descending key order: listed keys (one each) or
// histogram buckets, with inclusive counts and masses.
struct Items {
  bool list;
  int n;
  const uint32_t* keys;                     // list: sorted keys
  const uint32_t* cc;                       // buckets: inclusive counts
  const unsigned long long* cm;             // inclusive masses
  __device__ uint32_t count_at(int i) const { return list ? static_cast<uint32_t>(i + 1) : cc[i]; }
};

__device__ int first_count(const Items& it, uint32_t need) {      // count_at(n - 1) >= need
  int lo = 0, hi = it.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (it.count_at(mid) >= need) hi = mid; else lo = mid + 1;
  }
  return lo;
}
__device__ int first_mass(const Items& it, unsigned long long tgt) {   // cm[n - 1] >= tgt
  int lo = 0, hi = it.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (it.cm[mid] >= tgt) hi = mid; else lo = mid + 1;
  }
  return lo;
}
// last index of a descending key list whose key is >= K (-1: none)
__device__ int last_ge(const uint32_t* keys, int n, uint32_t K) {
  int lo = -1, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (keys[mid] >= K) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Keys of bucket b (non-empty) of a window.
__device__ void bucket_range(const LinWin& w, int b, uint32_t& lo, uint32_t& hi) {
  if (w.mode == WIN_KEY) {
    hi = w.whi - (static_cast<uint32_t>(b) << w.shift);
    const uint32_t span = (1u << w.shift) - 1u;
    lo = (hi - w.wlo > span) ? hi - span : w.wlo;
    return;
  }
  // value buckets fall as the key rises: bucket b is the keys from the
  // smallest with bucket <= b to the largest with bucket >= b
  uint32_t a = w.wlo, z = w.whi;
  while (a < z) {
    const uint32_t mid = a + (z - a + 1u) / 2u;
    if (value_bucket(key32_value(mid), w.va, w.vg) >= b) a = mid; else z = mid - 1u;
  }
  hi = a;
  a = w.wlo;
  z = w.whi;
  while (a < z) {
    const uint32_t mid = a + (z - a) / 2u;
    if (value_bucket(key32_value(mid), w.va, w.vg) <= b) z = mid; else a = mid + 1u;
  }
  lo = a;
}

// One thread: advance the row's search on this round's window contents.
__device__ void decide(const Items& it, LinWin& w, LinSel& s, int64_t row, const PairArgs& A) {
  const uint32_t tot_c = it.n ? it.count_at(it.n - 1) : 0u;
  const unsigned long long tot_m = it.n ? it.cm[it.n - 1] : 0ull;
  auto resolve = [&](uint32_t sup, unsigned long long zs, uint32_t min_key) {
    const float zf = __ull2float_rn(zs) * (1.0f / FX_SCALE);
    A.out_restr[row] = s.kt >= min_key ? s.d - logf(zf) : -INFINITY;
    if (A.out_support) A.out_support[row] = static_cast<int32_t>(sup);
    w.mode = WIN_IDLE;
  };
  auto fail = [&]() {
    A.out_restr[row] = __int_as_float(0x7fc00000);
    if (A.out_support) A.out_support[row] = -2;
    if (A.err) atomicAdd(A.err, 1);
    w.mode = WIN_IDLE;
  };
  auto range = [&](int i, uint32_t& lo, uint32_t& hi) {
    if (it.list) lo = hi = it.keys[i]; else bucket_range(w, i, lo, hi);
  };
  auto narrow = [&](int i, uint32_t lo, uint32_t hi) {
    if (i > 0) {
      s.carry_c += it.count_at(i - 1);
      s.carry_m += it.cm[i - 1];
    }
    key_window(w, lo, hi);
  };
  auto below = [&](uint32_t bottom) {       // the boundary lies under the window
    if (w.wlo <= bottom) { fail(); return; }
    s.carry_c += tot_c;
    s.carry_m += tot_m;
    key_window(w, bottom, w.wlo - 1u);
  };
  for (int pass = 0; pass < 2; ++pass) {
    if (s.stage == 0u) {
      const uint32_t need = static_cast<uint32_t>(s.k) - s.carry_c;
      if (tot_c < need) { below(KEY_BOTTOM); return; }
      const int i = first_count(it, need);
      uint32_t lo, hi;
      range(i, lo, hi);
      if (lo != hi) { narrow(i, lo, hi); return; }
      const int j = it.list ? last_ge(it.keys, it.n, hi) : i;      // every tie of the k-th key
      const uint32_t sup = s.carry_c + it.count_at(j);
      const unsigned long long zk = s.carry_m + it.cm[j];
      if (!(s.p < 1.0f)) { resolve(sup, zk, hi); return; }
      s.T = nucleus_bound(s.p, zk);
      s.stage = 1u;
      s.floor_key = hi;
      if (it.list && s.carry_c == 0u) continue;                     // all of S_k is in this list
      s.carry_c = 0u;
      s.carry_m = 0ull;
      open_window(w, hi, s.top_key);
      return;
    }
    const unsigned long long tgt = s.T - s.carry_m;
    int imax = it.n - 1;
    if (it.list && s.floor_key >= w.wlo) imax = last_ge(it.keys, it.n, s.floor_key);
    const unsigned long long reach = imax >= 0 ? it.cm[imax] : 0ull;
    if (reach < tgt) {
      if (w.wlo <= s.floor_key)                                     // never reached: all of S_k
        resolve(s.carry_c + (imax >= 0 ? it.count_at(imax) : 0u), s.carry_m + reach, s.floor_key);
      else
        below(s.floor_key);
      return;
    }
    const int i = first_mass(it, tgt);
    uint32_t lo, hi;
    range(i, lo, hi);
    if (lo != hi) { narrow(i, lo, hi); return; }
    const int j = it.list ? last_ge(it.keys, it.n, hi) : i;
    resolve(s.carry_c + it.count_at(j), s.carry_m + it.cm[j], hi);
    return;
  }
}

// Listed windows of at most WARP_LIST keys are resolved by the prep warp.
constexpr int WARP_LIST = 512;

// Bitonic sort of n <= WARP_LIST keys into descending order by one warp.
__device__ void warp_sort_desc(uint32_t* keys, int n, int lane) {
  int p2 = 32;
  while (p2 < n) p2 <<= 1;
  for (int i = n + lane; i < p2; i += 32) keys[i] = 0u;
  __syncwarp();
  for (int k = 2; k <= p2; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = lane; i < p2; i += 32) {
        const int ix = i ^ j;
        if (ix > i) {
          const uint32_t a = keys[i], b = keys[ix];
          if (((i & k) == 0) ? a < b : a > b) {
            keys[i] = b;
            keys[ix] = a;
          }
        }
      }
      __syncwarp();
    }
}

// Inclusive prefix sums, in place, of n masses by one warp.
__device__ void warp_prefix(unsigned long long* cm, int n, int lane) {
  const int per = (n + 31) / 32;
  const int i0 = min(n, lane * per), i1 = min(n, i0 + per);
  unsigned long long sum = 0ull;
  for (int i = i0; i < i1; ++i) sum += cm[i];
  unsigned long long inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  unsigned long long run = inc - sum;
  for (int i = i0; i < i1; ++i) {
    run += cm[i];
    cm[i] = run;
  }
  __syncwarp();
}

// One warp per row: validate, merge the tile summaries (the full logprob,
// bit-identical to rlk_linear_logp), finish the rows with nothing to select
// and open the first window of the others; clear the row's round buffers.
__global__ void __launch_bounds__(128) pair_prep_kernel(const LinArgs P, const PairArgs A) {
  __shared__ uint32_t wkeys[4][WARP_LIST];
  __shared__ unsigned long long wcm[4][WARP_LIST];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (row >= P.T) return;
  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const int t = P.target[row];
  const float p = A.top_p ? A.top_p[row] : A.top_p_s;
  const int k = A.top_k ? A.top_k[row] : A.top_k_s;
  LinWin w;
  memset(&w, 0, sizeof(w));
  LinSel s;
  memset(&s, 0, sizeof(s));
  const float qnan = __int_as_float(0x7fc00000);
  if (!tau_ok(tau) || t < 0 || t >= VREAL || !(p > 0.0f && p <= 1.0f) || !(k == -1 || (k >= 1 && k <= VREAL))) {
    if (lane == 0) {
      if (A.out_full) A.out_full[row] = qnan;
      A.out_restr[row] = qnan;
      if (A.out_support) A.out_support[row] = -1;
      if (A.err) atomicAdd(A.err, 1);
      A.listn[row] = 0u;
      A.win[row] = w;
    }
    return;
  }
  const float c = __fdiv_rn(LOG2E, tau);
  float M, z;
  lin_merge(P, row, lane, c, M, z);
  const float xt = P.ws_xt[row];
  const float d = __fdiv_rn(xt - M, tau);
  const float full = d - logf(z);
  const bool k_on = !(k == -1 || k >= VREAL), p_on = p < 1.0f;
  const bool finite = M > -INFINITY && M < INFINITY && z > 0.0f && z < INFINITY;
  w.M = M;
  w.c = c;
  s.kt = key32(xt);
  s.d = d;
  s.top_key = key32(M);
  s.p = p_on ? p : 1.0f;
  s.k = k_on ? k : 0;
  const float* tp = P.ws_top + row * NTILE * TOPR;             // each tile's 8 largest, descending
  uint32_t listed = 0u;
  // When every tile's 8th kept logit lies below the window, the window's
  // logits are all among the kept ones: list them (no GEMM round needed).
  auto try_list = [&]() -> bool {
    bool covered = true;
#pragma unroll
    for (int q0 = 0; q0 < NTILE; q0 += 32) {                   // independent loads, no short circuit
      const int q = q0 + lane;
      if (q < NTILE) covered &= key32(__ldg(tp + q * TOPR + TOPR - 1)) < w.wlo;
    }
    if (!__all_sync(0xffffffffu, covered)) return false;
    // lane-strided (coalesced) pass, eight loads in flight; ballots keep the
    // list order fixed; the first WARP_LIST keys also go to the warp's slice
    uint32_t* dst = A.list + row * LIST_CAP;
    uint32_t total = 0u;
    constexpr int NV = NTILE * TOPR;
    for (int i0 = 0; i0 < NV; i0 += 256) {
      float v8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + 32 * u + lane;
        v8[u] = i < NV ? __ldg(tp + i) : -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t K = key32(v8[u]);
        const bool in = K >= w.wlo && i0 + 32 * u + lane < NV;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        const uint32_t at = total + __popc(m & ((1u << lane) - 1u));
        if (in && at < static_cast<uint32_t>(LIST_CAP)) dst[at] = K;
        if (in && at < static_cast<uint32_t>(WARP_LIST)) wkeys[warp][at] = K;
        total += __popc(m);
      }
    }
    if (total > static_cast<uint32_t>(LIST_CAP)) return false;
    w.mode |= WIN_LISTED;
    listed = total;
    return true;
  };
  if (finite && k_on) {
    // first bound: the k-th largest tile maximum (k distinct real tokens reach it)
    const float2* ml = P.ws_ml + row * NTILE;
    uint32_t tk[(NTILE + 31) / 32];
#pragma unroll
    for (int i = 0; i < (NTILE + 31) / 32; ++i) {
      const int q = lane + 32 * i;
      tk[i] = q < NTILE ? key32(ml[q].x) : 0u;
    }
    uint32_t pre = 0u;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = pre | (1u << bit);
      int n = 0;
#pragma unroll
      for (int i = 0; i < (NTILE + 31) / 32; ++i) n += tk[i] >= cand;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
      if (n >= k) pre = cand;
    }
    s.stage = 0u;
    open_window(w, (k <= NTILE && pre > KEY_BOTTOM) ? pre : KEY_BOTTOM, s.top_key);
    if (!try_list() && k <= NTILE * TOPR) {
      // tighter: the k-th largest kept logit, to its top 16 key bits
      uint32_t p16 = 0u;
      for (int bit = 15; bit >= 0; --bit) {
        const uint32_t cand = (p16 | (1u << bit)) << 16;
        int n = 0;
        for (int i = lane; i < NTILE * TOPR; i += 32) n += key32(tp[i]) >= cand;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
        if (n >= k) p16 |= 1u << bit;
      }
      if ((p16 << 16) > w.wlo) {
        open_window(w, p16 << 16, s.top_key);
        try_list();
      }
    }
  } else if (finite && p_on) {
    s.T = nucleus_bound(p, __float2ull_rn(z * FX_SCALE));
    s.stage = 1u;
    s.floor_key = KEY_BOTTOM;
    uint32_t lo = KEY_BOTTOM;
    if (1.0f - p >= 1e-4f) {
      const float L = log2f((1.0f - p) * z / (2.0f * static_cast<float>(VREAL)));
      const float B = M + L / c;
      if (B > -INFINITY && B < M) lo = key32(B);
    }
    open_window(w, lo, s.top_key);
    try_list();
  }
  if ((w.mode & WIN_LISTED) && listed <= static_cast<uint32_t>(WARP_LIST)) {
    // resolve here: sort the listed keys, prefix their masses, one decision
    const int n = static_cast<int>(listed);
    uint32_t* kk = wkeys[warp];
    unsigned long long* cmw = wcm[warp];
    __syncwarp();
    warp_sort_desc(kk, n, lane);
    for (int i = lane; i < n; i += 32) cmw[i] = lmass(key32_value(kk[i]), w.M, w.c);
    __syncwarp();
    warp_prefix(cmw, n, lane);
    if (lane == 0) {
      decide(Items{true, n, kk, nullptr, cmw}, w, s, row, A);   // lane 0's state is kept below
      if (w.mode != WIN_IDLE) listed = 0u;                      // a new window: GEMM rounds
    }
  }
  if (lane == 0) {
    if (A.out_full) A.out_full[row] = full;
    if (!finite) {
      A.out_restr[row] = qnan;
      if (A.out_support) A.out_support[row] = -1;
    } else if (!k_on && !p_on) {
      A.out_restr[row] = full;
      if (A.out_support) A.out_support[row] = VREAL;
    }
    A.listn[row] = (w.mode & WIN_LISTED) ? listed : 0u;
    A.win[row] = w;
    A.sel[row] = s;
    if (w.mode != WIN_IDLE) enqueue_row(A, 0, row, !(w.mode & WIN_LISTED));
  }
  // a row going through GEMM rounds starts from clear bucket counts
  const uint32_t mode = __shfl_sync(0xffffffffu, w.mode, 0);
  if (mode != WIN_IDLE && !(mode & WIN_LISTED)) {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4* hc = reinterpret_cast<uint4*>(A.hcnt + row * NB);
    for (int i = lane; i < NB / 4; i += 32) hc[i] = zero;
    uint4* hm = reinterpret_cast<uint4*>(A.hmass + row * NB);
    for (int i = lane; i < NB / 2; i += 32) hm[i] = zero;
  }
}

// Rows of the round, one block at a time: resolve from the list or narrow
// the window; clear the row's counts for the next round.
__global__ void __launch_bounds__(RT) pair_round_kernel(const PairArgs A, int round) {
  extern __shared__ __align__(16) unsigned char rsm[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(rsm);                        // LIST_CAP keys, or NB counts
  unsigned long long* cm = reinterpret_cast<unsigned long long*>(rsm + LIST_CAP * 4);
  __shared__ unsigned long long wm[RT / 32];
  __shared__ uint32_t wc[RT / 32];
  __shared__ LinWin sw;
  __shared__ LinSel ss;
  const int tid = threadIdx.x;
  const uint32_t nrows = A.counters[2 * round];
  for (uint32_t idx = blockIdx.x; idx < nrows; idx += gridDim.x) {
    const int64_t row = A.rowlist[(round & 1) * A.T + idx];
    const uint32_t ln = A.listn[row];
    if (tid == 0) {
      sw = A.win[row];
      ss = A.sel[row];
    }
    __syncthreads();
    if (ln & LIST_FAILED) {
      if (tid == 0) {
        A.out_restr[row] = __int_as_float(0x7fc00000);
        if (A.out_support) A.out_support[row] = -1;
        if (A.err) atomicAdd(A.err, 1);
        sw.mode = WIN_IDLE;
      }
    } else if (ln <= static_cast<uint32_t>(LIST_CAP)) {
      const int n = static_cast<int>(ln);
      const uint32_t* src = A.list + row * LIST_CAP;
      for (int i = tid; i < n; i += RT) keys[i] = src[i];
      sort_desc(keys, n);
      for (int i = tid; i < n; i += RT) cm[i] = lmass(key32_value(keys[i]), sw.M, sw.c);
      __syncthreads();
      block_prefix(cm, nullptr, n, wm, wc);
      if (tid == 0) decide(Items{true, n, keys, nullptr, cm}, sw, ss, row, A);
    } else {
      uint32_t* cc = keys;
      for (int i = tid; i < NB; i += RT) {
        cc[i] = A.hcnt[row * NB + i];
        cm[i] = A.hmass[row * NB + i];
      }
      __syncthreads();
      block_prefix(cm, cc, NB, wm, wc);
      if (tid == 0) decide(Items{false, NB, nullptr, cc, cm}, sw, ss, row, A);
    }
    __syncthreads();
    if (sw.mode != WIN_IDLE) {
      for (int i = tid; i < NB; i += RT) {
        A.hcnt[row * NB + i] = 0u;
        A.hmass[row * NB + i] = 0ull;
      }
      if (tid == 0) A.listn[row] = 0u;
    }
    if (tid == 0) {
      A.win[row] = sw;
      A.sel[row] = ss;
      if (sw.mode != WIN_IDLE) enqueue_row(A, round + 1, row, true);
    }
    __syncthreads();
  }
}

// Rows still searching after the last round (none is expected: a search
// takes at most five rounds per stage) get NaN and support -2.
__global__ void __launch_bounds__(256) pair_final_kernel(const PairArgs A) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (row >= A.T || A.win[row].mode == WIN_IDLE) return;
  A.out_restr[row] = __int_as_float(0x7fc00000);
  if (A.out_support) A.out_support[row] = -2;
  if (A.err) atomicAdd(A.err, 1);
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

// Host checks, tensor maps, arguments and the one-time kernel attributes
// shared by both entry points.
struct LinLaunch {
  CUtensorMap ta, tb;
  LinArgs P;
  unsigned grid;                            // one CTA per SM, at most one per tile
  int sms;
};

rlk_status lin_setup(LinLaunch& L, const void* hidden, int64_t T, int64_t H, int64_t hidden_stride,
                     const void* weight, int64_t weight_stride, const int32_t* target,
                     const float* temperature, float temperature_scalar, int32_t* err_count) {
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
  if (temperature) {
    if (!aligned(temperature, 4)) return fail(RLK_EALIGN, "temperature is not 4-byte aligned");
  } else if (!(temperature_scalar > 0.0f && temperature_scalar <= 3.402823466e38f)) {
    return fail(RLK_EINVAL, "temperature %g must be finite and > 0", (double)temperature_scalar);
  }
  if (err_count && !aligned(err_count, 4)) return fail(RLK_EALIGN, "err_count is not 4-byte aligned");

  if ((s = encode_tiled(&L.ta, hidden, static_cast<uint64_t>(H), static_cast<uint64_t>(T), hidden_stride, LM)) != RLK_OK)
    return s;
  if ((s = encode_tiled(&L.tb, weight, static_cast<uint64_t>(H), static_cast<uint64_t>(VPAD), weight_stride, LN)) != RLK_OK)
    return s;
  LinArgs& P = L.P;
  memset(&P, 0, sizeof(P));
  P.T = T;
  P.mt = static_cast<int>((T + LM - 1) / LM);
  P.nk = static_cast<int>(H / LK);
  P.target = target;
  P.tau_arr = temperature;
  P.tau_s = temperature_scalar;
  P.err = err_count;

  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(linear_kernel<EPI_SUMMARY>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(LIN_SMEM));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(linear_kernel<EPI_WINDOW>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(LIN_SMEM));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(linear_kernel<EPI_SUMMARY_TOP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(LIN_SMEM));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(pair_round_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ROUND_SMEM));
    // one shared-memory carveout for every kernel of a call, so that the SMs
    // are not reconfigured between the GEMM rounds and the small kernels
    const void* kernels[] = {reinterpret_cast<const void*>(linear_kernel<EPI_SUMMARY>),
                             reinterpret_cast<const void*>(linear_kernel<EPI_WINDOW>),
                             reinterpret_cast<const void*>(linear_kernel<EPI_SUMMARY_TOP8>),
                             reinterpret_cast<const void*>(merge_lin_kernel),
                             reinterpret_cast<const void*>(pair_prep_kernel),
                             reinterpret_cast<const void*>(pair_round_kernel),
                             reinterpret_cast<const void*>(pair_final_kernel)};
    for (const void* kf : kernels)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kf, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  e = cudaDeviceGetAttribute(&L.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  const int64_t ntiles = static_cast<int64_t>(P.mt) * NTILE;
  L.grid = static_cast<unsigned>(ntiles < L.sms ? ntiles : L.sms);
  return RLK_OK;
}

inline rlk_status launched() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? RLK_OK : fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
}

// Workspace of the pair entry point, regions 256-byte aligned.
struct PairLayout {
  size_t hmass, ml, top, sel, win, hcnt, list, xt, listn, rowlist, mlist, counters, mflag, total;
};
inline PairLayout pair_layout(int64_t T) {
  auto up = [](size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); };
  const size_t t = static_cast<size_t>(T), mt = (t + LM - 1) / LM;
  PairLayout L;
  size_t o = 0;
  L.hmass = o;    o = up(o + t * NB * 8);
  L.ml = o;       o = up(o + t * NTILE * 8);
  L.top = o;      o = up(o + t * NTILE * TOPR * 4);
  L.sel = o;      o = up(o + t * sizeof(LinSel));
  L.win = o;      o = up(o + t * sizeof(LinWin));
  L.hcnt = o;     o = up(o + t * NB * 4);
  L.list = o;     o = up(o + t * LIST_CAP * 4);
  L.xt = o;       o = up(o + t * 4);
  L.listn = o;    o = up(o + t * 4);
  L.rowlist = o;  o = up(o + 2 * t * 4);
  L.mlist = o;    o = up(o + 2 * mt * 4);
  L.counters = o; o = up(o + 2 * PAIR_ROUNDS * 4);       // counters and flags are contiguous:
  L.mflag = o;    o = up(o + PAIR_ROUNDS * mt * 4);      // one memset clears both
  L.total = o;
  return L;
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
  rlk_status s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  if (!workspace) return fail(RLK_EINVAL, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(RLK_EALIGN, "workspace is not 16-byte aligned");
  LinLaunch L;
  if ((s = lin_setup(L, hidden, T, H, hidden_stride, weight, weight_stride, target, temperature,
                     temperature_scalar, err_count)) != RLK_OK)
    return s;
  L.P.ws_ml = static_cast<float2*>(workspace);
  L.P.ws_xt = reinterpret_cast<float*>(static_cast<char*>(workspace) + static_cast<size_t>(T) * NTILE * 8);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  linear_kernel<EPI_SUMMARY><<<L.grid, LIN_THREADS, LIN_SMEM, st>>>(L.ta, L.tb, L.P);
  if ((s = launched()) != RLK_OK) return s;
  merge_lin_kernel<<<static_cast<unsigned>((T + 3) / 4), 128, 0, st>>>(L.P, out_full);
  return launched();
}

rlk_status rlk_linear_logp_pair(const void* hidden, int64_t T, int64_t H, int64_t hidden_stride,
                                const void* weight, int64_t weight_stride, const int32_t* target,
                                const float* temperature, float temperature_scalar, const float* top_p,
                                float top_p_scalar, const int32_t* top_k, int32_t top_k_scalar,
                                float* out_full, float* out_restr, int32_t* out_support, void* workspace,
                                int32_t* err_count, void* stream) {
  if (T < 0 || T >= (int64_t(1) << 24)) return fail(RLK_EINVAL, "T = %lld out of range [0, 2^24)", (long long)T);
  if (T == 0) return RLK_OK;
  rlk_status s;
  if ((s = check_out(out_restr, "out_restr", true)) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  if ((s = check_top_p(top_p, top_p_scalar)) != RLK_OK) return s;
  if ((s = check_top_k(top_k, top_k_scalar)) != RLK_OK) return s;
  if (!workspace) return fail(RLK_EINVAL, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(RLK_EALIGN, "workspace is not 256-byte aligned");
  const PairLayout W = pair_layout(T);
  if (W.total > RLK_LINEAR_PAIR_WORKSPACE_BYTES(T))
    return fail(RLK_EINVAL, "internal: workspace layout exceeds RLK_LINEAR_PAIR_WORKSPACE_BYTES");
  LinLaunch L;
  if ((s = lin_setup(L, hidden, T, H, hidden_stride, weight, weight_stride, target, temperature,
                     temperature_scalar, err_count)) != RLK_OK)
    return s;
  char* ws = static_cast<char*>(workspace);
  LinArgs& P = L.P;
  P.ws_ml = reinterpret_cast<float2*>(ws + W.ml);
  P.ws_xt = reinterpret_cast<float*>(ws + W.xt);
  P.ws_top = reinterpret_cast<float*>(ws + W.top);
  PairArgs A;
  memset(&A, 0, sizeof(A));
  A.T = T;
  A.top_p = top_p;
  A.top_p_s = top_p_scalar;
  A.top_k = top_k;
  A.top_k_s = top_k_scalar;
  A.out_full = out_full;
  A.out_restr = out_restr;
  A.out_support = out_support;
  A.err = err_count;
  A.win = reinterpret_cast<LinWin*>(ws + W.win);
  A.sel = reinterpret_cast<LinSel*>(ws + W.sel);
  A.hcnt = reinterpret_cast<uint32_t*>(ws + W.hcnt);
  A.hmass = reinterpret_cast<unsigned long long*>(ws + W.hmass);
  A.list = reinterpret_cast<uint32_t*>(ws + W.list);
  A.listn = reinterpret_cast<uint32_t*>(ws + W.listn);
  A.rowlist = reinterpret_cast<int32_t*>(ws + W.rowlist);
  A.mlist = reinterpret_cast<int32_t*>(ws + W.mlist);
  A.counters = reinterpret_cast<uint32_t*>(ws + W.counters);
  A.mflag = reinterpret_cast<uint32_t*>(ws + W.mflag);
  A.mt = P.mt;
  P.win = A.win;
  P.hcnt = A.hcnt;
  P.hmass = A.hmass;
  P.list = A.list;
  P.listn = A.listn;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t me = cudaMemsetAsync(ws + W.counters, 0, W.total - W.counters, st);
  if (me != cudaSuccess) return fail(RLK_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(me));
  linear_kernel<EPI_SUMMARY_TOP8><<<L.grid, LIN_THREADS, LIN_SMEM, st>>>(L.ta, L.tb, P);
  if ((s = launched()) != RLK_OK) return s;
  pair_prep_kernel<<<static_cast<unsigned>((T + 3) / 4), 128, 0, st>>>(P, A);
  if ((s = launched()) != RLK_OK) return s;
  const unsigned rgrid = static_cast<unsigned>(T < 4 * L.sms ? T : 4 * L.sms);
  for (int r = 0; r < PAIR_ROUNDS; ++r) {
    P.np = A.counters + 2 * r + 1;
    P.mlist = A.mlist + (r & 1) * P.mt;
    linear_kernel<EPI_WINDOW><<<static_cast<unsigned>(L.sms), LIN_THREADS, LIN_SMEM, st>>>(L.ta, L.tb, P);
    if ((s = launched()) != RLK_OK) return s;
    pair_round_kernel<<<rgrid, RT, ROUND_SMEM, st>>>(A, r);
    if ((s = launched()) != RLK_OK) return s;
  }
  pair_final_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, st>>>(A);
  return launched();
}

}  // extern "C"
