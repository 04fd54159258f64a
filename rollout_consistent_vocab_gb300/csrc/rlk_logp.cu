// rlk_logp.cu -- strict, batch-invariant token logprob for GB300 (sm_103a).
//
// One thread-block cluster of 8 CTAs per row; CTA r of the cluster plays
// virtual TP rank r of the fixed TP8 vocabulary partition ("Configurable
// H100 consistency runs", topology paragraph) and owns columns
// [19072 r, 19072 (r+1)).  Per CTA:
//
//   1. one mbarrier-tracked bulk copy (TMA, cp.async.bulk) streams the shard
//      (38144 B, 36864 B for the last shard whose 640 padded columns are
//      never read) from HBM into shared memory;
//   2. exact shard maximum with packed bf16x2 max;
//   3. shard sum-exp l_r = sum exp(s_j - m_r) in a fixed tree: thread t owns
//      16-byte chunks t, t+256, ... in that order, keeps even and odd columns
//      in the two lanes of a packed f32x2 accumulator, then a shuffle-xor
//      butterfly (IEEE addition is commutative, so every lane ends with the
//      same bits) and a left fold over the 8 warp sums;
//   4. restricted side only: an exact per-key count histogram (u16 counts
//      packed in pairs) over a window of at most 2048 bf16 order keys below
//      the shard maximum, holding every element that can belong to the
//      support.  The window's lower edge is a proven-safe cutoff: for top-k,
//      the k-th largest of the 256 per-thread maxima; for top-p, the value
//      below which the mass of the whole vocabulary cannot reach 1-p of the
//      total.
//   5. the CTA stores its summary (m_r, l_r, window) into the leader CTA's
//      shared memory over DSMEM and arrives on the cluster barrier.
//
// The leader (rank 0) merges the summaries as a left fold over shard index:
// each vocabulary shard contributes one summary and the summaries combine in
// one fixed order of vocabulary position (Reproduce and profile the Qwen3-8B
// TP4/CP2 experiment, "How non-default CUDA topology reuses TP4/CP2"), sums the 8
// histograms over DSMEM, and finds the top-k and top-p thresholds on the
// merged histogram.  Masses there are per-key exp values times integer
// counts in 2^-44 fixed point, so every sum is an exact integer sum and the
// support decision cannot depend on summation order.  If a threshold lies
// below the window (a row whose support reaches more than 2048 keys under
// its maximum) the leader re-counts further windows from the row in global
// memory; this path is slow but exact.
//
// Nothing depends on T or on where the row sits: the kernel configuration is
// fixed and every reduction tree is a function of the column index only.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "rlk_logp.h"

namespace rlk {

constexpr int VPAD = RLK_VOCAB_PADDED;
constexpr int VREAL = RLK_VOCAB_REAL;
constexpr int NSHARD = RLK_NUM_SHARDS;
constexpr int SW = RLK_SHARD_WIDTH;
constexpr int SHARD_CHUNKS = SW / 8;                        // 2384 16-byte chunks
constexpr int LAST_CHUNKS = (VREAL - (NSHARD - 1) * SW) / 8;  // 2304 real chunks
#ifndef RLK_NTHR
#define RLK_NTHR 128
#endif
constexpr int NTHR = RLK_NTHR;       // threads per CTA
constexpr int NWARP = NTHR / 32;
constexpr int ROW_WARPS = NSHARD * NWARP;
constexpr int CTAS_PER_SM = 5;
constexpr int MAXCH = (SHARD_CHUNKS + NTHR - 1) / NTHR;     // chunks per thread (9 or 10)
constexpr int KEEPCH = MAXCH;        // chunk maxima kept in registers
constexpr int WIN = 1024;            // candidate window, in bf16 order keys (8 binades)
constexpr int TMA_PIECES = 4;
constexpr int BUSY_HITS = 16;        // candidate chunks per warp above which it counts locally
constexpr float LOG2E = 1.4426950408889634f;   // log2(e)
constexpr float FX_SCALE = 17592186044416.0f;  // 2^44: fixed-point scale of masses
constexpr unsigned long long TIMEOUT_NS = 200000000ull;   // 0.2 s bound on every wait
constexpr int KEY_NEG_INF = 0x007F;  // order key of -inf; smaller keys are NaN patterns

static_assert(SW % 8 == 0 && (VREAL - (NSHARD - 1) * SW) % 8 == 0, "chunking");
static_assert((MAXCH - 1) * NTHR <= LAST_CHUNKS, "every thread owns MAXCH-1 chunks in every shard");
static_assert(SHARD_CHUNKS % TMA_PIECES == 0 && LAST_CHUNKS % TMA_PIECES == 0, "pieces");

enum : uint32_t { FLAG_TIMEOUT = 1u, FLAG_NAN = 2u };

// Sent by every CTA to every CTA before the candidate pass.
struct __align__(16) MidSlot {
  float xm;        // shard maximum (a bf16 value or -inf / +inf)
  int32_t lkey;    // order key reached by ceil(k/W) lane maxima of every warp of the shard
  uint32_t flags;
  float l;         // top-p-only rows: the shard's sum-exp (0 otherwise)
};

// Sent by every CTA to the leader at the end.
struct __align__(16) Summary {
  float xm;        // shard maximum
  float l;         // sum over the shard of exp(s_j - m_r) (NaN if the shard holds a NaN)
  uint32_t aux;    // greedy: first column holding the maximum; otherwise candidate messages sent
  uint32_t flags;
};

struct __align__(128) Smem {
  uint4 shard[SHARD_CHUNKS];       // 38144 B; the leader reuses it as scratch at the end
  uint32_t merged[WIN];            // leader: per-key candidate counts of the whole row
  uint32_t hist[WIN / 2];          // busy warps' per-key counts (u16 pairs), pushed once
  MidSlot mid[NSHARD];
  Summary slot[NSHARD];
  uint32_t red_u[NWARP];
  int32_t red_i[NWARP];
  float red_f[NWARP];
  uint32_t scan_c[NWARP];
  unsigned long long scan_m[NWARP];
  int32_t found_i;
  uint32_t found_c;
  unsigned long long found_m;
  uint32_t npush;
  int32_t win[4];
  float bc_f[4];
  int32_t sel_done;
  unsigned long long bar_load, bar_mid, bar_sum, bar_hist;
};
// five CTAs per SM: 5 * (sizeof + 1 KB reserved) <= 228 KB
static_assert(sizeof(Smem) + 1024 <= 233472 / CTAS_PER_SM, "shared memory budget of 5 CTAs per SM");

struct KParams {
  const uint16_t* logits;
  int64_t stride;
  const int32_t* target;
  const float* tau_arr;
  const float* p_arr;
  const int32_t* k_arr;
  float tau_s, p_s;
  int32_t k_s;
  float* out_full;
  float* out_restr;
  int32_t* out_support;
  const float* kl_policy_full;  // reference pass: out_kl = kl_policy_full - full
  float* out_kl;
  int32_t* err;
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 16-byte store into a peer CTA's shared memory, completing 16 bytes of
// transaction count on that CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar) : "memory");
}
// atomic add into a peer CTA's shared memory, completing 4 bytes on its mbarrier
__device__ __forceinline__ void red_async_add(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("red.async.relaxed.cluster.shared::cluster.mbarrier::complete_tx::bytes.add.u32 [%0], %1, [%2];"
               :: "r"(addr), "r"(v), "r"(bar) : "memory");
}
// shared-memory add without a return value (nothing waits for it)
__device__ __forceinline__ void red_shared_add(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" :: "r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long global_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
// the single expected arrival of a barrier, announcing `bytes` of transactions
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// One test of a barrier phase; a thread whose phase is not complete sleeps
// (up to 20 us) instead of spinning, so waiting warps leave the issue slots
// to working ones.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(20000u) : "memory");
  return ok != 0;
}
// Bounded wait on phase 0 of a barrier: gives up after TIMEOUT_NS of wall time.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar) {
  if (mbar_try(bar, 0)) return true;
  const unsigned long long t0 = global_timer();
  while (!mbar_try(bar, 0)) {
    if (global_timer() - t0 > TIMEOUT_NS) return false;
  }
  return true;
}

// packed f32x2 arithmetic (sm_100+ FP32x2 instructions)
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ bf16 keys

// Order key of a bf16 bit pattern: unsigned order equals numeric order for
// non-NaN values; -0 shares the key of +0.
__device__ __forceinline__ int okey(uint32_t b16) {
  if (b16 == 0x8000u) return 0x8000;
  return (b16 & 0x8000u) ? static_cast<int>(~b16 & 0xFFFFu) : static_cast<int>(b16 | 0x8000u);
}
__device__ __forceinline__ int okey_of(float x) { return okey(__float_as_uint(x) >> 16); }
__device__ __forceinline__ float key_value(int k) {
  const uint32_t b = (k >= 0x8000) ? static_cast<uint32_t>(k & 0x7FFF)
                                   : (~static_cast<uint32_t>(k) & 0xFFFFu);
  return __uint_as_float(b << 16);
}
// Largest order key whose value is <= x (x finite float, not necessarily bf16).
__device__ __forceinline__ int okey_floor(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t k32 = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  const int k = static_cast<int>(k32 >> 16) - 1;   // one key of slack covers both signs
  return k < 0 ? 0 : k;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  return *reinterpret_cast<__nv_bfloat162*>(&w);
}

// fixed-point mass of one element at key value v: exp(s - M) * 2^44
__device__ __forceinline__ unsigned long long qfx(float v, float M, float c) {
  const float q = ex2((v - M) * c);
  return __float2ull_rn(q * FX_SCALE);
}

// ------------------------------------------------------------ block helpers

// Fixed-order sum: butterfly inside each warp, then a left fold over warps.
__device__ __forceinline__ float block_sum_fixed(float v, Smem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) S.red_f[warp] = v;
  __syncthreads();
  float r = S.red_f[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) r = r + S.red_f[w];
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_min_int(int v, Smem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_min_sync(0xffffffffu, v);
  if (lane == 0) S.red_i[warp] = v;
  __syncthreads();
  int r = S.red_i[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) r = min(r, S.red_i[w]);
  __syncthreads();
  return r;
}

// j-th largest (1 <= j <= 32) of the warp's 32 keys, on every lane: peel off
// the maximum value with its multiplicity until j keys are covered.
__device__ __forceinline__ int warp_kth_largest(int key, int j) {
  unsigned v = static_cast<unsigned>(key);
  int covered = 0;
  for (;;) {
    const unsigned m = __reduce_max_sync(0xffffffffu, v);
    covered += __popc(__ballot_sync(0xffffffffu, v == m));
    if (covered >= j || m == 0u) return static_cast<int>(m);
    if (v == m) v = 0u;
  }
}

// Exclusive block scan of (count, mass); also returns the block totals.
__device__ __forceinline__ void block_excl_scan(uint32_t c, unsigned long long m, uint32_t& ec,
                                                unsigned long long& em, uint32_t& tc,
                                                unsigned long long& tm, Smem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ic = c;
  unsigned long long im = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t yc = __shfl_up_sync(0xffffffffu, ic, o);
    const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, o);
    if (lane >= o) { ic += yc; im += ym; }
  }
  if (lane == 31) { S.scan_c[warp] = ic; S.scan_m[warp] = im; }
  __syncthreads();
  uint32_t bc = 0, sc = 0;
  unsigned long long bm = 0, sm = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    if (w < warp) { bc += S.scan_c[w]; bm += S.scan_m[w]; }
    sc += S.scan_c[w];
    sm += S.scan_m[w];
  }
  ec = bc + ic - c;
  em = bm + im - m;
  tc = sc;
  tm = sm;
  __syncthreads();
}

// ceil(p * z) for a fixed-point mass z < 2^63 and p in (0, 1], exact in p's
// float value: p * 2^32 is an integer for every float p >= 2^-9, and the
// product is formed in 128 bits.
__device__ __forceinline__ unsigned long long nucleus_bound(float p, unsigned long long z) {
  const unsigned long long pf = __float2ull_rn(p * 4294967296.0f);
  const unsigned long long lo = z * pf;
  const unsigned long long hi = __umul64hi(z, pf);
  const unsigned long long fl = (hi << 32) | (lo >> 32);
  return fl + ((lo & 0xFFFFFFFFull) != 0ull);
}

// ------------------------------------------------------------ leader: selection

struct SelResult { uint32_t support; unsigned long long zs; int min_key; };

// Count the row's real elements whose key lies in [wlo, whi] (global memory
// re-read; fallback for supports that reach below the first window).
__device__ void count_window_global(const uint16_t* rowp, int wlo, int whi, uint32_t* cnt) {
  const int n = whi - wlo + 1;
  for (int i = threadIdx.x; i < n; i += NTHR) cnt[i] = 0;
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(rowp);
  for (int ch = threadIdx.x; ch < VREAL / 8; ch += NTHR) {
    const uint4 v = __ldg(src + ch);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = (w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
      const int K = okey(b);
      if (K >= wlo && K <= whi) atomicAdd(&cnt[whi - K], 1u);
    }
  }
  __syncthreads();
}

struct WinScan {
  int i0, i1;                 // this thread's key range [i0, i1) in the window
  uint32_t base_c;            // counts of all keys before i0 (carry included)
  unsigned long long base_m;
  uint32_t tot_c;             // window totals
  unsigned long long tot_m;
};

__device__ __forceinline__ WinScan scan_window(const uint32_t* cnt, int n, int whi, float M, float c,
                                               uint32_t carry_c, unsigned long long carry_m,
                                               Smem& S) {
  WinScan w;
  const int per = (n + NTHR - 1) / NTHR;
  w.i0 = min(n, static_cast<int>(threadIdx.x) * per);
  w.i1 = min(n, w.i0 + per);
  uint32_t lc = 0;
  unsigned long long lm = 0;
  for (int i = w.i0; i < w.i1; ++i) {
    const uint32_t k = cnt[i];
    if (k) { lc += k; lm += k * qfx(key_value(whi - i), M, c); }
  }
  uint32_t ec;
  unsigned long long em;
  block_excl_scan(lc, lm, ec, em, w.tot_c, w.tot_m, S);
  w.base_c = carry_c + ec;
  w.base_m = carry_m + em;
  return w;
}

// General selection over successive windows of WIN keys from the top: exact
// for any support size.  Used when the first window does not hold every
// threshold.
__device__ __noinline__ SelResult select_support(Smem& S, uint32_t* cnt0, uint32_t* cntB, int hi,
                                                 int lo, const uint16_t* rowp, float M, float c,
                                                 float Z, float p, int k, bool k_on, bool p_on) {
  const int tid = threadIdx.x;
  int vk_key = -1;                    // lowest key of S_k (-1: top-k off)
  uint32_t sup_k = VREAL;
  unsigned long long zk = __float2ull_rn(Z * FX_SCALE);

  // ---- stage K: k-th largest value and the top-k mass
  if (k_on) {
    int whi = hi, wlo = lo;
    const uint32_t* cnt = cnt0;
    uint32_t carry_c = 0;
    unsigned long long carry_m = 0;
    for (;;) {
      const int n = whi - wlo + 1;
      const WinScan w = scan_window(cnt, n, whi, M, c, carry_c, carry_m, S);
      if (tid == 0) S.found_i = -1;
      __syncthreads();
      uint32_t rc = w.base_c;
      unsigned long long rm = w.base_m;
      for (int i = w.i0; i < w.i1; ++i) {
        const uint32_t ci = cnt[i];
        const unsigned long long mi = ci ? ci * qfx(key_value(whi - i), M, c) : 0ull;
        const bool last_window = (wlo == 0) && (i == n - 1);
        if (rc < static_cast<uint32_t>(k) && (rc + ci >= static_cast<uint32_t>(k) || last_window)) {
          S.found_i = whi - i;
          S.found_c = rc + ci;
          S.found_m = rm + mi;
        }
        rc += ci;
        rm += mi;
      }
      __syncthreads();
      if (S.found_i >= 0) {
        vk_key = S.found_i;
        sup_k = S.found_c;
        zk = S.found_m;
        __syncthreads();
        break;
      }
      carry_c += w.tot_c;
      carry_m += w.tot_m;
      if (wlo == 0) { vk_key = 0; sup_k = carry_c; zk = carry_m; break; }
      whi = wlo - 1;
      wlo = max(0, whi - (WIN - 1));
      count_window_global(rowp, wlo, whi, cntB);
      cnt = cntB;
    }
  }
  if (!p_on) return SelResult{sup_k, zk, vk_key};

  // ---- stage P: nucleus threshold inside S_k
  const unsigned long long T = nucleus_bound(p, zk);
  int whi = hi, wlo = lo;
  const uint32_t* cnt = cnt0;
  uint32_t carry_c = 0;
  unsigned long long carry_m = 0;
  for (;;) {
    const int n = whi - wlo + 1;
    const bool k_in_window = vk_key >= wlo;
    const int imax = k_in_window ? (whi - vk_key) : (n - 1);
    const bool bounded = k_in_window || (wlo == 0);
    const WinScan w = scan_window(cnt, n, whi, M, c, carry_c, carry_m, S);
    if (tid == 0) S.found_i = -1;
    __syncthreads();
    uint32_t rc = w.base_c;
    unsigned long long rm = w.base_m;
    for (int i = w.i0; i < w.i1 && i <= imax; ++i) {
      const uint32_t ci = cnt[i];
      const unsigned long long mi = ci ? ci * qfx(key_value(whi - i), M, c) : 0ull;
      if (rm < T && (rm + mi >= T || (i == imax && bounded))) {
        S.found_i = whi - i;
        S.found_c = rc + ci;
        S.found_m = rm + mi;
      }
      rc += ci;
      rm += mi;
    }
    __syncthreads();
    if (S.found_i >= 0) {
      SelResult r{S.found_c, S.found_m, S.found_i};
      __syncthreads();
      return r;
    }
    carry_c += w.tot_c;
    carry_m += w.tot_m;
    if (bounded) return SelResult{carry_c, carry_m, wlo};   // unreachable in practice
    whi = wlo - 1;
    wlo = max(0, whi - (WIN - 1));
    count_window_global(rowp, wlo, whi, cntB);
    cnt = cntB;
  }
}

// Selection by one warp when the first window holds every threshold (the
// common case).  Keys hi, hi-1, ..., lo are taken in blocks of 128 (4
// consecutive keys per lane): first a scan of the counts alone finds the
// top-k boundary, then one scan of the fixed-point masses over S_k finds the
// nucleus boundary.  Returns false if a threshold may lie below the window.
__device__ __forceinline__ uint32_t warp_incl_scan_u32(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__device__ __forceinline__ bool select_warp(const uint32_t* cnt, int hi, int lo, float M, float c,
                                         float Z, float p, int k, bool k_on, bool p_on,
                                         SelResult& out) {
  constexpr int BLK = 4 * 32;
  const int lane = threadIdx.x & 31;
  const int n = hi - lo + 1;
  int imax = n - 1;
  uint32_t sup_k = 0;
  // ---- top-k boundary from the counts
  if (k_on) {
    uint32_t carry = 0;
    int fi = -1;
    for (int b0 = 0; b0 < n && fi < 0; b0 += BLK) {
      uint32_t cj[4], lc = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = b0 + 4 * lane + j;
        cj[j] = (i < n) ? cnt[i] : 0u;
        lc += cj[j];
      }
      const uint32_t ic = warp_incl_scan_u32(lc);
      uint32_t rc = carry + ic - lc;
      int f = -1;
      uint32_t fc = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (f < 0 && rc < static_cast<uint32_t>(k) && rc + cj[j] >= static_cast<uint32_t>(k)) {
          f = b0 + 4 * lane + j;
          fc = rc + cj[j];
        }
        rc += cj[j];
      }
      const unsigned bal = __ballot_sync(0xffffffffu, f >= 0);
      if (bal) {
        const int src = __ffs(bal) - 1;
        fi = __shfl_sync(0xffffffffu, f, src);
        sup_k = __shfl_sync(0xffffffffu, fc, src);
      }
      carry += __shfl_sync(0xffffffffu, ic, 31);
    }
    if (fi < 0) return false;                  // k-th value below the window
    imax = fi;
  }
  // ---- masses over S_k (all of it in one block in the common case)
  unsigned long long zk = k_on ? 0ull : __float2ull_rn(Z * FX_SCALE);
  const bool one_block = imax < BLK;
  if (k_on && !one_block) {
    for (int b0 = 0; b0 <= imax; b0 += BLK) {
      unsigned long long lm = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = b0 + 4 * lane + j;
        const uint32_t ci = (i <= imax) ? cnt[i] : 0u;
        if (ci) lm += ci * qfx(key_value(hi - i), M, c);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lm += __shfl_xor_sync(0xffffffffu, lm, o);
      zk += lm;
    }
  }
  if (k_on && !p_on && !one_block) {
    out = SelResult{sup_k, zk, hi - imax};
    return true;
  }
  unsigned long long T = (k_on && one_block) ? 0ull : nucleus_bound(p, zk);
  uint32_t carry_c = 0;
  unsigned long long carry_m = 0;
  for (int b0 = 0; b0 <= imax; b0 += BLK) {
    uint32_t cj[4], lc = 0;
    unsigned long long mj[4], lm = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = b0 + 4 * lane + j;
      cj[j] = (i <= imax) ? cnt[i] : 0u;
      mj[j] = cj[j] ? cj[j] * qfx(key_value(hi - i), M, c) : 0ull;
      lc += cj[j];
      lm += mj[j];
    }
    const uint32_t ic = warp_incl_scan_u32(lc);
    const unsigned long long im = warp_incl_scan_u64(lm);
    if (k_on && one_block) {
      zk = __shfl_sync(0xffffffffu, im, 31);   // the whole of S_k
      if (!p_on) {
        out = SelResult{sup_k, zk, hi - imax};
        return true;
      }
      T = nucleus_bound(p, zk);
    }
    uint32_t rc = carry_c + ic - lc;
    unsigned long long rm = carry_m + im - lm;
    int f = -1;
    uint32_t fc = 0;
    unsigned long long fm = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = b0 + 4 * lane + j;
      if (f < 0 && i <= imax && rm < T && (rm + mj[j] >= T || (i == imax && k_on))) {
        f = i;
        fc = rc + cj[j];
        fm = rm + mj[j];
      }
      rc += cj[j];
      rm += mj[j];
    }
    const unsigned bal = __ballot_sync(0xffffffffu, f >= 0);
    if (bal) {
      const int src = __ffs(bal) - 1;
      out = SelResult{__shfl_sync(0xffffffffu, fc, src), __shfl_sync(0xffffffffu, fm, src),
                      hi - __shfl_sync(0xffffffffu, f, src)};
      return true;
    }
    carry_c += __shfl_sync(0xffffffffu, ic, 31);
    carry_m += __shfl_sync(0xffffffffu, im, 31);
  }
  return false;                                  // nucleus reaches below the window
}

// The 16-byte exchange message of this CTA (rank r) to CTA `to` (a local
// store when `to` is this CTA).
__device__ __forceinline__ void send_mid(Smem& S, uint32_t r, int to, float xm, int lkey,
                                         uint32_t flags, float l, uint32_t bar_mid) {
  const uint4 msg = make_uint4(__float_as_uint(xm), static_cast<uint32_t>(lkey), flags,
                               __float_as_uint(l));
  if (to == static_cast<int>(r))
    *reinterpret_cast<uint4*>(&S.mid[r]) = msg;
  else
    st_async_v4(map_rank(smem_addr(&S.mid[r]), to), msg, map_rank(bar_mid, to));
}

// ------------------------------------------------------------ the kernel

template <bool RESTR>
__global__ void __cluster_dims__(NSHARD, 1, 1) __launch_bounds__(NTHR, CTAS_PER_SM)
logp_kernel(const KParams P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const uint32_t r = cluster_rank();
  const int64_t row = blockIdx.x / NSHARD;

  const int nchunks = (r == NSHARD - 1) ? LAST_CHUNKS : SHARD_CHUNKS;
  const uint16_t* rowp = P.logits + row * P.stride;
  const uint32_t bar_load = smem_addr(&S.bar_load);
  const uint32_t bar_mid = smem_addr(&S.bar_mid);
  const uint32_t bar_sum = smem_addr(&S.bar_sum);
  const uint32_t bar_hist = smem_addr(&S.bar_hist);

  // ---- 1. the bulk copy of the shard into shared memory goes out first
  if (tid == 0) {
    mbar_init(bar_load, 1);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = static_cast<uint32_t>(nchunks) * 16u;
    mbar_arrive_expect_tx(bar_load, bytes);
    const uint64_t pol = evict_first_policy();
    const uint32_t piece = bytes / TMA_PIECES;
    const char* src = reinterpret_cast<const char*>(rowp + static_cast<int64_t>(r) * SW);
    const uint32_t dst = smem_addr(S.shard);
#pragma unroll
    for (int i = 0; i < TMA_PIECES; ++i) bulk_load(dst + i * piece, src + i * piece, piece, bar_load, pol);
  }

  // ---- row parameters (every CTA of the cluster takes the same decisions)
  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const float p = RESTR ? (P.p_arr ? P.p_arr[row] : P.p_s) : 1.0f;
  const int k = RESTR ? (P.k_arr ? P.k_arr[row] : P.k_s) : -1;
  const int t = P.target[row];
  const bool valid = (tau >= 0.0f) && (tau <= 3.402823466e38f) && (p > 0.0f) && (p <= 1.0f) &&
                     (k == -1 || (k >= 1 && k <= VREAL)) && (t >= 0) && (t < VREAL);
  if (!valid) {
    if (tid == 0) {
      // the copy writes this CTA's shared memory: let it land before leaving
      mbar_wait_bounded(bar_load);
      if (r == 0) {
        if (P.out_full) P.out_full[row] = __int_as_float(0x7fc00000);
        if (RESTR && P.out_restr) P.out_restr[row] = __int_as_float(0x7fc00000);
        if (RESTR && P.out_support) P.out_support[row] = -1;
        if (P.out_kl) P.out_kl[row] = __int_as_float(0x7fc00000);
        if (P.err) atomicAdd(P.err, 1);
      }
    }
    return;
  }
  const bool greedy = (tau == 0.0f);
  const bool k_on = (k != -1) && (k < VREAL);
  const bool p_on = (p < 1.0f);
  const bool sel = RESTR && !greedy && (k_on || p_on);
  // the leader needs the target's logit at the end: start the load now
  const float xt = (r == 0) ? __uint_as_float(static_cast<uint32_t>(__ldg(rowp + t)) << 16) : 0.0f;

  // ---- barriers that peers signal, and the leader's histogram
  if (tid == 0) {
    mbar_init(bar_mid, 1);
    mbar_init(bar_sum, 1);
    mbar_init(bar_hist, 1);
    // messages from the 7 peers: 16 bytes each
    if (sel) mbar_arrive_expect_tx(bar_mid, (NSHARD - 1) * 16);
    if (r == 0) mbar_arrive_expect_tx(bar_sum, (NSHARD - 1) * 16);
    S.npush = 0u;
  }
  if (sel) {
    if (r == 0)
      for (int i = tid; i < WIN; i += NTHR) S.merged[i] = 0u;
    else
      for (int i = tid; i < WIN / 2; i += NTHR) S.hist[i] = 0u;
  }
  __syncthreads();
  // S0: barriers initialised and the leader's histogram zeroed.  One thread
  // publishes all of it to the cluster (the block barrier above orders the
  // other threads' stores before its fence); everyone arrives relaxed.
  if (tid == 0) {
    if (sel && r == 0) asm volatile("fence.acq_rel.cluster;" ::: "memory");
    else asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_arrive_relaxed();
  uint32_t flags = 0;
  if (!mbar_wait_bounded(bar_load)) {
    flags |= FLAG_TIMEOUT;
    mbar_wait_bounded(bar_load);   // give copies in flight a second bounded chance to land
  }

  // ---- 2. shard maximum; per-chunk maxima stay in registers for the candidate pass.
  // bf16 max ignores NaN; a NaN shows up as a NaN sum-exp (or in the scan below).
  const uint4* sh = S.shard;
  const __nv_bfloat162 ninf2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
  __nv_bfloat162 cm[KEEPCH];      // later chunks' maxima are recomputed when needed
  __nv_bfloat162 m2 = ninf2;
#pragma unroll
  for (int i = 0; i < MAXCH; ++i) {
    const int ch = tid + i * NTHR;
    __nv_bfloat162 cmax = ninf2;
    if (i < MAXCH - 1 || ch < nchunks) {   // all but the last chunk of every thread exist
      const uint4 v = sh[ch];
      cmax = __hmax2(__hmax2(as_bf2(v.x), as_bf2(v.y)), __hmax2(as_bf2(v.z), as_bf2(v.w)));
      m2 = __hmax2(m2, cmax);
    }
    if (i < KEEPCH) cm[i] = cmax;
  }
  const int tkey = okey_of(fmaxf(__low2float(m2), __high2float(m2)));
  // Pooled top-k bound: warp w certifies kw = ceil(k/W) lane maxima at or above
  // lw (its kw-th largest lane maximum), so the W warps of the row certify
  // W*kw >= k tokens at or above the minimum of lw over the cluster.
  const int kw = (k + ROW_WARPS - 1) / ROW_WARPS;
  const bool k_bound = sel && k_on && kw <= 32;
  {
    const int lane = tid & 31, warp = tid >> 5;
    const int lw = k_bound ? warp_kth_largest(tkey, kw) : 0;
    const unsigned wmax = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(tkey));
    if (lane == 0) { S.red_u[warp] = wmax; S.red_i[warp] = lw; }
  }
  __syncthreads();
  unsigned xkey = S.red_u[0];
  int lkey = S.red_i[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) { xkey = max(xkey, S.red_u[w]); lkey = min(lkey, S.red_i[w]); }
  const float xm = key_value(static_cast<int>(xkey));
  const bool xm_finite = (xm > -INFINITY) && (xm < INFINITY);

  uint32_t first = 0x7fffffffu;
  if (greedy || xm == -INFINITY) {
    // greedy: first column of this shard holding its maximum; both cases: NaN scan
    bool nan_seen = false;
    int f = 0x7fffffff;
    for (int ch = tid; ch < nchunks; ch += NTHR) {
      const uint4 v = sh[ch];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        const float x = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
        nan_seen |= (x != x);
        if (x == xm) f = min(f, ch * 8 + j);
      }
    }
    if (__syncthreads_or(nan_seen)) flags |= FLAG_NAN;
    if (greedy) {
      f = block_min_int(f, S);
      if (f != 0x7fffffff) first = static_cast<uint32_t>(f + static_cast<int>(r) * SW);
    }
  }

  cluster_wait();              // S0 complete: peers' barriers and histogram are ready
  // Rows with top-k send their maximum and bound now and overlap the exchange
  // with the sum-exp pass; top-p-only rows also send their sum-exp, which
  // tightens the candidate window, so they send after that pass.
  const bool late_mid = sel && !k_on;
  if (sel && !late_mid && tid < NSHARD) send_mid(S, r, tid, xm, lkey, flags, 0.0f, bar_mid);

  // ---- 3. shard sum-exp, fixed tree (while the peers' messages travel)
  float l = 0.0f;
  if (!greedy && xm_finite) {
    const float c = __fdiv_rn(LOG2E, tau);
    const uint64_t nxm2 = pack2(-xm, -xm);
    const uint64_t c2 = pack2(c, c);
    uint64_t acc = pack2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < MAXCH; ++i) {
      const int ch = tid + i * NTHR;
      if (i < MAXCH - 1 || ch < nchunks) {   // all but the last chunk of every thread exist
        const uint4 v = sh[ch];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t a = mul2(add2(pack2(bf16_lo(w[j]), bf16_hi(w[j])), nxm2), c2);
          float a0, a1;
          unpack2(a, a0, a1);
          acc = add2(acc, pack2(ex2(a0), ex2(a1)));
        }
      }
    }
    float e0, e1;
    unpack2(acc, e0, e1);
    l = block_sum_fixed(e0 + e1, S);
  }
  if (late_mid && tid < NSHARD) send_mid(S, r, tid, xm, lkey, flags, l, bar_mid);

  // ---- 4. candidate pass: every element of the window is counted straight
  //           into the leader's histogram (one shared-memory add per element)
  int hi = 0, lo = 1;
  if (sel) {
    if (tid == 0) {
      // the window of candidate keys, the same in every CTA of the cluster
      if (!mbar_wait_bounded(bar_mid)) flags |= FLAG_TIMEOUT;
      int L = 0x7fffffff;
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < NSHARD; ++q) {
        M = fmaxf(M, S.mid[q].xm);
        L = min(L, S.mid[q].lkey);
      }
      int whi = 0, wlo = 1;
      if (M > -INFINITY && M < INFINITY) {
        whi = okey_of(M);
        wlo = max(0, whi - (WIN - 1));
        if (k_on) {
          wlo = max(wlo, L);
        } else {
          // Tokens with s <= s_max + ln((1-p) Z / V) cannot reach the nucleus:
          // even all V of them would hold at most 1-p of the total mass Z
          // (relative to the maximum), so the mass strictly above any of them is
          // at least p Z.  Z is merged here exactly as the leader merges it; the
          // slack keeps the float evaluation on the safe side.
          const float cz = __fdiv_rn(LOG2E, tau);
          float Z = 0.0f;
#pragma unroll
          for (int q = 0; q < NSHARD; ++q)
            if (S.mid[q].xm > -INFINITY) Z = fmaf(S.mid[q].l, ex2((S.mid[q].xm - M) * cz), Z);
          const float lnz = fmaxf(0.0f, logf(Z * 0.9999f));
          const float width =
              tau * (logf(static_cast<float>(VREAL) / (1.0f - p)) * 1.0001f + 1e-3f - lnz);
          wlo = max(wlo, okey_floor(M - width));
        }
        wlo = max(wlo, KEY_NEG_INF);
      }
      S.win[0] = whi;
      S.win[1] = wlo;
      S.win[2] = static_cast<int>(flags);
    }
    __syncthreads();
    hi = S.win[0];
    lo = S.win[1];
    flags = static_cast<uint32_t>(S.win[2]);
    uint32_t sent = 0;
    if (xm_finite && lo <= hi && static_cast<int>(xkey) >= lo) {
      const float vlo_f = key_value(lo);
      const __nv_bfloat162 vlo2 = __floats2bfloat162_rn(vlo_f, vlo_f);
      const uint32_t dst = map_rank(smem_addr(S.merged), 0);
      const uint32_t rbar = map_rank(bar_hist, 0);
      // chunks whose maximum reaches the window, from the register chunk maxima
      uint32_t hitmask = 0;
#pragma unroll
      for (int i = 0; i < MAXCH; ++i)
        if (__hge2_mask(cm[i], vlo2) != 0u) hitmask |= 1u << i;
      // warps with many candidate chunks count locally and push per key;
      // the others send one add per element
      const bool busy = (r != 0) && __reduce_add_sync(0xffffffffu, __popc(hitmask)) > BUSY_HITS;
      // with a positive window every candidate is positive: its key is b | 0x8000
      const bool pos_window = vlo_f > 0.0f;
      while (hitmask) {
        const int i = __ffs(hitmask) - 1;
        hitmask &= hitmask - 1;
        const uint4 v = sh[tid + i * NTHR];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t bits = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) bits |= (__hge2_mask(as_bf2(w[j]), vlo2) & 0x00010001u) << j;
        while (bits) {
          const int pos = __ffs(bits) - 1;
          bits &= bits - 1;
          const int j = pos & 3;
          const uint32_t wj = (j == 0) ? w[0] : (j == 1) ? w[1] : (j == 2) ? w[2] : w[3];
          const uint32_t b = (pos & 16) ? (wj >> 16) : (wj & 0xFFFFu);
          const int idx = hi - (pos_window ? static_cast<int>(b | 0x8000u) : okey(b));
          if (r == 0) {
            red_shared_add(&S.merged[idx], 1u);
          } else if (busy) {
            red_shared_add(&S.hist[idx >> 1], 1u << ((idx & 1) * 16));
          } else {
            red_async_add(dst + 4u * static_cast<uint32_t>(idx), 1u, rbar);
            ++sent;
          }
        }
      }
      if (__syncthreads_or(busy)) {
        // push the busy warps' counts, one add per nonzero key
        const int nwords = (hi - lo + 2) >> 1;
        for (int iw = tid; iw < nwords; iw += NTHR) {
          const uint32_t hw = S.hist[iw];
          if (hw & 0xFFFFu) { red_async_add(dst + 8u * iw, hw & 0xFFFFu, rbar); ++sent; }
          if (hw >> 16) { red_async_add(dst + 8u * iw + 4u, hw >> 16, rbar); ++sent; }
        }
      }
    }
    // the leader learns how many adds each peer sent from its summary
    sent = __reduce_add_sync(0xffffffffu, sent);
    if ((tid & 31) == 0 && sent) atomicAdd(&S.npush, sent);
    __syncthreads();
  }

  // ---- 5. summary to the leader
  if (tid == 0) {
    const uint4 msg = make_uint4(__float_as_uint(xm), __float_as_uint(l), sel ? S.npush : first, flags);
    if (r == 0) *reinterpret_cast<uint4*>(&S.slot[0]) = msg;
    else st_async_v4(map_rank(smem_addr(&S.slot[r]), 0), msg, map_rank(bar_sum, 0));
  }
  if (r != 0) return;          // messages carry everything the leader needs

  // ================= leader: merge in fixed shard order =================
  // One thread waits for the peers' messages; warp 0 merges and selects; the
  // whole block joins only for the general (wide-support) selection.
  if (tid == 0) {
    bool timed_out = !mbar_wait_bounded(bar_sum);
    uint32_t pushed = 0;
#pragma unroll
    for (int q = 1; q < NSHARD; ++q) pushed += S.slot[q].aux;
    if (sel) {
      mbar_arrive_expect_tx(bar_hist, 4u * pushed);
      if (!mbar_wait_bounded(bar_hist)) timed_out = true;
    }
    S.win[3] = timed_out ? 1 : 0;
  }
  __syncthreads();
  const bool timed_out = S.win[3] != 0;
  if (tid >= 32 && !sel) return;   // only warp 0 finishes rows without a support search
  bool bad = timed_out;
  float M = -INFINITY;
  float full = __int_as_float(0x7fc00000), restr = full;
  int support = -1;
  float Z = 0.0f, d = 0.0f;
  const float c = greedy ? 0.0f : __fdiv_rn(LOG2E, tau);
  bool done = true;
  SelResult sr{0u, 0ull, 0};
  if (tid < 32) {
#pragma unroll
    for (int q = 0; q < NSHARD; ++q) {
      const Summary& s = S.slot[q];
      if ((s.flags & (FLAG_NAN | FLAG_TIMEOUT)) || s.xm == INFINITY || s.l != s.l) bad = true;
      M = fmaxf(M, s.xm);
    }
    bad |= !(M > -INFINITY);
    if (!bad && greedy) {
      uint32_t amax = 0x7fffffffu;
#pragma unroll
      for (int q = NSHARD - 1; q >= 0; --q)
        if (S.slot[q].xm == M) amax = S.slot[q].aux;
      full = restr = (static_cast<uint32_t>(t) == amax) ? 0.0f : -INFINITY;
      support = 1;
    } else if (!bad) {
      if (isinf(__fdiv_rn(M, tau))) {
        bad = true;
      } else {
#pragma unroll
        for (int q = 0; q < NSHARD; ++q) {
          const Summary& s = S.slot[q];
          if (s.xm > -INFINITY) Z = fmaf(s.l, ex2((s.xm - M) * c), Z);
        }
        d = __fdiv_rn(xt - M, tau);
        full = d - logf(Z);
        restr = full;
        support = VREAL;
      }
    }
    if (sel && !bad) done = select_warp(S.merged, hi, lo, M, c, Z, p, k, k_on, p_on, sr);
    if (sel && tid == 0) {
      S.sel_done = done ? 1 : 0;
      S.bc_f[0] = M;
      S.bc_f[1] = Z;
    }
  }
  if (sel) {
    __syncthreads();
    if (!S.sel_done) {
      // wide support: the whole block scans further windows
      uint32_t* cntB = reinterpret_cast<uint32_t*>(S.shard);
      sr = select_support(S, S.merged, cntB, hi, lo, rowp, S.bc_f[0], c, S.bc_f[1], p, k, k_on, p_on);
    }
    if (tid != 0) return;
    if (!bad) {
      const bool in_s = okey_of(xt) >= sr.min_key;
      const float zs = __ull2float_rn(sr.zs) * (1.0f / FX_SCALE);
      restr = in_s ? d - logf(zs) : -INFINITY;
      support = static_cast<int>(sr.support);
    }
  }

  if (tid == 0) {
    if (P.out_full) P.out_full[row] = full;
    if (RESTR && P.out_restr) P.out_restr[row] = restr;
    if (RESTR && P.out_support) P.out_support[row] = support;
    if (P.out_kl) P.out_kl[row] = P.kl_policy_full[row] - full;
    if (timed_out && P.err) atomicAdd(P.err, 1);
  }
}

// ------------------------------------------------------------ host side

thread_local char g_last_error[512] = "";

rlk_status fail(rlk_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

rlk_status check_logits(const void* logits, int64_t T, int64_t stride, const char* what) {
  if (!logits) return fail(RLK_EINVAL, "%s is NULL", what);
  if (stride < VPAD) return fail(RLK_EINVAL, "%s row_stride %lld < %d", what, (long long)stride, VPAD);
  if (!aligned(logits, 16)) return fail(RLK_EALIGN, "%s base is not 16-byte aligned", what);
  if (stride % 8 != 0) return fail(RLK_EALIGN, "%s row_stride %lld is not a multiple of 8", what, (long long)stride);
  (void)T;
  return RLK_OK;
}

rlk_status check_args(const rlk_logp_args* a, bool restr) {
  if (!a) return fail(RLK_EINVAL, "args is NULL");
  if (a->T < 0) return fail(RLK_EINVAL, "T = %lld < 0", (long long)a->T);
  if (a->T >= (int64_t(1) << 28)) return fail(RLK_EINVAL, "T = %lld: at most 2^28 - 1 rows per call", (long long)a->T);
  if (a->vocab_real != VREAL || a->vocab_padded != VPAD)
    return fail(RLK_EINVAL, "vocab sizes must be %d/%d, got %d/%d", VREAL, VPAD, a->vocab_real, a->vocab_padded);
  if (a->T == 0) return RLK_OK;
  rlk_status s = check_logits(a->logits, a->T, a->row_stride, "logits");
  if (s != RLK_OK) return s;
  if (!a->target) return fail(RLK_EINVAL, "target is NULL");
  if (!aligned(a->target, 4)) return fail(RLK_EALIGN, "target is not 4-byte aligned");
  if (a->temperature) {
    if (!aligned(a->temperature, 4)) return fail(RLK_EALIGN, "temperature is not 4-byte aligned");
  } else if (!(a->temperature_scalar >= 0.0f && a->temperature_scalar <= 3.402823466e38f)) {
    return fail(RLK_EINVAL, "temperature %g must be finite and >= 0", (double)a->temperature_scalar);
  }
  if (restr) {
    if (a->top_p) {
      if (!aligned(a->top_p, 4)) return fail(RLK_EALIGN, "top_p is not 4-byte aligned");
    } else if (!(a->top_p_scalar > 0.0f && a->top_p_scalar <= 1.0f)) {
      return fail(RLK_EINVAL, "top_p %g must be in (0, 1]", (double)a->top_p_scalar);
    }
    if (a->top_k) {
      if (!aligned(a->top_k, 4)) return fail(RLK_EALIGN, "top_k is not 4-byte aligned");
    } else if (!(a->top_k_scalar == -1 || (a->top_k_scalar >= 1 && a->top_k_scalar <= VREAL))) {
      return fail(RLK_EINVAL, "top_k %d must be -1 or 1..%d", a->top_k_scalar, VREAL);
    }
  }
  if (a->err_count && !aligned(a->err_count, 4)) return fail(RLK_EALIGN, "err_count is not 4-byte aligned");
  return RLK_OK;
}

rlk_status check_out(const void* p, const char* what, bool required) {
  if (!p) return required ? fail(RLK_EINVAL, "%s is NULL", what) : RLK_OK;
  if (!aligned(p, 4)) return fail(RLK_EALIGN, "%s is not 4-byte aligned", what);
  return RLK_OK;
}

KParams make_params(const rlk_logp_args* a) {
  KParams P;
  memset(&P, 0, sizeof(P));
  P.logits = static_cast<const uint16_t*>(a->logits);
  P.stride = a->row_stride;
  P.target = a->target;
  P.tau_arr = a->temperature;
  P.p_arr = a->top_p;
  P.k_arr = a->top_k;
  P.tau_s = a->temperature_scalar;
  P.p_s = a->top_p_scalar;
  P.k_s = a->top_k_scalar;
  P.err = a->err_count;
  return P;
}

template <bool RESTR>
rlk_status launch(const KParams& P, int64_t T, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(logp_kernel<RESTR>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = cudaFuncSetAttribute(logp_kernel<RESTR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(Smem)));
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  const dim3 grid(static_cast<unsigned>(T * NSHARD));
  logp_kernel<RESTR><<<grid, NTHR, sizeof(Smem), stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

}  // namespace rlk

using namespace rlk;

extern "C" {

rlk_status rlk_logp_full(const rlk_logp_args* args, float* out_full, void* stream) {
  rlk_status s = check_args(args, false);
  if (s != RLK_OK || args->T == 0) return s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  KParams P = make_params(args);
  P.out_full = out_full;
  return launch<false>(P, args->T, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_logp_pair(const rlk_logp_args* args, float* out_full, float* out_restr,
                         int32_t* out_support, void* stream) {
  rlk_status s = check_args(args, true);
  if (s != RLK_OK || args->T == 0) return s;
  if (!out_full && !out_restr) return fail(RLK_EINVAL, "out_full and out_restr are both NULL");
  if ((s = check_out(out_full, "out_full", false)) != RLK_OK) return s;
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  KParams P = make_params(args);
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  return launch<true>(P, args->T, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_logp_restricted(const rlk_logp_args* args, float* out_restr, int32_t* out_support,
                               void* stream) {
  if (args && args->T > 0 && !out_restr) return fail(RLK_EINVAL, "out_restr is NULL");
  return rlk_logp_pair(args, nullptr, out_restr, out_support, stream);
}

rlk_status rlk_logp_kl(const rlk_logp_args* policy, const void* ref_logits, int64_t ref_row_stride,
                       float* out_full, float* out_restr, int32_t* out_support,
                       float* out_full_ref, float* out_kl, void* stream) {
  rlk_status s = check_args(policy, true);
  if (s != RLK_OK || policy->T == 0) return s;
  if ((s = check_logits(ref_logits, policy->T, ref_row_stride, "ref_logits")) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  if ((s = check_out(out_full_ref, "out_full_ref", true)) != RLK_OK) return s;
  if ((s = check_out(out_kl, "out_kl", true)) != RLK_OK) return s;
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KParams P = make_params(policy);
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  if ((s = launch<true>(P, policy->T, st)) != RLK_OK) return s;
  KParams R = make_params(policy);
  R.logits = static_cast<const uint16_t*>(ref_logits);
  R.stride = ref_row_stride;
  R.out_full = out_full_ref;
  R.kl_policy_full = out_full;
  R.out_kl = out_kl;
  R.err = nullptr;   // the policy pass already counted rejected rows
  return launch<false>(R, policy->T, st);
}

rlk_status rlk_logp_kl_ref(const rlk_logp_args* ref, const float* full_policy,
                           float* out_full_ref, float* out_kl, void* stream) {
  rlk_status s = check_args(ref, false);
  if (s != RLK_OK || ref->T == 0) return s;
  if ((s = check_out(full_policy, "full_policy", true)) != RLK_OK) return s;
  if ((s = check_out(out_full_ref, "out_full_ref", true)) != RLK_OK) return s;
  if ((s = check_out(out_kl, "out_kl", true)) != RLK_OK) return s;
  KParams R = make_params(ref);
  R.out_full = out_full_ref;
  R.kl_policy_full = full_policy;
  R.out_kl = out_kl;
  return launch<false>(R, ref->T, static_cast<cudaStream_t>(stream));
}

const char* rlk_status_string(rlk_status status) {
  switch (status) {
    case RLK_OK: return "ok";
    case RLK_EINVAL: return "invalid argument";
    case RLK_EALIGN: return "misaligned pointer or stride";
    case RLK_ECUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* rlk_last_error(void) { return g_last_error; }

int rlk_abi_version(void) { return RLK_ABI_VERSION; }

}  // extern "C"
