// rlk_shard.cu -- the vocabulary-sharded form of the strict token logprob.
//
// Each shard of the fixed virtual TP8 partition sits in its own buffer, as a
// tensor-parallel rank would hold it.  Every shard yields a summary and the
// summaries combine in one fixed order of vocabulary position (Reproduce and
// profile the Qwen3-8B TP4/CP2 experiment, "How non-default CUDA topology
// reuses TP4/CP2"):
//
//   phase 1  shard_summary_kernel, one CTA per row of one shard: the same
//            max pass, top-k witness, greedy/NaN scan and fixed-tree sum-exp
//            as a CTA of the fused kernel, so the (max, sum-exp) pair has the
//            same bits;
//   phase 2  shard_counts_kernel: the row's candidate window from the 8
//            gathered summaries (candidate_window, as in the fused kernel)
//            and the exact per-key counts of this shard's tokens in it;
//   merge    merge_kernel, one warp per row: the left fold over shard index
//            of the fused kernel's leader, then the same warp selection on
//            the summed counts.
//
// The fused kernel resolves a support that reaches below the window by
// re-reading the row; a shard cannot, so rlk_logp_merge reports such rows
// (support -2).  The resumable pair continues them instead:
//
//   merge_kernel<true, true>  the merge with a per-row state: a row whose
//            threshold lies below the window records the next window (and
//            the exact integer carries above it) and stays pending;
//   window_counts_kernel      exact per-key counts of this shard's tokens on
//            each pending row's next window;
//
// repeated by the caller until no row is pending.  The windows and carries
// are those of the fused kernel's fallback (select_support), so the
// results are the same bits.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "rlk_logp.h"
#include "rlk_device.cuh"
#include "rlk_host.h"

namespace rlk {

// The shard's copy comes last: the counts kernel, given phase 1's chunk
// maxima, reads its few chunks from global memory and is launched without it.
struct __align__(128) ShardSmem {
  uint32_t hist[WIN];              // counts kernel: per-key counts of this shard
  uint32_t red_u[NWARP];
  int32_t red_i[NWARP];
  float red_f[NWARP];
  unsigned long long bar_load;
  alignas(128) uint4 shard[SHARD_CHUNKS];
};
constexpr size_t SHARD_SMEM_NO_COPY = offsetof(ShardSmem, shard);
// the counts kernel given chunk maxima copies the row's maxima (2 bytes per
// chunk) into the start of the shard area
constexpr uint32_t CMAX_ROW_BYTES = SHARD_CHUNKS * 2u;
static_assert(CMAX_ROW_BYTES % 16u == 0u, "bulk copies move 16-byte multiples");
static_assert(sizeof(ShardSmem) + 1024 <= 233472 / CTAS_PER_SM, "shared memory budget of 5 CTAs per SM");

struct ShardParams {
  const uint16_t* logits;
  int64_t stride;
  int64_t T;
  int shard;
  const int32_t* target;
  const float* tau_arr;
  const float* p_arr;
  const int32_t* k_arr;
  float tau_s, p_s;
  int32_t k_s;
  // phase 1 outputs
  float* out_max;
  float* out_sumexp;
  int32_t* out_aux;
  float* out_xt;
  uint16_t* out_cmax;           // optional: per 16-byte chunk, its maximum (bf16 bits), [T][SHARD_CHUNKS]
  // phase 2: gathered summaries in, counts out
  const uint16_t* in_cmax;      // optional: phase 1's chunk maxima (only the chunks reaching
                                // the window are then read)
  const float* g_max;
  const float* g_sumexp;
  const int32_t* g_aux;
  uint32_t* out_counts;
  int32_t* err;
};

struct RowParams {
  float tau, p;
  int k, t;
  bool valid, greedy, k_on, p_on;
};

// The row's parameters and the validity rule of the fused kernel.
__device__ __forceinline__ RowParams row_params(const float* tau_arr, float tau_s, const float* p_arr,
                                                float p_s, const int32_t* k_arr, int32_t k_s,
                                                const int32_t* target, int64_t row) {
  RowParams rp;
  rp.tau = tau_arr ? tau_arr[row] : tau_s;
  rp.p = p_arr ? p_arr[row] : p_s;
  rp.k = k_arr ? k_arr[row] : k_s;
  rp.t = target[row];
  rp.valid = (rp.tau >= 0.0f) && (rp.tau <= 3.402823466e38f) && (rp.p > 0.0f) && (rp.p <= 1.0f) &&
             (rp.k == -1 || (rp.k >= 1 && rp.k <= VREAL)) && (rp.t >= 0) && (rp.t < VREAL);
  rp.greedy = (rp.tau == 0.0f);
  rp.k_on = (rp.k != -1) && (rp.k < VREAL);
  rp.p_on = (rp.p < 1.0f);
  return rp;
}

// Thread 0 starts the bulk copy of one shard row into shared memory.
__device__ __forceinline__ void load_shard_row(ShardSmem& S, const uint16_t* rowp, int nchunks) {
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_addr(&S.bar_load);
    mbar_init(bar, 1);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = static_cast<uint32_t>(nchunks) * 16u;
    mbar_arrive_expect_tx(bar, bytes);
    const uint64_t pol = evict_first_policy();
    const uint32_t piece = bytes / TMA_PIECES;
    const char* src = reinterpret_cast<const char*>(rowp);
    const uint32_t dst = smem_addr(S.shard);
#pragma unroll
    for (int i = 0; i < TMA_PIECES; ++i) bulk_load(dst + i * piece, src + i * piece, piece, bar, pol);
  }
}

// ------------------------------------------------------------ phase 1

__global__ void __launch_bounds__(NTHR, CTAS_PER_SM) shard_summary_kernel(const ShardParams P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ShardSmem& S = *reinterpret_cast<ShardSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int r = P.shard;
  const int nchunks = (r == NSHARD - 1) ? LAST_CHUNKS : SHARD_CHUNKS;
  const uint32_t bar = smem_addr(&S.bar_load);
  load_shard_row(S, P.logits + row * P.stride, nchunks);

  const RowParams rp = row_params(P.tau_arr, P.tau_s, P.p_arr, P.p_s, P.k_arr, P.k_s, P.target, row);
  const float qnan = __int_as_float(0x7fc00000);
  if (!rp.valid) {
    if (tid == 0) {
      mbar_wait_bounded(bar);   // the copy writes this CTA's shared memory: let it land
      P.out_max[row] = qnan;
      P.out_sumexp[row] = qnan;
      P.out_aux[row] = 0;
      if (r == 0 && P.err) atomicAdd(P.err, 1);
    }
    return;
  }
  __syncthreads();              // barrier initialised before anyone waits on it
  bool bad = false;
  if (!mbar_wait_bounded(bar)) {
    bad = true;
    mbar_wait_bounded(bar);     // give copies in flight a second bounded chance to land
  }

  const uint4* sh = S.shard;
  __nv_bfloat162 cm[MAXCH];
  const int tkey = pass_max(sh, tid, nchunks, cm);
  if (P.out_cmax) {
    // each chunk's maximum, for phase 2 to read only the chunks reaching the window
    uint16_t* dst = P.out_cmax + row * SHARD_CHUNKS;
#pragma unroll
    for (int i = 0; i < MAXCH; ++i) {
      const int ch = tid + i * NTHR;
      if (ch < nchunks)
        dst[ch] = __bfloat16_as_ushort(__hmax(__low2bfloat16(cm[i]), __high2bfloat16(cm[i])));
    }
  }
  const int kw = (rp.k + ROW_WARPS - 1) / ROW_WARPS;
  const bool k_bound = !rp.greedy && rp.k_on && kw <= 32;
  stage_max_bound(tkey, k_bound ? kw : 0, S);
  __syncthreads();
  unsigned xkey = S.red_u[0];
  int lkey = S.red_i[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) { xkey = max(xkey, S.red_u[w]); lkey = min(lkey, S.red_i[w]); }
  const float xm = key_value(static_cast<int>(xkey));
  const bool xm_finite = (xm > -INFINITY) && (xm < INFINITY);
  if (xm != xm) bad = true;     // a thread whose every element is NaN

  uint32_t first = 0x7fffffffu;
  if (rp.greedy || xm == -INFINITY) {
    // greedy: first column of this shard holding its maximum; both: NaN scan
    bool nan_seen;
    int f = scan_nan_first(sh, tid, nchunks, cm, xm, rp.greedy, nan_seen);
    if (__syncthreads_or(nan_seen)) bad = true;
    if (rp.greedy) {
      f = block_min_int(f, S);
      if (f != 0x7fffffff) first = static_cast<uint32_t>(f + r * SW);
    }
  }
  float l = 0.0f;
  if (!rp.greedy && xm_finite) l = block_sum_fixed(pass_sumexp(sh, tid, nchunks, xm, __fdiv_rn(LOG2E, rp.tau)), S);
  if (tid == 0) {
    P.out_max[row] = xm;
    P.out_sumexp[row] = bad ? qnan : l;
    P.out_aux[row] = rp.greedy ? static_cast<int32_t>(first) : (k_bound ? lkey : 0);
    const int local_t = rp.t - r * SW;
    if (local_t >= 0 && local_t < nchunks * 8) {
      const uint16_t* elem = reinterpret_cast<const uint16_t*>(S.shard);
      P.out_xt[row] = __uint_as_float(static_cast<uint32_t>(elem[local_t]) << 16);
    }
  }
}

// ------------------------------------------------------------ phase 2

// The row's candidate window from the gathered summaries: maximum and top-k
// witness folded over the shards, and for top-p-only rows the total mass Z
// folded in shard order exactly as the fused kernel folds the exchanged
// sum-exps.  Also returns M.
__device__ __forceinline__ void gathered_window(const float* g_max, const float* g_sumexp,
                                                const int32_t* g_aux, int64_t T, int64_t row,
                                                const RowParams& rp, float& M, int& hi, int& lo) {
  int L = 0x7fffffff;
  M = -INFINITY;
#pragma unroll
  for (int q = 0; q < NSHARD; ++q) {
    M = fmaxf(M, g_max[q * T + row]);
    L = min(L, g_aux[q * T + row]);
  }
  float Z = 0.0f;
  if (!rp.k_on) {
    const float cz = __fdiv_rn(LOG2E, rp.tau);
#pragma unroll
    for (int q = 0; q < NSHARD; ++q) {
      const float xq = g_max[q * T + row];
      if (xq > -INFINITY) Z = fmaf(g_sumexp[q * T + row], ex2((xq - M) * cz), Z);
    }
  }
  candidate_window(M, L, Z, rp.tau, rp.p, rp.k_on, hi, lo);
}

// CMAX: phase 1's chunk maxima are given; the kernel then reads only the
// chunks that reach the window, from global memory, holds no shard copy and
// runs more blocks per SM to cover the load latency.
template <bool CMAX>
__global__ void __launch_bounds__(NTHR, CMAX ? 16 : CTAS_PER_SM) shard_counts_kernel(const ShardParams P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ShardSmem& S = *reinterpret_cast<ShardSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int r = P.shard;
  const int nchunks = (r == NSHARD - 1) ? LAST_CHUNKS : SHARD_CHUNKS;
  const uint32_t bar = smem_addr(&S.bar_load);
  if (CMAX && tid == 0) {
    // the row's chunk maxima go out first, while the window is formed from
    // the gathered summaries (every row waits for the copy before it ends)
    mbar_init(bar, 1);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, CMAX_ROW_BYTES);
    bulk_load(smem_addr(S.shard), P.in_cmax + row * SHARD_CHUNKS, CMAX_ROW_BYTES, bar, evict_first_policy());
  }
  const RowParams rp = row_params(P.tau_arr, P.tau_s, P.p_arr, P.p_s, P.k_arr, P.k_s, P.target, row);
  const bool sel = rp.valid && !rp.greedy && (rp.k_on || rp.p_on);
  for (int i = tid; i < WIN; i += NTHR) S.hist[i] = 0u;
  if (sel) {
    float M;
    int hi, lo;
    gathered_window(P.g_max, P.g_sumexp, P.g_aux, P.T, row, rp, M, hi, lo);
    // the fused kernel's CTA counts only if its shard maximum is finite and
    // reaches the window
    const float xm = P.g_max[static_cast<int64_t>(r) * P.T + row];
    const bool count = (xm > -INFINITY) && (xm < INFINITY) && lo <= hi && okey_of(xm) >= lo;
    if (CMAX && count) {
      // phase 1's chunk maxima (copied to shared memory) pick the chunks to
      // read, straight from global memory
      __syncthreads();          // histogram zeroed, copy barrier initialised
      if (!mbar_wait_bounded(bar)) mbar_wait_bounded(bar);
      const float vlo_f = key_value(lo);
      const uint16_t* cmax = reinterpret_cast<const uint16_t*>(S.shard);
      const uint4* rowv = reinterpret_cast<const uint4*>(P.logits + row * P.stride);
      uint32_t hit = 0;
#pragma unroll
      for (int i = 0; i < MAXCH; ++i) {
        const int ch = tid + i * NTHR;
        if (ch < nchunks && __uint_as_float(static_cast<uint32_t>(cmax[ch]) << 16) >= vlo_f)
          hit |= 1u << i;
      }
      while (hit) {
        const int i = __ffs(hit) - 1;
        hit &= hit - 1;
        const uint4 v = __ldg(rowv + tid + i * NTHR);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t b = (w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
          if (__uint_as_float(b << 16) >= vlo_f) red_shared_add(&S.hist[hi - okey(b)], 1u);
        }
      }
    } else if (!CMAX && count) {
      const uint32_t bar = smem_addr(&S.bar_load);
      load_shard_row(S, P.logits + row * P.stride, nchunks);
      __syncthreads();          // barrier initialised and histogram zeroed
      if (!mbar_wait_bounded(bar)) mbar_wait_bounded(bar);
      __nv_bfloat162 cm[MAXCH];
      pass_max(S.shard, tid, nchunks, cm);
      const float vlo_f = key_value(lo);
      const __nv_bfloat162 vlo2 = __floats2bfloat162_rn(vlo_f, vlo_f);
#pragma unroll
      for (int i = 0; i < MAXCH; ++i) {
        // an absent last chunk holds -inf in cm: skip it even when the
        // window's bottom is -inf itself
        if (i == MAXCH - 1 && tid + i * NTHR >= nchunks) continue;
        if (__hge2_mask(cm[i], vlo2) == 0u) continue;
        const uint4 v = S.shard[tid + i * NTHR];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t b = (w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
          if (__uint_as_float(b << 16) >= vlo_f) red_shared_add(&S.hist[hi - okey(b)], 1u);
        }
      }
    }
    if (!count && xm == -INFINITY && lo <= KEY_NEG_INF && lo <= hi) {
      // every element of this shard is -inf and the window reaches -inf: the
      // whole shard counts at that key (as in the fused kernel)
      __syncthreads();          // the histogram is zeroed
      if (tid == 0) S.hist[hi - KEY_NEG_INF] = static_cast<uint32_t>(nchunks) * 8u;
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(P.out_counts + row * WIN);
  const uint4* src = reinterpret_cast<const uint4*>(S.hist);
  for (int i = tid; i < WIN / 4; i += NTHR) dst[i] = src[i];
  // the chunk-maxima copy writes this CTA's shared memory: it lands before the CTA ends
  if (CMAX && tid == 0 && !mbar_wait_bounded(bar)) mbar_wait_bounded(bar);
}

// ------------------------------------------------------------ lower windows

// Counts of this shard's real tokens on each pending row's next window
// (order keys state.lo .. state.hi, entry i = key state.hi - i), read from
// global memory: every real chunk, or with phase 1's chunk maxima only the
// chunks whose maximum reaches state.lo.  Rows that are not pending get zeros.
template <bool CMAX>
__global__ void __launch_bounds__(NTHR) window_counts_kernel(const ShardParams P,
                                                             const rlk_merge_state* state) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ShardSmem& S = *reinterpret_cast<ShardSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int nchunks = (P.shard == NSHARD - 1) ? LAST_CHUNKS : SHARD_CHUNKS;
  const rlk_merge_state st = state[row];
  for (int i = tid; i < WIN; i += NTHR) S.hist[i] = 0u;
  __syncthreads();
  if ((st.stage == 1 || st.stage == 2) && st.lo <= st.hi && st.hi - st.lo < WIN) {
    const uint4* rowv = reinterpret_cast<const uint4*>(P.logits + row * P.stride);
    const uint16_t* cmax = CMAX ? P.in_cmax + row * SHARD_CHUNKS : nullptr;
    for (int ch = tid; ch < nchunks; ch += NTHR) {
      if (CMAX && okey(__ldg(cmax + ch)) < st.lo) continue;
      const uint4 v = __ldg(rowv + ch);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int K = okey((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu);
        if (K >= st.lo && K <= st.hi) red_shared_add(&S.hist[st.hi - K], 1u);
      }
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(P.out_counts + row * WIN);
  const uint4* src = reinterpret_cast<const uint4*>(S.hist);
  for (int i = tid; i < WIN / 4; i += NTHR) dst[i] = src[i];
}

// ------------------------------------------------------------ merge

struct MergeParams {
  const float* g_max;
  const float* g_sumexp;
  const int32_t* g_aux;
  const float* xt;
  int64_t T;
  const int32_t* target;
  const float* tau_arr;
  const float* p_arr;
  const int32_t* k_arr;
  float tau_s, p_s;
  int32_t k_s;
  const uint32_t* counts;
  int count_shards;
  float* out_full;
  float* out_restr;
  int32_t* out_support;
  rlk_merge_state* state;       // resumable merge: per-row state
  int32_t* out_pending;
};

constexpr int MERGE_ROWS = NTHR / 32;   // one warp per row

// One window of the resumable selection, on one warp: keys hi, hi - 1, ...
// with per-key counts cnt[i] and masses count * qfx(key).  Finds the first
// index i < nlim whose condition holds, given the counts and masses (rc, rm)
// of the keys before it plus the carry:
//   topk:  rc < k and (rc + c_i >= k, or i is the row's last key (last));
//   else:  rm < T and (rm + m_i >= T, or i == nlim - 1 and last).
// Returns i with (rc + c_i, rm + m_i) in fc, fm; or -1, after adding the
// totals of keys 0 .. nlim - 1 to the carry.
__device__ __forceinline__ int window_find(const uint32_t* cnt, int nlim, int hi, float M, float c,
                                           bool topk, uint32_t k, unsigned long long T, bool last,
                                           uint32_t& carry_c, unsigned long long& carry_m,
                                           uint32_t& fc, unsigned long long& fm) {
  constexpr int KPL = 4, BLK = 32 * KPL;
  const int lane = threadIdx.x & 31;
  for (int b0 = 0; b0 < nlim; b0 += BLK) {
    uint32_t cj[KPL], lc = 0;
    unsigned long long mj[KPL], lm = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      const int i = b0 + KPL * lane + j;
      cj[j] = (i < nlim) ? cnt[i] : 0u;
      mj[j] = cj[j] ? cj[j] * qfx(key_value(hi - i), M, c) : 0ull;
      lc += cj[j];
      lm += mj[j];
    }
    const uint32_t ic = warp_incl_scan_u32(lc);
    const unsigned long long im = warp_incl_scan_u64(lm);
    uint32_t rc = carry_c + ic - lc;
    unsigned long long rm = carry_m + im - lm;
    int f = -1;
    uint32_t f_c = 0;
    unsigned long long f_m = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      const int i = b0 + KPL * lane + j;
      const bool at_last = last && i == nlim - 1;
      const bool hit = topk ? (rc < k && (rc + cj[j] >= k || at_last))
                            : (rm < T && (rm + mj[j] >= T || at_last));
      if (f < 0 && i < nlim && hit) {
        f = i;
        f_c = rc + cj[j];
        f_m = rm + mj[j];
      }
      rc += cj[j];
      rm += mj[j];
    }
    const unsigned bal = __ballot_sync(0xffffffffu, f >= 0);
    if (bal) {
      const int src = __ffs(bal) - 1;
      fc = __shfl_sync(0xffffffffu, f_c, src);
      fm = __shfl_sync(0xffffffffu, f_m, src);
      return __shfl_sync(0xffffffffu, f, src);
    }
    carry_c += __shfl_sync(0xffffffffu, ic, 31);
    carry_m += __shfl_sync(0xffffffffu, im, 31);
  }
  return -1;
}

// One step of the fallback selection over lower windows (the fused kernel's
// select_support, one window per call): top-k from the top window down to
// the k-th largest value, then the nucleus from the top window down to its
// threshold.  cnt holds the counts of the window st names; (hi0, lo0) is the
// row's first window.  Returns true with the result when the row is
// resolved, else advances st to the window to count next.
__device__ __forceinline__ bool resume_select(const uint32_t* cnt, rlk_merge_state& st, int hi0,
                                              int lo0, float M, float c, float p, int k, bool p_on,
                                              SelResult& out) {
  const int n = st.hi - st.lo + 1;
  uint32_t fc = 0;
  unsigned long long fm = 0;
  unsigned long long carry_m = st.carry_m;
  if (st.stage == 1) {
    const int f = window_find(cnt, n, st.hi, M, c, true, static_cast<uint32_t>(k), 0ull, st.lo == 0,
                              st.carry_c, carry_m, fc, fm);
    st.carry_m = carry_m;
    if (f >= 0) {
      if (!p_on) {
        out = SelResult{fc, fm, st.hi - f};
        return true;
      }
      // the nucleus inside the top-k set, from the top window again
      st.vk_key = st.hi - f;
      st.zk = fm;
      st.stage = 2;
      st.hi = hi0;
      st.lo = lo0;
      st.carry_c = 0;
      st.carry_m = 0;
      return false;
    }
    if (st.lo == 0) {                       // not reached: the last key always resolves
      out = SelResult{st.carry_c, st.carry_m, 0};
      return true;
    }
  } else {
    const unsigned long long T = nucleus_bound(p, st.zk);
    const bool k_in = st.vk_key >= st.lo;
    const int nlim = k_in ? st.hi - st.vk_key + 1 : n;
    const bool bounded = k_in || st.lo == 0;
    const int f = window_find(cnt, nlim, st.hi, M, c, false, 0u, T, bounded, st.carry_c, carry_m,
                              fc, fm);
    st.carry_m = carry_m;
    if (f >= 0) {
      out = SelResult{fc, fm, st.hi - f};
      return true;
    }
    if (bounded) {                          // not reached: the bound always resolves
      out = SelResult{st.carry_c, st.carry_m, st.lo};
      return true;
    }
  }
  st.hi = st.lo - 1;
  st.lo = max(0, st.hi - (WIN - 1));
  return false;
}

template <bool RESTR, bool RESUME = false>
__global__ void __launch_bounds__(NTHR) merge_kernel(const MergeParams P) {
  __shared__ uint32_t cnt[MERGE_ROWS][WIN];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * MERGE_ROWS + warp;
  if (row >= P.T) return;
  rlk_merge_state st{};
  if (RESUME) {
    st = P.state[row];
    if (st.stage == 3) return;              // resolved by an earlier call
  }
  bool pending = false;
  const int64_t T = P.T;
  const RowParams rp = row_params(P.tau_arr, P.tau_s, P.p_arr, P.p_s, P.k_arr, P.k_s, P.target, row);
  const float qnan = __int_as_float(0x7fc00000);
  float full = qnan, restr = qnan;
  int support = -1;
  if (rp.valid) {
    const bool sel = RESTR && !rp.greedy && (rp.k_on || rp.p_on);
    bool bad = false;
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < NSHARD; ++q) {
      const float xq = P.g_max[q * T + row];
      const float lq = P.g_sumexp[q * T + row];
      if (xq == INFINITY || xq != xq || lq != lq) bad = true;
      M = fmaxf(M, xq);
    }
    bad |= !(M > -INFINITY);
    const float c = rp.greedy ? 0.0f : __fdiv_rn(LOG2E, rp.tau);
    float Z = 0.0f, d = 0.0f;
    const float xt = P.xt[row];
    if (!bad && rp.greedy) {
      uint32_t amax = 0x7fffffffu;
#pragma unroll
      for (int q = NSHARD - 1; q >= 0; --q)
        if (P.g_max[q * T + row] == M) amax = static_cast<uint32_t>(P.g_aux[q * T + row]);
      full = restr = (static_cast<uint32_t>(rp.t) == amax) ? 0.0f : -INFINITY;
      support = 1;
    } else if (!bad) {
      if (isinf(__fdiv_rn(M, rp.tau))) {
        bad = true;
      } else {
#pragma unroll
        for (int q = 0; q < NSHARD; ++q) {
          const float xq = P.g_max[q * T + row];
          if (xq > -INFINITY) Z = fmaf(P.g_sumexp[q * T + row], ex2((xq - M) * c), Z);
        }
        d = __fdiv_rn(xt - M, rp.tau);
        full = d - logf(Z);
        restr = full;
        support = VREAL;
      }
    }
    if (sel && !bad) {
      float Mw;
      int hi, lo;
      gathered_window(P.g_max, P.g_sumexp, P.g_aux, T, row, rp, Mw, hi, lo);
      // the window these counts cover: the first one, or the one the state names
      const bool first = !RESUME || st.stage == 0;
      const int whi = first ? hi : st.hi, wlo = first ? lo : st.lo;
      const int n = whi - wlo + 1;
      for (int i = lane; i < n; i += 32) {
        uint32_t sum = 0;
        for (int q = 0; q < P.count_shards; ++q) sum += P.counts[(q * T + row) * WIN + i];
        cnt[warp][i] = sum;
      }
      __syncwarp();
      SelResult sr{0u, 0ull, 0};
      bool done = first && n > 0 && select_warp(cnt[warp], hi, lo, M, c, Z, rp.p, rp.k, rp.k_on, rp.p_on, sr);
      if (RESUME && !done && n > 0) {
        if (first) {
          // as the fused kernel's fallback: top-k (or the nucleus) from the top window
          st.stage = rp.k_on ? 1 : 2;
          st.hi = hi;
          st.lo = lo;
          st.vk_key = -1;
          st.carry_c = 0;
          st.carry_m = 0;
          st.zk = rp.k_on ? 0ull : __float2ull_rn(Z * FX_SCALE);
        }
        done = resume_select(cnt[warp], st, hi, lo, M, c, rp.p, rp.k, rp.p_on, sr);
        pending = !done;
      }
      if (done) {
        const bool in_s = okey_of(xt) >= sr.min_key;
        const float zs = __ull2float_rn(sr.zs) * (1.0f / FX_SCALE);
        restr = in_s ? d - logf(zs) : -INFINITY;
        support = static_cast<int>(sr.support);
      } else {
        restr = qnan;           // the support reaches below this window
        support = -2;
      }
    }
  }
  if (RESUME && lane == 0) {
    if (!pending) st.stage = 3;
    P.state[row] = st;
    if (pending && P.out_pending) atomicAdd(P.out_pending, 1);
  }
  if (lane == 0) {
    P.out_full[row] = full;
    if (RESTR) {
      if (P.out_restr) P.out_restr[row] = restr;
      if (P.out_support) P.out_support[row] = support;
    }
  }
}

// ------------------------------------------------------------ host side

rlk_status check_shard_args(const rlk_shard_args* a) {
  if (!a) return fail(RLK_EINVAL, "args is NULL");
  if (a->T < 0 || a->T >= (int64_t(1) << 31)) return fail(RLK_EINVAL, "T = %lld out of range [0, 2^31)", (long long)a->T);
  if (a->shard < 0 || a->shard >= NSHARD) return fail(RLK_EINVAL, "shard %d must be 0..%d", a->shard, NSHARD - 1);
  if (a->T == 0) return RLK_OK;
  if (!a->logits) return fail(RLK_EINVAL, "logits is NULL");
  if (a->row_stride < SW) return fail(RLK_EINVAL, "row_stride %lld < %d", (long long)a->row_stride, SW);
  if (!aligned(a->logits, 16)) return fail(RLK_EALIGN, "logits base is not 16-byte aligned");
  if (a->row_stride % 8 != 0) return fail(RLK_EALIGN, "row_stride %lld is not a multiple of 8", (long long)a->row_stride);
  if (!a->target) return fail(RLK_EINVAL, "target is NULL");
  if (!aligned(a->target, 4)) return fail(RLK_EALIGN, "target is not 4-byte aligned");
  rlk_status s;
  if ((s = check_tau(a->temperature, a->temperature_scalar)) != RLK_OK) return s;
  if ((s = check_top_p(a->top_p, a->top_p_scalar)) != RLK_OK) return s;
  if ((s = check_top_k(a->top_k, a->top_k_scalar)) != RLK_OK) return s;
  if (a->err_count && !aligned(a->err_count, 4)) return fail(RLK_EALIGN, "err_count is not 4-byte aligned");
  return RLK_OK;
}

ShardParams make_shard_params(const rlk_shard_args* a) {
  ShardParams P;
  memset(&P, 0, sizeof(P));
  P.logits = static_cast<const uint16_t*>(a->logits);
  P.stride = a->row_stride;
  P.T = a->T;
  P.shard = a->shard;
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

template <int WHICH>
rlk_status launch_shard(void (*kernel)(ShardParams), const ShardParams& P, cudaStream_t stream) {
  static bool configured_by_kind[2][64] = {};
  bool* configured = configured_by_kind[(WHICH == 1 && P.in_cmax) ? 1 : 0];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(ShardSmem)));
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  // the counts kernel with chunk maxima never touches the shard copy
  const size_t smem = (WHICH == 1 && P.in_cmax) ? SHARD_SMEM_NO_COPY + CMAX_ROW_BYTES : sizeof(ShardSmem);
  kernel<<<static_cast<unsigned>(P.T), NTHR, smem, stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

}  // namespace rlk

using namespace rlk;

extern "C" {

rlk_status rlk_logp_shard_summary(const rlk_shard_args* args, float* out_max, float* out_sumexp,
                                  int32_t* out_aux, float* out_target_logit, uint16_t* out_chunk_max,
                                  void* stream) {
  rlk_status s = check_shard_args(args);
  if (s != RLK_OK || args->T == 0) return s;
  if ((s = check_out(out_max, "out_max", true)) != RLK_OK) return s;
  if ((s = check_out(out_sumexp, "out_sumexp", true)) != RLK_OK) return s;
  if ((s = check_out(out_aux, "out_aux", true)) != RLK_OK) return s;
  if ((s = check_out(out_target_logit, "out_target_logit", true)) != RLK_OK) return s;
  ShardParams P = make_shard_params(args);
  P.out_max = out_max;
  P.out_sumexp = out_sumexp;
  P.out_aux = out_aux;
  P.out_xt = out_target_logit;
  if (out_chunk_max && !aligned(out_chunk_max, 16))
    return fail(RLK_EALIGN, "out_chunk_max is not 16-byte aligned");
  P.out_cmax = out_chunk_max;
  return launch_shard<0>(shard_summary_kernel, P, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_logp_shard_counts(const rlk_shard_args* args, const float* maxes,
                                 const float* sumexps, const int32_t* aux,
                                 const uint16_t* chunk_max, uint32_t* out_counts, void* stream) {
  rlk_status s = check_shard_args(args);
  if (s != RLK_OK || args->T == 0) return s;
  if ((s = check_out(maxes, "maxes", true)) != RLK_OK) return s;
  if ((s = check_out(sumexps, "sumexps", true)) != RLK_OK) return s;
  if ((s = check_out(aux, "aux", true)) != RLK_OK) return s;
  if (!out_counts) return fail(RLK_EINVAL, "out_counts is NULL");
  if (!aligned(out_counts, 16)) return fail(RLK_EALIGN, "out_counts is not 16-byte aligned");
  ShardParams P = make_shard_params(args);
  P.g_max = maxes;
  P.g_sumexp = sumexps;
  P.g_aux = aux;
  P.out_counts = out_counts;
  if (chunk_max && !aligned(chunk_max, 16)) return fail(RLK_EALIGN, "chunk_max is not 16-byte aligned");
  P.in_cmax = chunk_max;
  return chunk_max ? launch_shard<1>(shard_counts_kernel<true>, P, static_cast<cudaStream_t>(stream))
                   : launch_shard<1>(shard_counts_kernel<false>, P, static_cast<cudaStream_t>(stream));
}

rlk_status rlk_logp_merge(const float* maxes, const float* sumexps, const int32_t* aux,
                          const float* target_logit, int64_t T, const int32_t* target,
                          const float* temperature, float temperature_scalar,
                          const float* top_p, float top_p_scalar,
                          const int32_t* top_k, int32_t top_k_scalar,
                          const uint32_t* counts, int32_t count_shards,
                          float* out_full, float* out_restr, int32_t* out_support,
                          void* stream) {
  if (T < 0 || T >= (int64_t(1) << 31)) return fail(RLK_EINVAL, "T = %lld out of range [0, 2^31)", (long long)T);
  if (T == 0) return RLK_OK;
  rlk_status s;
  if ((s = check_out(maxes, "maxes", true)) != RLK_OK) return s;
  if ((s = check_out(sumexps, "sumexps", true)) != RLK_OK) return s;
  if ((s = check_out(aux, "aux", true)) != RLK_OK) return s;
  if ((s = check_out(target_logit, "target_logit", true)) != RLK_OK) return s;
  if ((s = check_out(target, "target", true)) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  if ((s = check_tau(temperature, temperature_scalar)) != RLK_OK) return s;
  const bool restr = counts != nullptr;
  if (restr) {
    if (count_shards != 1 && count_shards != NSHARD)
      return fail(RLK_EINVAL, "count_shards %d must be 1 or %d", count_shards, NSHARD);
    if (!aligned(counts, 4)) return fail(RLK_EALIGN, "counts is not 4-byte aligned");
    if ((s = check_top_p(top_p, top_p_scalar)) != RLK_OK) return s;
    if ((s = check_top_k(top_k, top_k_scalar)) != RLK_OK) return s;
    if (!out_restr && !out_support) return fail(RLK_EINVAL, "out_restr and out_support are both NULL");
    if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
    if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  }
  MergeParams P;
  memset(&P, 0, sizeof(P));
  P.g_max = maxes;
  P.g_sumexp = sumexps;
  P.g_aux = aux;
  P.xt = target_logit;
  P.T = T;
  P.target = target;
  P.tau_arr = temperature;
  P.tau_s = temperature_scalar;
  P.p_arr = restr ? top_p : nullptr;
  P.p_s = restr ? top_p_scalar : 1.0f;
  P.k_arr = restr ? top_k : nullptr;
  P.k_s = restr ? top_k_scalar : -1;
  P.counts = counts;
  P.count_shards = count_shards;
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  const unsigned grid = static_cast<unsigned>((T + MERGE_ROWS - 1) / MERGE_ROWS);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (restr) merge_kernel<true><<<grid, NTHR, 0, st>>>(P);
  else merge_kernel<false><<<grid, NTHR, 0, st>>>(P);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

rlk_status rlk_logp_merge_resumable(const float* maxes, const float* sumexps, const int32_t* aux,
                                    const float* target_logit, int64_t T, const int32_t* target,
                                    const float* temperature, float temperature_scalar,
                                    const float* top_p, float top_p_scalar,
                                    const int32_t* top_k, int32_t top_k_scalar,
                                    const uint32_t* counts, int32_t count_shards,
                                    rlk_merge_state* state, float* out_full, float* out_restr,
                                    int32_t* out_support, int32_t* out_pending, void* stream) {
  if (T < 0 || T >= (int64_t(1) << 31)) return fail(RLK_EINVAL, "T = %lld out of range [0, 2^31)", (long long)T);
  if (T == 0) return RLK_OK;
  rlk_status s;
  if (!counts) return fail(RLK_EINVAL, "counts is NULL");
  if (!state) return fail(RLK_EINVAL, "state is NULL");
  if (!aligned(state, 8)) return fail(RLK_EALIGN, "state is not 8-byte aligned");
  if ((s = check_out(out_pending, "out_pending", false)) != RLK_OK) return s;
  if ((s = check_out(maxes, "maxes", true)) != RLK_OK) return s;
  if ((s = check_out(sumexps, "sumexps", true)) != RLK_OK) return s;
  if ((s = check_out(aux, "aux", true)) != RLK_OK) return s;
  if ((s = check_out(target_logit, "target_logit", true)) != RLK_OK) return s;
  if ((s = check_out(target, "target", true)) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", true)) != RLK_OK) return s;
  if ((s = check_tau(temperature, temperature_scalar)) != RLK_OK) return s;
  if (count_shards != 1 && count_shards != NSHARD)
    return fail(RLK_EINVAL, "count_shards %d must be 1 or %d", count_shards, NSHARD);
  if (!aligned(counts, 4)) return fail(RLK_EALIGN, "counts is not 4-byte aligned");
  if ((s = check_top_p(top_p, top_p_scalar)) != RLK_OK) return s;
  if ((s = check_top_k(top_k, top_k_scalar)) != RLK_OK) return s;
  if (!out_restr && !out_support) return fail(RLK_EINVAL, "out_restr and out_support are both NULL");
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  MergeParams P;
  memset(&P, 0, sizeof(P));
  P.g_max = maxes;
  P.g_sumexp = sumexps;
  P.g_aux = aux;
  P.xt = target_logit;
  P.T = T;
  P.target = target;
  P.tau_arr = temperature;
  P.tau_s = temperature_scalar;
  P.p_arr = top_p;
  P.p_s = top_p_scalar;
  P.k_arr = top_k;
  P.k_s = top_k_scalar;
  P.counts = counts;
  P.count_shards = count_shards;
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  P.state = state;
  P.out_pending = out_pending;
  const unsigned grid = static_cast<unsigned>((T + MERGE_ROWS - 1) / MERGE_ROWS);
  merge_kernel<true, true><<<grid, NTHR, 0, static_cast<cudaStream_t>(stream)>>>(P);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

rlk_status rlk_logp_shard_counts_window(const rlk_shard_args* args, const rlk_merge_state* state,
                                        const uint16_t* chunk_max, uint32_t* out_counts, void* stream) {
  rlk_status s = check_shard_args(args);
  if (s != RLK_OK || args->T == 0) return s;
  if (!state) return fail(RLK_EINVAL, "state is NULL");
  if (!aligned(state, 8)) return fail(RLK_EALIGN, "state is not 8-byte aligned");
  if (!out_counts) return fail(RLK_EINVAL, "out_counts is NULL");
  if (!aligned(out_counts, 16)) return fail(RLK_EALIGN, "out_counts is not 16-byte aligned");
  if (chunk_max && !aligned(chunk_max, 16)) return fail(RLK_EALIGN, "chunk_max is not 16-byte aligned");
  ShardParams P = make_shard_params(args);
  P.out_counts = out_counts;
  P.in_cmax = chunk_max;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(args->T);
  if (chunk_max)
    window_counts_kernel<true><<<grid, NTHR, SHARD_SMEM_NO_COPY, st>>>(P, state);
  else
    window_counts_kernel<false><<<grid, NTHR, SHARD_SMEM_NO_COPY, st>>>(P, state);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

}  // extern "C"
