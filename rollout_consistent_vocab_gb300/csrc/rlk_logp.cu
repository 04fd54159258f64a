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
//   2. exact shard maximum with packed bf16x2 max, chunk maxima kept in
//      registers, and (top-k rows) each warp's pooled top-k witness;
//   3. shard sum-exp l_r = sum exp(s_j - m_r) in a fixed tree: thread t owns
//      16-byte chunks t, t+128, ... in that order, keeps even and odd columns
//      in the two lanes of a packed f32x2 accumulator, then a shuffle-xor
//      butterfly (IEEE addition is commutative, so every lane ends with the
//      same bits) and a left fold over the 4 warp sums;
//   4. restricted side only: every CTA receives every shard's maximum and
//      witness (and, for top-p-only rows, its sum-exp) over DSMEM, derives
//      the same candidate window of at most 1024 bf16 order keys below the
//      row maximum, and counts its elements in the window into the leader's
//      per-key histogram (remote shared-memory adds, or counts in the CTA's
//      own array pushed once by warps with many candidates);
//   5. the CTA stores its summary (m_r, l_r, aux, flags) into the leader
//      CTA's shared memory.
//
// The leader (rank 0) merges the summaries as a left fold over shard index:
// each vocabulary shard contributes one summary and the summaries combine in
// one fixed order of vocabulary position (Reproduce and profile the Qwen3-8B
// TP4/CP2 experiment, "How non-default CUDA topology reuses TP4/CP2"), and
// finds the top-k and top-p thresholds on the merged histogram.  Masses there
// are per-key exp values times integer counts in 2^-44 fixed point, so every
// sum is an exact integer sum and the support decision cannot depend on
// summation order.  If a threshold lies below the window (a row whose support
// reaches more than 1024 keys under its maximum) the leader re-counts further
// windows from the row in global memory; this path is slow but exact.
//
// Nothing depends on T or on where the row sits: the kernel configuration is
// fixed and every reduction tree is a function of the column index only.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include "rlk_logp.h"
#include "rlk_device.cuh"
#include "rlk_host.h"

namespace rlk {

// Sent by every CTA to every CTA before the candidate pass.
struct __align__(16) MidSlot {
  float xm;        // shard maximum (a bf16 value or -inf / +inf)
  int32_t lkey;    // order key reached by ceil(k/W) lane maxima of every warp of the shard
  uint32_t flags;
  float l;         // unused (0)
};
// Top-p-only rows' second exchange, once the row maximum is known.
struct __align__(16) Mid2Slot {
  float l;         // the shard's sum-exp
  uint32_t unused0, unused1;
  uint32_t flags;
};

// Sent by every CTA to the leader at the end.
struct __align__(16) Summary {
  float xm;        // shard maximum
  float l;         // sum over the shard of exp(s_j - m_r) (NaN if the shard holds a NaN)
  uint32_t aux;    // greedy: first column holding the maximum; otherwise 0
  uint32_t flags;
};

struct __align__(128) Smem {
  uint4 shard[SHARD_CHUNKS];       // 38144 B; the leader reuses it as scratch at the end
  uint32_t merged[WIN];            // leader: per-key candidate counts of the whole row;
                                   // peer: its busy warps' per-key counts, pushed once
  MidSlot mid[NSHARD];
  Mid2Slot mid2[NSHARD];
  Summary slot[NSHARD];
  uint32_t red_u[NWARP];
  int32_t red_i[NWARP];
  float red_f[NWARP];
  uint32_t scan_c[NWARP];
  unsigned long long scan_m[NWARP];
  int32_t found_i;
  uint32_t found_c;
  unsigned long long found_m;
  uint32_t npush;                  // leader: the peers' histogram adds, in 4-byte units
  int32_t win[4];
  float bc_f[4];
  int32_t sel_done;
  alignas(16) uint4 lead;          // backward: the leader's resolution of the row
  unsigned long long bar_load, bar_mid, bar_mid2, bar_sum, bar_hist, bar_lead;
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
  rlk_row_stats* out_stats;     // optional per-row record for a later backward
  // backward
  const float* g_full;          // upstream gradients (NULL: 0)
  const float* g_restr;
  char* grad;                   // [T, grad_stride] bf16 or f32
  int64_t grad_stride;          // elements
  int grad_f32;
  // sampler
  const uint32_t* uniform;      // per-row random words, or NULL for Philox
  const unsigned long long* counter;
  unsigned long long seed;
  int32_t* out_token;
  struct SampMsg* out_samp;     // resolution pass: per-row record for the draw
  const struct SampMsg* in_samp;
  uint32_t* samp_bits;          // resolution pass: per row and shard, the chunks reaching the
                                // candidate window (SAMP_BITWORDS words); NULL: not kept
  // rlk_logp_kl: the reference logits, interleaved with the policy rows
  const uint16_t* ref_logits;
  int64_t ref_stride;
  float* out_full_ref;
};

enum { MODE_FWD = 0, MODE_BWD = 1, MODE_SAMPLE = 2 };

// Sampler: per-row record of the resolved row, written by the leader of the
// pair pass and read by the draw kernel (16 bytes).
enum : uint32_t { SAMP_DRAW = 1u, SAMP_SEL = 2u, SAMP_BITS = 4u, SAMP_WORDS = 8u };
struct __align__(16) SampMsg {
  float M, Z;
  int32_t min_key;
  uint32_t flags;                  // SAMP_DRAW: the row draws (not greedy / NaN); SAMP_SEL: filtered;
                                   // SAMP_BITS: the support lies in the chunks the bitmap marks;
                                   // SAMP_WORDS: an unfiltered row's word masses are in the workspace
};

// Unfiltered rows (every real token in the support) are drawn on float
// masses: relative to its shard's maximum xm_q, an element's mass is
// ex2((x - xm_q) c), a chunk's the fixed tree ((e0+e1)+(e2+e3))+((e4+e5)+
// (e6+e7)), a word's (32 consecutive chunks) a fixed shuffle-down tree over
// its chunks read in lane 0 (as pass_sumexp_words forms them), and each is
// brought to the row maximum M by one product with s_q = ex2((xm_q - M) c).
// The pair pass writes the word masses and xm_q (in the shard's 76th word,
// past its last chunk); the draw recomputes only the chunks of the word it
// lands in, with the same arithmetic.
constexpr int SAMP_XM_WORD = SAMP_BITWORDS - 1;
static_assert(SAMP_XM_WORD * 32 >= SHARD_CHUNKS, "the last word of a shard holds no chunk");
__device__ __forceinline__ float chunk_mass_f(const uint4 v, float M, float c) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float e[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    e[2 * j] = ex2(__fmul_rn(__fsub_rn(bf16_lo(w[j]), M), c));
    e[2 * j + 1] = ex2(__fmul_rn(__fsub_rn(bf16_hi(w[j]), M), c));
  }
  return __fadd_rn(__fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3])),
                   __fadd_rn(__fadd_rn(e[4], e[5]), __fadd_rn(e[6], e[7])));
}
__device__ __forceinline__ float word_sum_lane0(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
  return v;
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

template <bool RESTR, int MODE>
__global__ void __cluster_dims__(NSHARD, 1, 1) __launch_bounds__(NTHR, CTAS_PER_SM)
logp_kernel(const KParams P) {
  constexpr bool BWD = MODE == MODE_BWD;
  constexpr bool SAMPLE = MODE == MODE_SAMPLE;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const uint32_t r = cluster_rank();
  // rlk_logp_kl's single launch: clusters alternate between the policy pair
  // pass of row i and the reference full pass of row i (a latency-bound and a
  // bandwidth-bound workload sharing the SMs)
  const int64_t cid = blockIdx.x / NSHARD;
  const bool pair_kl = MODE == MODE_FWD && P.ref_logits != nullptr;
  const bool is_ref = pair_kl && (cid & 1);
  const int64_t row = pair_kl ? (cid >> 1) : cid;
  float* const o_full = is_ref ? P.out_full_ref : P.out_full;
  float* const o_restr = is_ref ? nullptr : P.out_restr;
  int32_t* const o_support = is_ref ? nullptr : P.out_support;
  int32_t* const o_err = is_ref ? nullptr : P.err;

  const int nchunks = (r == NSHARD - 1) ? LAST_CHUNKS : SHARD_CHUNKS;
  const uint16_t* rowp = is_ref ? P.ref_logits + row * P.ref_stride : P.logits + row * P.stride;
  const uint32_t bar_load = smem_addr(&S.bar_load);
  const uint32_t bar_mid = smem_addr(&S.bar_mid);
  const uint32_t bar_mid2 = smem_addr(&S.bar_mid2);
  const uint32_t bar_sum = smem_addr(&S.bar_sum);
  const uint32_t bar_hist = smem_addr(&S.bar_hist);
  const uint32_t bar_lead = smem_addr(&S.bar_lead);
  char* const gshard = BWD ? P.grad + (row * P.grad_stride + static_cast<int64_t>(r) * SW) *
                                          (P.grad_f32 ? 4 : 2)
                           : nullptr;

  // ---- 1. the bulk copy of the shard into shared memory goes out first
  // (thread 0 also notes the start time, from which the drain deadlines of
  // a timed-out wait are measured)
  const unsigned long long t_start = (tid == 0) ? global_timer() : 0ull;
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
  const float p = (RESTR && !is_ref) ? (P.p_arr ? P.p_arr[row] : P.p_s) : 1.0f;
  const int k = (RESTR && !is_ref) ? (P.k_arr ? P.k_arr[row] : P.k_s) : -1;
  const int t = SAMPLE ? 0 : P.target[row];     // the sampler's pass has no target
  const bool valid = (tau >= 0.0f) && (tau <= 3.402823466e38f) && (p > 0.0f) && (p <= 1.0f) &&
                     (k == -1 || (k >= 1 && k <= VREAL)) && (t >= 0) && (t < VREAL);
  if (!valid) {
    if (tid == 0) {
      // the copy writes this CTA's shared memory: let it land before leaving
      if (!mbar_wait_bounded(bar_load)) mbar_wait_bounded(bar_load);
      if (r == 0) {
        if (o_full) o_full[row] = __int_as_float(0x7fc00000);
        if (RESTR && o_restr) o_restr[row] = __int_as_float(0x7fc00000);
        if (RESTR && o_support) o_support[row] = -1;
        if (P.out_kl) P.out_kl[row] = __int_as_float(0x7fc00000);
        if (P.out_stats) P.out_stats[row] = nan_stats();
        if (SAMPLE) {
          P.out_token[row] = -1;
          P.out_samp[row] = SampMsg{};     // nothing to draw
        }
        if (o_err) atomicAdd(o_err, 1);
      }
    }
    if (BWD)
      write_grad_shard(nullptr, false, nchunks, static_cast<int>(r) * SW, -1, nan_coeffs(), gshard,
                       P.grad_f32 != 0);
    return;
  }
  const bool greedy = (tau == 0.0f);
  const bool k_on = (k != -1) && (k < VREAL);
  const bool p_on = (p < 1.0f);
  const bool sel = RESTR && !greedy && (k_on || p_on);
  // sampler, unfiltered drawing rows: each CTA writes the float mass of every
  // word (32 chunks) of its shard, relative to its own maximum, and that maximum
  const bool wmass = SAMPLE && P.samp_bits != nullptr && !greedy && !sel;
  // ---- barriers that peers signal, and the leader's histogram
  if (tid == 0) {
    mbar_init(bar_mid, 1);
    mbar_init(bar_mid2, 1);
    mbar_init(bar_sum, 1);
    mbar_init(bar_hist, 1);
    // messages from the 7 peers: 16 bytes each
    if (sel) mbar_arrive_expect_tx(bar_mid, (NSHARD - 1) * 16);
    if (sel && !k_on) mbar_arrive_expect_tx(bar_mid2, (NSHARD - 1) * 16);
    // the peers' summaries (16 bytes each) and, on restricted rows, each peer
    // warp's 4-byte add of the number of histogram adds it sent
    if (r == 0)
      mbar_arrive_expect_tx(bar_sum, (NSHARD - 1) * 16 + (sel ? (NSHARD - 1) * NWARP * 4 : 0));
    if (BWD && r != 0) {
      mbar_init(bar_lead, 1);
      mbar_arrive_expect_tx(bar_lead, 16);
    }
    S.npush = 0u;
  }
  if (sel)
    for (int i = tid; i < WIN; i += NTHR) S.merged[i] = 0u;
  __syncthreads();
  // S0: barriers initialised; one thread publishes the initialisations to the
  // cluster and everyone arrives relaxed.  The leader's zeroed histogram
  // needs no fence here: a peer adds to it only after its window wait has
  // acquired, at cluster scope, every exchange message including the
  // leader's, and the leader sends that message after the block barrier
  // above, so the message's release covers the zero stores.
  if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  cluster_arrive_relaxed();
  // the leader needs the target's logit at the end: start the load now
  const float xt = (r == 0 && !SAMPLE) ? __uint_as_float(static_cast<uint32_t>(__ldg(rowp + t)) << 16) : 0.0f;
  uint32_t flags = 0;
  if (!mbar_wait_bounded(bar_load)) {
    flags |= FLAG_TIMEOUT;
    mbar_wait_bounded(bar_load);   // give copies in flight a second bounded chance to land
  }

  // ---- 2. shard maximum; per-chunk maxima stay in registers for the candidate pass.
  // bf16 max ignores NaN; a NaN shows up as a NaN sum-exp (or in the scan below).
  const uint4* sh = S.shard;
  __nv_bfloat162 cm[MAXCH];
  const int tkey = pass_max(sh, tid, nchunks, cm);
  // Pooled top-k bound: warp w certifies kw = ceil(k/W) lane maxima at or above
  // lw (its kw-th largest lane maximum), so the W warps of the row certify
  // W*kw >= k tokens at or above the minimum of lw over the cluster.
  const int kw = (k + ROW_WARPS - 1) / ROW_WARPS;
  const bool k_bound = sel && k_on && kw <= 32;
  stage_max_bound(tkey, k_bound ? kw : 0, S);
  __syncthreads();
  unsigned xkey = S.red_u[0];
  int lkey = S.red_i[0];
#pragma unroll
  for (int w = 1; w < NWARP; ++w) { xkey = max(xkey, S.red_u[w]); lkey = min(lkey, S.red_i[w]); }
  const float xm = key_value(static_cast<int>(xkey));
  const bool xm_finite = (xm > -INFINITY) && (xm < INFINITY);
  // A thread whose every element is NaN has a NaN maximum, whose key sorts
  // above +inf (or below -inf): the shard maximum is then NaN.
  if (xm != xm) flags |= FLAG_NAN;

  uint32_t first = 0x7fffffffu;
  if (greedy || xm == -INFINITY) {
    // greedy: first column of this shard holding its maximum; both cases: NaN scan
    bool nan_seen;
    int f = scan_nan_first(sh, tid, nchunks, cm, xm, greedy, nan_seen);
    if (__syncthreads_or(nan_seen)) flags |= FLAG_NAN;
    if (greedy) {
      f = block_min_int(f, S);
      if (f != 0x7fffffff) first = static_cast<uint32_t>(f + static_cast<int>(r) * SW);
    }
  }

  cluster_wait();              // S0 complete: every CTA's barriers are initialised
  // Restricted rows send their maximum and bound now and overlap the
  // exchange with the sum-exp pass; top-p-only rows then exchange their
  // sum-exp (which sets the candidate window) in a second round.
  const bool late_mid = sel && !k_on;
  if (sel && tid < NSHARD) send_mid(S, r, tid, xm, lkey, flags, 0.0f, bar_mid);

  // ---- 3. shard sum-exp, fixed tree (while the peers' messages travel)
  float l = 0.0f;
  const float cexp = __fdiv_rn(LOG2E, tau);
  if (wmass) {
    uint32_t* dst = P.samp_bits + (row * NSHARD + r) * SAMP_BITWORDS;
    if (xm_finite) {
      l = block_sum_fixed(pass_sumexp_words(sh, tid, nchunks, xm, cexp, dst), S);
    } else {
      for (int i = tid; i < SAMP_XM_WORD; i += NTHR) dst[i] = 0u;    // -inf shard: no mass
    }
    if (tid == 0) dst[SAMP_XM_WORD] = __float_as_uint(xm);
  } else if (!greedy && xm_finite) {
    l = block_sum_fixed(pass_sumexp(sh, tid, nchunks, xm, cexp), S);
  }
  if (late_mid && tid < NSHARD) {
    // the shard's sum-exp to every CTA: the window needs the row's total mass
    const uint4 msg = make_uint4(__float_as_uint(l), 0u, 0u, flags);
    if (tid == static_cast<int>(r))
      *reinterpret_cast<uint4*>(&S.mid2[r]) = msg;
    else
      st_async_v4(map_rank(smem_addr(&S.mid2[r]), tid), msg, map_rank(bar_mid2, tid));
  }

  // ---- 4. candidate pass: every element of the window is counted straight
  //           into the leader's histogram (one shared-memory add per element)
  int hi = 0, lo = 1;
  if (sel) {
    if (tid == 0) {
      // the window of candidate keys, the same in every CTA of the cluster
      // (top-p-only rows: both exchanges in).  The waits acquire at cluster
      // scope: after them this CTA's adds into the leader's histogram are
      // ordered after the leader's zeroing of it.
      if (late_mid && !mbar_wait_bounded_cl(bar_mid)) {
        flags |= FLAG_TIMEOUT;
        mbar_wait_until_cl(bar_mid, t_start + DRAIN_MID);   // resident for late messages
      }
      const uint32_t bar_w = late_mid ? bar_mid2 : bar_mid;
      if (!mbar_wait_bounded_cl(bar_w)) {
        flags |= FLAG_TIMEOUT;
        mbar_wait_until_cl(bar_w, t_start + (late_mid ? DRAIN_MID2 : DRAIN_MID));   // resident for late messages
      }
      int L = 0x7fffffff;
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < NSHARD; ++q) {
        M = fmaxf(M, S.mid[q].xm);
        L = min(L, S.mid[q].lkey);
      }
      int whi, wlo;
      if (!k_on) {
        // total mass from the second exchange
        float Z = 0.0f;
#pragma unroll
        for (int q = 0; q < NSHARD; ++q) {
          const float xq = S.mid[q].xm;
          if (xq > -INFINITY) Z = fmaf(S.mid2[q].l, ex2((xq - M) * cexp), Z);
        }
        candidate_window(M, L, Z, tau, p, false, whi, wlo);
      } else {
        candidate_window(M, L, 0.0f, tau, p, true, whi, wlo);
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
      // (an absent last chunk holds -inf in cm: excluded explicitly, for a
      // window whose bottom is -inf itself)
      uint32_t hitmask = 0;
#pragma unroll
      for (int i = 0; i < MAXCH; ++i)
        if ((i < MAXCH - 1 || tid + i * NTHR < nchunks) && __hge2_mask(cm[i], vlo2) != 0u)
          hitmask |= 1u << i;
      if (SAMPLE && P.samp_bits) {
        // the draw reads only these chunks when the support lies in the window
        uint32_t* wb = P.samp_bits + (row * NSHARD + r) * SAMP_BITWORDS;
#pragma unroll
        for (int i = 0; i < MAXCH; ++i) {
          const uint32_t word = __ballot_sync(0xffffffffu, (hitmask >> i) & 1u);
          if ((tid & 31) == 0) wb[i * NWARP + (tid >> 5)] = word;
        }
      }
      // warps with many candidate chunks count locally and push per key;
      // the others send one add per element
      const int warp_hits = __reduce_add_sync(0xffffffffu, __popc(hitmask));
      const bool busy = (r != 0) && warp_hits > BUSY_HITS;
      // with a positive window every candidate is positive: its key is b | 0x8000
      const bool pos_window = vlo_f > 0.0f;
      if ((r == 0 || busy) && warp_hits > DENSE_HITS) {
        // a dense window (most elements candidates): every element of a hit
        // chunk at fixed positions, each add a predicated instruction (the
        // address of a non-candidate is never used), instead of a
        // per-candidate search whose lanes diverge
        const uint32_t mbase = smem_addr(S.merged);
        if (pos_window) {
          // key 0x8000 + b: the add lands at A - 4 b
          const uint32_t A = mbase + 4u * static_cast<uint32_t>(hi - 0x8000);
          const unsigned short vlo16 = static_cast<unsigned short>(__float_as_uint(vlo_f) >> 16);
          if (warp_hits <= FULL_HITS) {
            while (hitmask) {
              const int i = __ffs(hitmask) - 1;
              hitmask &= hitmask - 1;
              const uint4 v = sh[tid + i * NTHR];
              count_pair_pos(v.x, vlo16, A);
              count_pair_pos(v.y, vlo16, A);
              count_pair_pos(v.z, vlo16, A);
              count_pair_pos(v.w, vlo16, A);
            }
          } else {
            // nearly every chunk hit: a fixed walk without branches.  A chunk
            // that is not hit has no element at or above the window bottom, so
            // its adds are all predicated off; only the last chunk, which a
            // thread may not own, keeps its test
#pragma unroll
            for (int i = 0; i < MAXCH - 1; ++i) {
              const uint4 v = sh[tid + i * NTHR];
              count_pair_pos(v.x, vlo16, A);
              count_pair_pos(v.y, vlo16, A);
              count_pair_pos(v.z, vlo16, A);
              count_pair_pos(v.w, vlo16, A);
            }
            if ((hitmask >> (MAXCH - 1)) & 1u) {
              const uint4 v = sh[tid + (MAXCH - 1) * NTHR];
              count_pair_pos(v.x, vlo16, A);
              count_pair_pos(v.y, vlo16, A);
              count_pair_pos(v.z, vlo16, A);
              count_pair_pos(v.w, vlo16, A);
            }
            hitmask = 0;
          }
        } else {
          while (hitmask) {
            const int i = __ffs(hitmask) - 1;
            hitmask &= hitmask - 1;
            const uint4 v = sh[tid + i * NTHR];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t m2 = __hge2_mask(as_bf2(w[j]), vlo2);
              const int i0 = hi - okey(w[j] & 0xFFFFu), i1 = hi - okey(w[j] >> 16);
              red_shared_add_if(mbase + 4u * static_cast<uint32_t>(i0), 1u, m2 & 1u);
              red_shared_add_if(mbase + 4u * static_cast<uint32_t>(i1), 1u, m2 & 0x10000u);
            }
          }
        }
      }
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
          if (r == 0 || busy) {
            red_shared_add(&S.merged[idx], 1u);
          } else {
            red_async_add(dst + 4u * static_cast<uint32_t>(idx), 1u, rbar);
            ++sent;
          }
        }
      }
      if (__syncthreads_or(busy)) {
        // push the busy warps' counts, two keys per 8-byte add (neither
        // 32-bit count can carry: a row has fewer than 2^32 tokens)
        const int npairs = (hi - lo + 2) >> 1;
        for (int iw = tid; iw < npairs; iw += NTHR) {
          const uint2 cw = *reinterpret_cast<const uint2*>(&S.merged[2 * iw]);
          if (cw.x | cw.y) {
            red_async_add_u64(dst + 8u * iw, (static_cast<unsigned long long>(cw.y) << 32) | cw.x, rbar);
            sent += 2;
          }
        }
      }
    } else {
      if (tid == 0 && xm == -INFINITY && lo <= KEY_NEG_INF && lo <= hi) {
        // every element of this shard is -inf (a NaN makes the row NaN) and
        // the window reaches -inf: the whole shard counts at that key
        const int idx = hi - KEY_NEG_INF;
        const uint32_t cnt = static_cast<uint32_t>(nchunks) * 8u;
        if (r == 0) {
          red_shared_add(&S.merged[idx], cnt);
        } else {
          red_async_add(map_rank(smem_addr(S.merged), 0) + 4u * static_cast<uint32_t>(idx), cnt,
                        map_rank(bar_hist, 0));
          ++sent;
        }
      }
      if (SAMPLE && P.samp_bits) {
        // no element of this shard reaches the window with any mass
        uint32_t* wb = P.samp_bits + (row * NSHARD + r) * SAMP_BITWORDS;
        for (int i = tid; i < SAMP_BITWORDS; i += NTHR) wb[i] = 0u;
      }
    }
    // the leader learns how many add bytes (in 4-byte units) the peers sent:
    // each peer warp adds its number into the leader's counter, completing
    // on the summaries' barrier (each warp on its own: no block barrier
    // before the peer ends)
    sent = __reduce_add_sync(0xffffffffu, sent);
    if (r != 0 && (tid & 31) == 0)
      red_async_add(map_rank(smem_addr(&S.npush), 0), sent, map_rank(bar_sum, 0));
  }

  // ---- 5. summary to the leader
  if (tid == 0) {
    const uint4 msg = make_uint4(__float_as_uint(xm), __float_as_uint(l), sel ? 0u : first, flags);
    if (r == 0) *reinterpret_cast<uint4*>(&S.slot[0]) = msg;
    else st_async_v4(map_rank(smem_addr(&S.slot[r]), 0), msg, map_rank(bar_sum, 0));
  }
  if (r != 0) {                // messages carry everything the leader needs
    if (BWD) {
      // the leader's resolution of the row (one thread waits; after a timeout
      // it stays resident for a late record), then this shard's gradient
      if (tid == 0) {
        const bool got = mbar_wait_bounded(bar_lead);
        if (!got) mbar_wait_until(bar_lead, t_start + DRAIN_LEAD);
        S.win[3] = got ? 1 : 0;
      }
      __syncthreads();
      const bool ok = S.win[3] != 0;
      const GradCoeffs m = ok ? grad_coeffs(*reinterpret_cast<const rlk_row_stats*>(&S.lead), tau,
                                            P.g_full ? P.g_full[row] : 0.0f,
                                            (RESTR && P.g_restr) ? P.g_restr[row] : 0.0f)
                              : nan_coeffs();
      write_grad_shard(sh, false, nchunks, static_cast<int>(r) * SW, t, m, gshard, P.grad_f32 != 0);
    }
    return;
  }

  // ================= leader: merge in fixed shard order =================
  // One thread waits for the peers' messages; warp 0 merges and selects; the
  // whole block joins only for the general (wide-support) selection.
  if (tid == 0) {
    bool timed_out = !mbar_wait_bounded(bar_sum);
    // after a timeout, stay resident until every peer is past its own
    // bounded waits (its summary and adds are then in); the adds can only be
    // awaited once every peer warp has announced their number
    const bool sums_in = !timed_out || mbar_wait_until(bar_sum, t_start + DRAIN_SUM);
    if (sel && sums_in) {
      const uint32_t pushed = S.npush;     // complete with the summaries
      mbar_arrive_expect_tx(bar_hist, 4u * pushed);
      if (!mbar_wait_bounded(bar_hist)) {
        timed_out = true;
        mbar_wait_until(bar_hist, t_start + DRAIN_SUM);
      }
    }
    S.win[3] = timed_out ? 1 : 0;
  }
  __syncthreads();
  const bool timed_out = S.win[3] != 0;
  if (!BWD && tid >= 32 && !sel) return;   // only warp 0 finishes rows without a support search
  bool bad = timed_out;
  float M = -INFINITY;
  float full = __int_as_float(0x7fc00000), restr = full;
  int support = -1;
  float Z = 0.0f, d = 0.0f;
  uint32_t amax = 0x7fffffffu;    // greedy rows: first column holding the maximum
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
  bool shard_reused = false;      // the leader's shard copy became scratch
  bool in_s = true;               // target in the support (every token is when !sel)
  float zs = Z;
  if (sel) {
    __syncthreads();
    if (!S.sel_done) {
      // wide support: the whole block scans further windows
      uint32_t* cntB = reinterpret_cast<uint32_t*>(S.shard);
      sr = select_support(S, S.merged, cntB, hi, lo, rowp, S.bc_f[0], c, S.bc_f[1], p, k, k_on, p_on);
      shard_reused = true;
    }
    if (!BWD && tid != 0) return;
    if (tid == 0 && !bad) {
      in_s = okey_of(xt) >= sr.min_key;
      zs = __ull2float_rn(sr.zs) * (1.0f / FX_SCALE);
      restr = in_s ? d - logf(zs) : -INFINITY;
      support = static_cast<int>(sr.support);
    }
  }

  if (tid == 0 && !SAMPLE) {
    if (o_full) o_full[row] = full;
    if (RESTR && o_restr) o_restr[row] = restr;
    if (RESTR && o_support) o_support[row] = support;
    if (P.out_kl) P.out_kl[row] = P.kl_policy_full[row] - full;
    if (timed_out && o_err) atomicAdd(o_err, 1);
  }

  if (BWD || P.out_stats) {
    // the row's resolution as a per-row record: saved for a later backward,
    // and sent to the 7 peers for this pass's gradient
    if (tid == 0) {
      rlk_row_stats st;
      st.max_logit = M;
      st.inv_z = bad ? __int_as_float(0x7fc00000) : (greedy ? 0.0f : __fdiv_rn(1.0f, Z));
      st.inv_z_support = (bad || greedy || !in_s) ? 0.0f : __fdiv_rn(1.0f, zs);
      st.min_key = sel ? sr.min_key : 0;
      if (P.out_stats) P.out_stats[row] = st;
      if (BWD) {
        const uint4 v = *reinterpret_cast<const uint4*>(&st);
        S.lead = v;
#pragma unroll
        for (int q = 1; q < NSHARD; ++q)
          st_async_v4(map_rank(smem_addr(&S.lead), q), v, map_rank(bar_lead, q));
      }
    }
  }
  if (BWD) {
    __syncthreads();
    const GradCoeffs m = grad_coeffs(*reinterpret_cast<const rlk_row_stats*>(&S.lead), tau,
                                     P.g_full ? P.g_full[row] : 0.0f,
                                     (RESTR && P.g_restr) ? P.g_restr[row] : 0.0f);
    write_grad_shard(shard_reused ? reinterpret_cast<const uint4*>(rowp) : sh, shard_reused, nchunks,
                     0, t, m, gshard, P.grad_f32 != 0);
  }

  if (SAMPLE && tid == 0) {
    // the row's resolution for the draw kernel; rows without a draw finish here
    SampMsg m{};
    m.M = M;
    m.Z = Z;
    m.min_key = sel ? sr.min_key : 0;
    m.flags = (!bad && !greedy ? SAMP_DRAW : 0u) | (sel ? SAMP_SEL : 0u) |
              (sel && !shard_reused && P.samp_bits ? SAMP_BITS : 0u) | (wmass ? SAMP_WORDS : 0u);
    P.out_samp[row] = m;
    if (P.out_support) P.out_support[row] = support;
    if (bad) {
      P.out_token[row] = -1;
      if (P.out_full) P.out_full[row] = __int_as_float(0x7fc00000);
      if (P.out_restr) P.out_restr[row] = __int_as_float(0x7fc00000);
    } else if (greedy) {
      P.out_token[row] = static_cast<int32_t>(amax);
      if (P.out_full) P.out_full[row] = 0.0f;
      if (P.out_restr) P.out_restr[row] = 0.0f;
    }
    if (timed_out && P.err) atomicAdd(P.err, 1);
  }
}

// ------------------------------------------------------------ the draw

// One block per row, after the pair pass resolved every row (greedy, NaN
// and rejected rows were finished there and exit at once).  The support mass
// of a 16-byte chunk is the sum of its support elements' fixed-point masses
// (the selection's per-key values, 2^-44 units); the drawn mass
// floor(u Z_S / 2^32) is located in column order.  The chunks read are the
// ones the pair pass marked as reaching the candidate window when the
// support lies inside it (SAMP_BITS: about 150 of a row's 19,000 on the
// 8192-row workload), otherwise every real chunk of the row.  Each thread
// takes a run of consecutive bitmap words (32 chunks each), so a block scan
// of the threads' masses is a scan in column order; the thread holding the
// draw finds the word from the per-word masses kept in shared memory, and
// warp 0 finds the chunk (one chunk per lane, a warp scan) and the column.
struct SampRowSmem {
  float wf[NSHARD * SAMP_BITWORDS];                  // unfiltered rows: float mass per word
  float xm[NSHARD], sq[NSHARD];                      // unfiltered rows: shard maxima, their factors
  uint32_t bw[NSHARD * SAMP_BITWORDS];               // the chunks to read
  unsigned long long wm[NSHARD * SAMP_BITWORDS];     // support mass per bitmap word
  uint32_t scan_c[NWARP];
  unsigned long long scan_m[NWARP];
  int32_t own_w;                                     // the word holding the draw
  unsigned long long own_res;                        // the draw's offset inside that word
};

// An unfiltered row: the word holding the draw from the float word masses
// (written by the pair pass, or computed here from every chunk), then the
// chunk and the column inside it.  With P(w) the running sum of the scaled
// word masses in column order (each lane of warp 0 sums a run of
// consecutive words from the lanes' exclusive scan), Z the scan's total and
// t = U Z for U = (u >> 8) / 2^24, the word is the first whose running sum
// exceeds t, the chunk the first whose running sum inside the word exceeds
// what is left of t, and likewise the column; where rounding leaves nothing
// to exceed, the last one with a nonzero mass is taken.
__device__ void draw_unfiltered(const KParams& P, SampRowSmem& S, int64_t row, const SampMsg& m) {
  constexpr int NW = NSHARD * SAMP_BITWORDS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const float c = __fdiv_rn(LOG2E, tau);
  const uint4* rowp = reinterpret_cast<const uint4*>(P.logits + row * P.stride);
  auto nch = [](int q) { return q == NSHARD - 1 ? LAST_CHUNKS : SHARD_CHUNKS; };
  if (m.flags & SAMP_WORDS) {
    const uint32_t* src = P.samp_bits + row * NW;
    for (int i = tid; i < NW; i += NTHR) {
      const bool xmw = (i % SAMP_BITWORDS) == SAMP_XM_WORD;
      if (xmw) S.xm[i / SAMP_BITWORDS] = __uint_as_float(src[i]);
      S.wf[i] = xmw ? 0.0f : __uint_as_float(src[i]);
    }
  } else {
    // the shard maxima (as the pair pass's bf16 maximum), then the word masses
    for (int q = warp; q < NSHARD; q += NWARP) {
      float mx = -INFINITY;
      for (int g = lane; g < nch(q); g += 32) {
        const uint4 v = __ldg(rowp + q * SHARD_CHUNKS + g);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fmaxf(bf16_lo(w4[j]), bf16_hi(w4[j])));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) S.xm[q] = mx;
    }
    __syncthreads();
    for (int wd = warp; wd < NW; wd += NWARP) {
      const int q = wd / SAMP_BITWORDS, g = (wd % SAMP_BITWORDS) * 32 + lane;
      const float cm = g < nch(q) ? chunk_mass_f(__ldg(rowp + q * SHARD_CHUNKS + g), S.xm[q], c) : 0.0f;
      const float ws = word_sum_lane0(cm);
      if (lane == 0) S.wf[wd] = ws;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  // each shard's factor to the row maximum, and the scaled word masses
  const float sq = lane < NSHARD && S.xm[lane] > -INFINITY
                       ? ex2(__fmul_rn(__fsub_rn(S.xm[lane], m.M), c)) : 0.0f;
  if (lane < NSHARD) S.sq[lane] = sq;
  __syncwarp();
  constexpr int PER = (NW + 31) / 32;
  const int w0 = min(NW, lane * PER), w1 = min(NW, w0 + PER);
  for (int w = w0; w < w1; ++w) S.wf[w] = __fmul_rn(S.wf[w], S.sq[w / SAMP_BITWORDS]);
  float run = 0.0f;
  for (int w = w0; w < w1; ++w) run = __fadd_rn(run, S.wf[w]);
  float incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = __fadd_rn(incl, t);
  }
  const float Zd = __shfl_sync(0xffffffffu, incl, 31);
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.0f;
  const uint32_t u = P.uniform ? P.uniform[row] : philox_word0(P.seed, P.counter[row]);
  const float tdraw = __fmul_rn(static_cast<float>(u >> 8) * 5.9604644775390625e-8f, Zd);
  // the first word whose running sum exceeds t; else the last nonzero word
  int wfound = -1, wlast = -1;
  float before = 0.0f, before_last = 0.0f, acc = excl;
  for (int w = w0; w < w1; ++w) {
    const float ww = S.wf[w];
    const float nxt = __fadd_rn(acc, ww);
    if (wfound < 0 && nxt > tdraw) { wfound = w; before = acc; }
    if (ww > 0.0f) { wlast = w; before_last = acc; }
    acc = nxt;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, wfound >= 0);
  int ws;
  float wbefore;
  if (hit) {
    const int src = __ffs(hit) - 1;
    ws = __shfl_sync(0xffffffffu, wfound, src);
    wbefore = __shfl_sync(0xffffffffu, before, src);
  } else {
    const unsigned has = __ballot_sync(0xffffffffu, wlast >= 0);
    const int src = has ? 31 - __clz(has) : 0;
    ws = __shfl_sync(0xffffffffu, wlast, src);
    wbefore = __shfl_sync(0xffffffffu, before_last, src);
  }
  if (ws < 0) return;                                  // no mass at all (not a drawing row)
  // the chunk: lane j takes chunk j of the word
  const int q = ws / SAMP_BITWORDS, g = (ws % SAMP_BITWORDS) * 32 + lane;
  const float xq = S.xm[q], sqq = S.sq[q];
  const bool real = g < nch(q);
  const uint4 v = real ? __ldg(rowp + q * SHARD_CHUNKS + g) : make_uint4(0u, 0u, 0u, 0u);
  const float cm = real ? __fmul_rn(chunk_mass_f(v, xq, c), sqq) : 0.0f;
  const float left = __fsub_rn(tdraw, wbefore);
  float cin = cm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, cin, o);
    if (lane >= o) cin = __fadd_rn(cin, t);
  }
  const unsigned chit = __ballot_sync(0xffffffffu, cin > left);
  const unsigned cnz = __ballot_sync(0xffffffffu, cm > 0.0f);
  const int cl = chit ? __ffs(chit) - 1 : 31 - __clz(cnz);
  if (lane != cl) return;
  float rest = __fsub_rn(left, __fsub_rn(cin, cm));
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  int jstar = -1, jlast = -1;
  uint32_t xb = 0, xlast = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t e16 = (w4[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
    const float e = __fmul_rn(ex2(__fmul_rn(__fsub_rn(__uint_as_float(e16 << 16), xq), c)), sqq);
    if (e > 0.0f) { jlast = j; xlast = e16; }
    if (jstar < 0) {
      if (rest < e) { jstar = j; xb = e16; } else { rest = __fsub_rn(rest, e); }
    }
  }
  if (jstar < 0) { jstar = jlast; xb = xlast; }
  const float xa = __uint_as_float(xb << 16);
  const float d = __fdiv_rn(xa - m.M, tau);
  const float full = d - logf(m.Z);
  P.out_token[row] = q * SW + g * 8 + jstar;
  if (P.out_full) P.out_full[row] = full;
  if (P.out_restr) P.out_restr[row] = full;
}

__global__ void __launch_bounds__(NTHR) sample_row_kernel(const KParams P) {
  __shared__ SampRowSmem S;
  constexpr int NW = NSHARD * SAMP_BITWORDS;
  const int64_t row = blockIdx.x;
  const SampMsg m = P.in_samp[row];
  if (!(m.flags & SAMP_DRAW)) return;                 // uniform over the block
  if (!(m.flags & SAMP_SEL)) {
    draw_unfiltered(P, S, row, m);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31;
  if (m.flags & SAMP_BITS) {
    const uint32_t* src_bits = P.samp_bits + row * NW;
    for (int i = tid; i < NW; i += NTHR) S.bw[i] = src_bits[i];
  } else {
    for (int i = tid; i < NW; i += NTHR) {         // every real chunk
      const int q = i / SAMP_BITWORDS, g0 = (i % SAMP_BITWORDS) * 32;
      const int n = (q == NSHARD - 1 ? LAST_CHUNKS : SHARD_CHUNKS) - g0;
      S.bw[i] = n >= 32 ? 0xffffffffu : (n > 0 ? (1u << n) - 1u : 0u);
    }
  }
  if (tid == 0) S.own_w = -1;
  __syncthreads();
  const float tau = P.tau_arr ? P.tau_arr[row] : P.tau_s;
  const float c = __fdiv_rn(LOG2E, tau);
  // keys at or below -inf's are the whole vocabulary (min_key 0 when
  // unfiltered; key_value of keys below -inf's would be a NaN pattern)
  const float vmin_f = m.min_key <= KEY_NEG_INF ? -INFINITY : key_value(m.min_key);
  const __nv_bfloat162 vmin2 = __floats2bfloat162_rn(vmin_f, vmin_f);
  const uint4* rowp = reinterpret_cast<const uint4*>(P.logits + row * P.stride);
  constexpr int PER = (NW + NTHR - 1) / NTHR;
  const int w0 = min(NW, tid * PER), w1 = min(NW, w0 + PER);
  // ---- support mass per word, four chunk loads in flight at a time
  unsigned long long mine = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = S.bw[w];
    const uint4* base = rowp + (w / SAMP_BITWORDS) * SHARD_CHUNKS + (w % SAMP_BITWORDS) * 32;
    unsigned long long ws = 0;
    while (bits) {
      int b[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        b[t] = bits ? __ffs(bits) - 1 : -1;
        bits &= bits - 1;
      }
      uint4 v[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (b[t] >= 0) v[t] = __ldg(base + b[t]);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (b[t] >= 0) ws += chunk_support_mass(v[t], vmin2, m.M, c);
    }
    S.wm[w] = ws;
    mine += ws;
  }
  uint32_t ec, tc;
  unsigned long long excl, zs;
  block_excl_scan(0u, mine, ec, excl, tc, zs, S);    // ends with a block barrier
  const uint32_t u = P.uniform ? P.uniform[row] : philox_word0(P.seed, P.counter[row]);
  const unsigned long long draw = scale_draw(u, zs);
  if (mine != 0 && draw >= excl && draw - excl < mine) {
    // this thread's run holds the draw: the word, from the kept word masses
    unsigned long long left = draw - excl;
    for (int w = w0; w < w1; ++w) {
      if (left < S.wm[w]) {
        S.own_w = w;
        S.own_res = left;
        break;
      }
      left -= S.wm[w];
    }
  }
  __syncthreads();
  const int w = S.own_w;
  if (tid >= 32 || w < 0) return;
  // ---- warp 0: the chunk (lane j takes chunk j of the word), then the column
  const uint32_t bits = S.bw[w];
  const int q = w / SAMP_BITWORDS, g0 = (w % SAMP_BITWORDS) * 32;
  const bool marked = (bits >> lane) & 1u;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  unsigned long long mc = 0;
  if (marked) {
    v = __ldg(rowp + q * SHARD_CHUNKS + g0 + lane);
    mc = chunk_support_mass(v, vmin2, m.M, c);
  }
  const unsigned long long ex = warp_incl_scan_u64(mc) - mc;
  const unsigned long long res = S.own_res;
  if (mc == 0 || res < ex || res - ex >= mc) return;
  unsigned long long left = res - ex;
  const uint32_t sb = chunk_support_bits(v, vmin2);
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  int jstar = -1;
  uint32_t xb = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t e = (w4[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
    if (jstar < 0 && ((sb >> ((j >> 1) + 16 * (j & 1))) & 1u)) {
      const unsigned long long qm = qfx(__uint_as_float(e << 16), m.M, c);
      if (left < qm) {
        jstar = j;
        xb = e;
      } else {
        left -= qm;
      }
    }
  }
  const float xa = __uint_as_float(xb << 16);
  const float d = __fdiv_rn(xa - m.M, tau);
  const float full = d - logf(m.Z);
  const float restr = (m.flags & SAMP_SEL) ? d - logf(__ull2float_rn(zs) * (1.0f / FX_SCALE)) : full;
  P.out_token[row] = q * SW + (g0 + lane) * 8 + jstar;
  if (P.out_full) P.out_full[row] = full;
  if (P.out_restr) P.out_restr[row] = restr;
}

// The KL term of each row: the policy's full logprob minus the reference's.
__global__ void kl_kernel(const float* full, const float* full_ref, float* kl, int64_t T) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < T) kl[i] = full[i] - full_ref[i];
}

// ------------------------------------------------------------ host side

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

template <bool RESTR, int MODE = MODE_FWD>
rlk_status launch(const KParams& P, int64_t T, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(logp_kernel<RESTR, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = cudaFuncSetAttribute(logp_kernel<RESTR, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(Smem)));
    if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  const dim3 grid(static_cast<unsigned>(T * NSHARD));
  logp_kernel<RESTR, MODE><<<grid, NTHR, sizeof(Smem), stream>>>(P);
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

rlk_status rlk_logp_pair_save(const rlk_logp_args* args, float* out_full, float* out_restr,
                              int32_t* out_support, rlk_row_stats* out_stats, void* stream) {
  rlk_status s = check_args(args, true);
  if (s != RLK_OK || args->T == 0) return s;
  if (!out_full && !out_restr) return fail(RLK_EINVAL, "out_full and out_restr are both NULL");
  if ((s = check_out(out_full, "out_full", false)) != RLK_OK) return s;
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  if (!out_stats) return fail(RLK_EINVAL, "out_stats is NULL");
  if (!aligned(out_stats, 16)) return fail(RLK_EALIGN, "out_stats is not 16-byte aligned");
  KParams P = make_params(args);
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  P.out_stats = out_stats;
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
  if (policy->T >= (int64_t(1) << 27))
    return fail(RLK_EINVAL, "T = %lld: at most 2^27 - 1 rows per rlk_logp_kl call", (long long)policy->T);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KParams P = make_params(policy);
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  P.ref_logits = static_cast<const uint16_t*>(ref_logits);
  P.ref_stride = ref_row_stride;
  P.out_full_ref = out_full_ref;
  if ((s = launch<true>(P, 2 * policy->T, st)) != RLK_OK) return s;
  kl_kernel<<<static_cast<unsigned>((policy->T + 255) / 256), 256, 0, st>>>(out_full, out_full_ref, out_kl,
                                                                             policy->T);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
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

rlk_status rlk_logp_backward(const rlk_logp_args* args, const float* grad_full,
                             const float* grad_restr, void* grad_logits, int64_t grad_row_stride,
                             int32_t grad_dtype, float* out_full, float* out_restr,
                             int32_t* out_support, void* stream) {
  const bool restr = grad_restr || out_restr || out_support;
  rlk_status s = check_args(args, restr);
  if (s != RLK_OK || args->T == 0) return s;
  if ((s = check_grad_args(grad_full, grad_restr, grad_logits, grad_row_stride, grad_dtype)) != RLK_OK)
    return s;
  if ((s = check_out(out_full, "out_full", false)) != RLK_OK) return s;
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  KParams P = make_params(args);
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  P.g_full = grad_full;
  P.g_restr = grad_restr;
  P.grad = static_cast<char*>(grad_logits);
  P.grad_stride = grad_row_stride;
  P.grad_f32 = grad_dtype == RLK_GRAD_F32 ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return restr ? launch<true, MODE_BWD>(P, args->T, st) : launch<false, MODE_BWD>(P, args->T, st);
}

rlk_status rlk_sample(const rlk_logp_args* args, unsigned long long seed,
                      const unsigned long long* counter, const uint32_t* uniform,
                      int32_t* out_token, float* out_restr, float* out_full,
                      int32_t* out_support, void* workspace, void* stream) {
  // the records first, then the chunk bitmaps (T * 16 keeps them 16-byte aligned)
  uint32_t* bits = (args && workspace && args->T > 0)
                       ? reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + args->T * 16)
                       : nullptr;
  return sample_impl(args, seed, counter, uniform, out_token, out_restr, out_full, out_support,
                     workspace, bits, stream);
}

}  // extern "C"

namespace rlk {

rlk_status sample_impl(const rlk_logp_args* args, unsigned long long seed,
                       const unsigned long long* counter, const uint32_t* uniform,
                       int32_t* out_token, float* out_restr, float* out_full,
                       int32_t* out_support, void* workspace, uint32_t* bits, void* stream) {
  rlk_status s = check_args(args, true, false);
  if (s != RLK_OK || args->T == 0) return s;
  if (!counter && !uniform) return fail(RLK_EINVAL, "counter and uniform are both NULL");
  if (counter && !aligned(counter, 8)) return fail(RLK_EALIGN, "counter is not 8-byte aligned");
  if ((s = check_out(uniform, "uniform", false)) != RLK_OK) return s;
  if ((s = check_out(out_token, "out_token", true)) != RLK_OK) return s;
  if ((s = check_out(out_restr, "out_restr", false)) != RLK_OK) return s;
  if ((s = check_out(out_full, "out_full", false)) != RLK_OK) return s;
  if ((s = check_out(out_support, "out_support", false)) != RLK_OK) return s;
  if (!workspace) return fail(RLK_EINVAL, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(RLK_EALIGN, "workspace is not 16-byte aligned");
  KParams P = make_params(args);
  P.target = nullptr;
  P.out_full = out_full;
  P.out_restr = out_restr;
  P.out_support = out_support;
  P.out_token = out_token;
  P.uniform = uniform;
  P.counter = counter;
  P.seed = seed;
  P.out_samp = static_cast<SampMsg*>(workspace);
  P.in_samp = static_cast<const SampMsg*>(workspace);
  P.samp_bits = bits;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = launch<true, MODE_SAMPLE>(P, args->T, st)) != RLK_OK) return s;
  sample_row_kernel<<<static_cast<unsigned>(args->T), NTHR, 0, st>>>(P);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

}  // namespace rlk

extern "C" {

const char* rlk_status_string(rlk_status status) {
  switch (status) {
    case RLK_OK: return "ok";
    case RLK_EINVAL: return "invalid argument";
    case RLK_EALIGN: return "misaligned pointer or stride";
    case RLK_ECUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* rlk_last_error(void) { return last_error_buf(); }

int rlk_abi_version(void) { return RLK_ABI_VERSION; }

}  // extern "C"
