// rlk_device.cuh -- device building blocks shared by the fused logprob kernel
// and the vocabulary-sharded kernels: constants, PTX wrappers, bf16 order
// keys, fixed-tree block reductions, the per-shard max and sum-exp passes,
// the candidate window, and the support selection on a per-key count
// histogram.
//
// Both kernel families call the same pass functions, so a shard's
// (max, sum-exp) summary has the same bits whichever kernel computes it.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "rlk_logp.h"

#ifndef RLK_NTHR
#define RLK_NTHR 128
#endif
#ifndef RLK_SEL_KPL
#define RLK_SEL_KPL 4            // keys per lane per step of the warp selection
#endif
#ifndef RLK_WAIT_HINT_NS
#define RLK_WAIT_HINT_NS 20000   // suspend-time hint of a barrier test (ns)
#endif

namespace rlk {

constexpr int VPAD = RLK_VOCAB_PADDED;
constexpr int VREAL = RLK_VOCAB_REAL;
constexpr int NSHARD = RLK_NUM_SHARDS;
constexpr int SW = RLK_SHARD_WIDTH;
constexpr int SHARD_CHUNKS = SW / 8;                        // 2384 16-byte chunks
constexpr int LAST_CHUNKS = (VREAL - (NSHARD - 1) * SW) / 8;  // 2304 real chunks
constexpr int NTHR = RLK_NTHR;       // threads per CTA
constexpr int NWARP = NTHR / 32;
constexpr int ROW_WARPS = NSHARD * NWARP;
constexpr int CTAS_PER_SM = 5;
constexpr int MAXCH = (SHARD_CHUNKS + NTHR - 1) / NTHR;     // chunks per thread (19)
// sampler: one bit per chunk of a shard, word i * NWARP + w holding chunks
// (i * NWARP + w) * 32 .. + 31 (76 words, 2432 >= 2384 bits)
constexpr int SAMP_BITWORDS = MAXCH * NWARP;
constexpr int WIN = 1024;            // candidate window, in bf16 order keys (8 binades)
constexpr int TMA_PIECES = 4;
constexpr int BUSY_HITS = 16;        // candidate chunks per warp above which it counts locally
constexpr int DENSE_HITS = 128;      // ... and above which it counts every element of a hit chunk
constexpr int FULL_HITS = 352;       // ... and above which it walks all its chunks in a fixed order
constexpr float LOG2E = 1.4426950408889634f;   // log2(e)
constexpr float FX_SCALE = 17592186044416.0f;  // 2^44: fixed-point scale of masses
constexpr unsigned long long TIMEOUT_NS = 200000000ull;   // 0.2 s bound on every wait
constexpr int KEY_NEG_INF = 0x007F;  // order key of -inf; smaller keys are NaN patterns

static_assert(SW % 8 == 0 && (VREAL - (NSHARD - 1) * SW) % 8 == 0, "chunking");
static_assert((MAXCH - 1) * NTHR <= LAST_CHUNKS, "every thread owns MAXCH-1 chunks in every shard");
static_assert(SHARD_CHUNKS % TMA_PIECES == 0 && LAST_CHUNKS % TMA_PIECES == 0, "pieces");

enum : uint32_t { FLAG_TIMEOUT = 1u, FLAG_NAN = 2u, FLAG_LEVELS = 4u };

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
// 64-bit atomic add into a peer CTA's shared memory, completing 8 bytes on its mbarrier
__device__ __forceinline__ void red_async_add_u64(uint32_t addr, unsigned long long v, uint32_t bar) {
  asm volatile("red.async.relaxed.cluster.shared::cluster.mbarrier::complete_tx::bytes.add.u64 [%0], %1, [%2];"
               :: "r"(addr), "l"(v), "r"(bar) : "memory");
}
// shared-memory add without a return value (nothing waits for it)
__device__ __forceinline__ void red_shared_add(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" :: "r"(smem_addr(p)), "r"(v) : "memory");
}
// the same add, issued only where pred != 0 (a predicated instruction, no branch);
// addr need not be valid where pred == 0
__device__ __forceinline__ void red_shared_add_if(uint32_t addr, uint32_t v, uint32_t pred) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q red.shared.add.u32 [%0], %1;\n\t}"
               :: "r"(addr), "r"(v), "r"(pred) : "memory");
}
// Dense count over a window of positive values: each bf16 half b of w at or
// above vlo (a positive bf16 value) adds one at byte address A - 4 b, where A
// is the address key 0x8000 (value +0) would have: a positive value's order
// key is 0x8000 + b.  Both comparisons are on the halves unpacked by name
// (lower, upper), each add a predicated instruction.
__device__ __forceinline__ void count_pair_pos(uint32_t w, unsigned short vlo, uint32_t A) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b16 h0, h1;\n\t.reg .b32 t0, t1;\n\t"
      "mov.b32 {h0, h1}, %0;\n\t"
      "setp.ge.bf16 p0, h0, %1;\n\t"
      "setp.ge.bf16 p1, h1, %1;\n\t"
      "and.b32 t0, %0, 65535;\n\t"
      "shl.b32 t0, t0, 2;\n\t"
      "sub.u32 t0, %2, t0;\n\t"
      "shr.b32 t1, %0, 16;\n\t"
      "shl.b32 t1, t1, 2;\n\t"
      "sub.u32 t1, %2, t1;\n\t"
      "@p0 red.shared.add.u32 [t0], 1;\n\t"
      "@p1 red.shared.add.u32 [t1], 1;\n\t}"
      :: "r"(w), "h"(vlo), "r"(A) : "memory");
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
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(static_cast<uint32_t>(RLK_WAIT_HINT_NS)) : "memory");
  return ok != 0;
}
// The same test with acquire semantics at cluster scope: a message that
// completes the barrier releases at cluster scope what its sender had
// observed, and this makes it visible to the waiting thread.
__device__ __forceinline__ bool mbar_try_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(static_cast<uint32_t>(RLK_WAIT_HINT_NS)) : "memory");
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
// Wait on phase 0 of a barrier until a wall-clock deadline (globaltimer ns).
// Used after a bounded wait gave up on a peer's messages: the CTA stays
// resident, so that a late message never lands in the shared memory of a
// CTA that has exited.  Deadlines are staged from each CTA's start (the
// CTAs of a cluster start together), every stage's senders finishing their
// own bounded waits before the stage's receivers stop draining:
//   DRAIN_MID:  exchange messages, sent once the sender's shard copy landed
//               (at most 2 TIMEOUT_NS after its start);
//   DRAIN_MID2: top-p-only rows' second exchange (the shard's sum-exp),
//               sent after the sender's sum-exp pass (its shard copy landed
//               at most 2 TIMEOUT_NS after its start);
//   DRAIN_SUM:  summaries and histogram adds, sent after the sender's
//               exchange waits (at most DRAIN_MID2);
//   DRAIN_LEAD: the backward's row record, sent after the leader's summary
//               wait (at most DRAIN_SUM) and its selection.
constexpr unsigned long long DRAIN_MID = 4 * TIMEOUT_NS;
constexpr unsigned long long DRAIN_MID2 = 5 * TIMEOUT_NS;
constexpr unsigned long long DRAIN_SUM = 6 * TIMEOUT_NS;
constexpr unsigned long long DRAIN_LEAD = 8 * TIMEOUT_NS;
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, unsigned long long deadline) {
  while (!mbar_try(bar, 0)) {
    if (global_timer() > deadline) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_bounded_cl(uint32_t bar) {
  if (mbar_try_cl(bar, 0)) return true;
  const unsigned long long t0 = global_timer();
  while (!mbar_try_cl(bar, 0)) {
    if (global_timer() - t0 > TIMEOUT_NS) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_until_cl(uint32_t bar, unsigned long long deadline) {
  while (!mbar_try_cl(bar, 0)) {
    if (global_timer() > deadline) return false;
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

// Round a float q in [0, 2^44] to the nearest integer, ties to even, without
// the float -> u64 converter (it runs on the FP64 pipe, which is narrow on
// this GPU).  Below 2^23 one IEEE add of 2^23 rounds q to an integer, read
// from the sum's bits (bits(2^23) = 0x4B000000; a sum that rounds up to 2^24
// reads as 2^23, also right); from 2^23 up q is an integer, mantissa <<
// (exponent - 150).  Equal to round-half-even for every float in [0, 2^44]
// (checked exhaustively).  Branch-free.
__device__ __forceinline__ unsigned long long fx_round(float q) {
  const uint32_t b = __float_as_uint(q);
  const uint32_t small = __float_as_uint(__fadd_rn(q, 8388608.0f)) - 0x4B000000u;
  const uint32_t sh = min(max(b >> 23, 150u) - 150u, 21u);
  const unsigned long long big = static_cast<unsigned long long>((b & 0x7FFFFFu) | 0x800000u) << sh;
  return q < 8388608.0f ? static_cast<unsigned long long>(small) : big;
}

// fixed-point mass of one element at key value v: exp(s - M) * 2^44, rounded
// to the nearest integer.  The selection's few per-key masses are latency-bound
// and keep the hardware conversion; the dense sampler path uses fx_round.
__device__ __forceinline__ unsigned long long qfx(float v, float M, float c) {
  const float q = ex2((v - M) * c);
  return __float2ull_rn(q * FX_SCALE);
}

// ------------------------------------------------------------ block helpers

// Fixed-order sum: butterfly inside each warp, then a left fold over warps.
template <class SM>
__device__ __forceinline__ float block_sum_fixed(float v, SM& S) {
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

template <class SM>
__device__ __forceinline__ int block_min_int(int v, SM& S) {
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

// ------------------------------------------------------------ per-shard passes

// Max pass over one shard staged in shared memory.  Thread t owns 16-byte
// chunks t, t+NTHR, ... ; cm[i] receives the packed bf16x2 maximum of chunk i
// (-inf for a chunk the thread does not own).  Returns the order key of the
// thread's maximum.  bf16 max ignores NaN; NaN is caught by the sum-exp.
__device__ __forceinline__ int pass_max(const uint4* sh, int tid, int nchunks,
                                        __nv_bfloat162 (&cm)[MAXCH]) {
  const __nv_bfloat162 ninf2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
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
    cm[i] = cmax;
  }
  return okey_of(fmaxf(__low2float(m2), __high2float(m2)));
}

// Two bf16 NaN tests on raw bits: a bf16 is NaN iff its magnitude bits
// exceed 0x7F80, i.e. iff adding 0x7F to them carries into bit 15 (no carry
// crosses into the other half).
__device__ __forceinline__ uint32_t nan_bits2(uint32_t w) {
  return ((w & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;
}

// Greedy rows, and rows whose shard maximum is -inf, get no sum-exp, so a NaN
// must be found by a scan: it tests the raw bits of this thread's chunks.
// For greedy rows it also returns this thread's lowest column (in shard
// coordinates) equal to the shard maximum xm, looking only inside the chunks
// whose register maximum reaches xm (0x7fffffff: none).
__device__ __forceinline__ int scan_nan_first(const uint4* sh, int tid, int nchunks,
                                              const __nv_bfloat162 (&cm)[MAXCH], float xm,
                                              bool want_first, bool& nan_seen) {
  uint32_t hit = 0;               // chunks (by register slot) whose maximum reaches xm
  if (want_first && xm > -INFINITY) {
    const __nv_bfloat162 xm2 = __floats2bfloat162_rn(xm, xm);   // xm is a bf16 value
#pragma unroll
    for (int i = 0; i < MAXCH; ++i)
      if (__hge2_mask(cm[i], xm2) != 0u) hit |= 1u << i;       // absent chunks hold -inf
  }
  uint32_t nb = 0;
#pragma unroll 2
  for (int ch = tid; ch < nchunks; ch += NTHR) {
    const uint4 v = sh[ch];
    nb |= nan_bits2(v.x) | nan_bits2(v.y) | nan_bits2(v.z) | nan_bits2(v.w);
  }
  nan_seen = nb != 0u;
  int f = 0x7fffffff;
  while (hit) {
    const int ch = tid + (__ffs(hit) - 1) * NTHR;
    hit &= hit - 1;
    const uint4 v = sh[ch];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      const float x = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
      if (x == xm) f = min(f, ch * 8 + j);
    }
  }
  return f;
}

// This thread's share of the shard sum-exp: exp(s_j - m) over its chunks in
// chunk order, even and odd columns in the two lanes of a packed f32x2
// accumulator; c = log2(e) / tau.  block_sum_fixed completes the tree.
__device__ __forceinline__ float pass_sumexp(const uint4* sh, int tid, int nchunks, float xm,
                                             float c) {
  const uint64_t nxm2 = pack2(-xm, -xm);
  const uint64_t c2 = pack2(c, c);
  uint64_t acc = pack2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < MAXCH; ++i) {
    const int ch = tid + i * NTHR;
    if (i < MAXCH - 1 || ch < nchunks) {
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
  return e0 + e1;
}

// pass_sumexp for a drawing row without top-k/top-p: the same sum (same
// operations, same order), and besides it the mass of every word of 32
// consecutive chunks relative to the shard maximum xm: a chunk's mass is the
// fixed tree ((e0+e1)+(e2+e3))+((e4+e5)+(e6+e7)) of its elements'
// exponentials, a word's a fixed shuffle-down tree over its chunks, written
// by lane 0 to dst[i * NWARP + warp] (word i * NWARP + warp covers chunks
// 32 (i * NWARP + warp) .. + 31).
__device__ __forceinline__ float pass_sumexp_words(const uint4* sh, int tid, int nchunks, float xm,
                                                   float c, uint32_t* dst) {
  const uint64_t nxm2 = pack2(-xm, -xm);
  const uint64_t c2 = pack2(c, c);
  uint64_t acc = pack2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < MAXCH; ++i) {
    const int ch = tid + i * NTHR;
    float cmass = 0.0f;
    if (i < MAXCH - 1 || ch < nchunks) {
      const uint4 v = sh[ch];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float e[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t a = mul2(add2(pack2(bf16_lo(w[j]), bf16_hi(w[j])), nxm2), c2);
        float a0, a1;
        unpack2(a, a0, a1);
        e[2 * j] = ex2(a0);
        e[2 * j + 1] = ex2(a1);
        acc = add2(acc, pack2(e[2 * j], e[2 * j + 1]));
      }
      cmass = __fadd_rn(__fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3])),
                        __fadd_rn(__fadd_rn(e[4], e[5]), __fadd_rn(e[6], e[7])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmass = __fadd_rn(cmass, __shfl_down_sync(0xffffffffu, cmass, o));
    if ((tid & 31) == 0) dst[i * NWARP + (tid >> 5)] = __float_as_uint(cmass);
  }
  float e0, e1;
  unpack2(acc, e0, e1);
  return e0 + e1;
}

// Per warp: the maximum key and, when kw > 0, the kw-th largest lane key (the
// pooled top-k witness), staged in red_u / red_i for a block fold.  Warp w
// certifies kw lane maxima at or above its witness, so the W warps of a row
// certify W*kw >= k tokens at or above the minimum witness.
template <class SM>
__device__ __forceinline__ void stage_max_bound(int tkey, int kw, SM& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lw = kw > 0 ? warp_kth_largest(tkey, kw) : 0;
  const unsigned wmax = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(tkey));
  if (lane == 0) { S.red_u[warp] = wmax; S.red_i[warp] = lw; }
}

// The candidate window [wlo, whi] of order keys of a restricted row, from the
// row maximum M (a bf16 value), the pooled top-k witness L (top-k rows) and
// the total mass Z relative to M, merged in shard order (top-p-only rows).
//  - top-k rows: at least k tokens sit at or above L, so the k-th largest
//    value is >= L;
//  - top-p-only rows: tokens with s <= s_max + ln((1-p) Z / V) cannot reach
//    the nucleus, because even all V of them would hold at most 1-p of the
//    total mass, so the mass strictly above any of them is at least p Z.
// The window spans at most WIN keys below the maximum; the slack terms keep
// the float evaluation on the safe side.  Empty (wlo > whi) if M is not finite.
__device__ __forceinline__ void candidate_window(float M, int L, float Z, float tau, float p,
                                                 bool k_on, int& whi, int& wlo) {
  whi = 0;
  wlo = 1;
  if (M > -INFINITY && M < INFINITY) {
    whi = okey_of(M);
    wlo = max(0, whi - (WIN - 1));
    if (k_on) {
      wlo = max(wlo, L);
    } else {
      const float lnz = fmaxf(0.0f, logf(Z * 0.9999f));
      const float width =
          tau * (logf(static_cast<float>(VREAL) / (1.0f - p)) * 1.0001f + 1e-3f - lnz);
      wlo = max(wlo, okey_floor(M - width));
    }
    wlo = max(wlo, KEY_NEG_INF);
  }
}

// ------------------------------------------------------------ selection

// Exclusive block scan of (count, mass); also returns the block totals.
template <class SM>
__device__ __forceinline__ void block_excl_scan(uint32_t c, unsigned long long m, uint32_t& ec,
                                                unsigned long long& em, uint32_t& tc,
                                                unsigned long long& tm, SM& S) {
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

struct SelResult { uint32_t support; unsigned long long zs; int min_key; };

// Count the row's real elements whose key lies in [wlo, whi] (global memory
// re-read; fallback for supports that reach below the first window).
__device__ inline void count_window_global(const uint16_t* rowp, int wlo, int whi, uint32_t* cnt) {
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

template <class SM>
__device__ __forceinline__ WinScan scan_window(const uint32_t* cnt, int n, int whi, float M, float c,
                                               uint32_t carry_c, unsigned long long carry_m,
                                               SM& S) {
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
template <class SM>
__device__ __noinline__ SelResult select_support(SM& S, uint32_t* cnt0, uint32_t* cntB, int hi,
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
// common case).  Keys hi, hi-1, ..., lo are taken in blocks of 32 x
// RLK_SEL_KPL (consecutive keys per lane; 4 measured fastest, 8 slower).  A
// top-k row whose k-th key lies in the first block is resolved in one pass
// over it (counts and fixed-point masses scanned together: the k-th key, the
// mass of S_k, then the nucleus boundary from the same registers); otherwise
// a scan of the counts alone finds the top-k boundary, then one scan of the
// masses over S_k finds the nucleus boundary.  Returns false if a threshold
// may lie below the window.
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
  constexpr int KPL = RLK_SEL_KPL;   // consecutive keys per lane in a block
  constexpr int BLK = KPL * 32;
  const int lane = threadIdx.x & 31;
  const int n = hi - lo + 1;
  int imax = n - 1;
  uint32_t sup_k = 0;
  // ---- top-k rows whose k-th key lies in the first block: counts, masses,
  // the k-th key and the nucleus in one pass over that block
  uint32_t carry0 = 0;          // counts of the blocks already scanned for the k-th key
  int b_start = 0;
  if (k_on) {
    uint32_t cj[KPL], lc = 0;
    unsigned long long mj[KPL], lm = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      const int i = KPL * lane + j;
      cj[j] = (i < n) ? cnt[i] : 0u;
      mj[j] = cj[j] ? cj[j] * qfx(key_value(hi - i), M, c) : 0ull;
      lc += cj[j];
      lm += mj[j];
    }
    const uint32_t ic = warp_incl_scan_u32(lc);
    const unsigned long long im = warp_incl_scan_u64(lm);
    // the k-th key: the first whose inclusive count reaches k
    uint32_t rc = ic - lc;
    unsigned long long rm = im - lm;
    int f = -1;
    uint32_t fc = 0;
    unsigned long long fm = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      if (f < 0 && rc < static_cast<uint32_t>(k) && rc + cj[j] >= static_cast<uint32_t>(k)) {
        f = KPL * lane + j;
        fc = rc + cj[j];
        fm = rm + mj[j];
      }
      rc += cj[j];
      rm += mj[j];
    }
    const unsigned bal = __ballot_sync(0xffffffffu, f >= 0);
    if (bal) {
      const int src = __ffs(bal) - 1;
      const int fi = __shfl_sync(0xffffffffu, f, src);
      const uint32_t skc = __shfl_sync(0xffffffffu, fc, src);
      const unsigned long long zk = __shfl_sync(0xffffffffu, fm, src);   // the mass of S_k
      if (!p_on) {
        out = SelResult{skc, zk, hi - fi};
        return true;
      }
      const unsigned long long T = nucleus_bound(p, zk);
      rc = ic - lc;
      rm = im - lm;
      int g = -1;
      uint32_t gc = 0;
      unsigned long long gm = 0;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        const int i = KPL * lane + j;
        if (g < 0 && i <= fi && rm < T && (rm + mj[j] >= T || i == fi)) {
          g = i;
          gc = rc + cj[j];
          gm = rm + mj[j];
        }
        rc += cj[j];
        rm += mj[j];
      }
      const unsigned bg = __ballot_sync(0xffffffffu, g >= 0);
      if (bg) {                          // (always: the maximum's own mass makes T >= 1)
        const int sg = __ffs(bg) - 1;
        out = SelResult{__shfl_sync(0xffffffffu, gc, sg), __shfl_sync(0xffffffffu, gm, sg),
                        hi - __shfl_sync(0xffffffffu, g, sg)};
        return true;
      }
    } else {
      // the k-th key lies further down: the count scan goes on from the next block
      carry0 = __shfl_sync(0xffffffffu, ic, 31);
      b_start = BLK;
    }
  }
  // ---- top-k boundary from the counts
  if (k_on) {
    uint32_t carry = carry0;
    int fi = -1;
    for (int b0 = b_start; b0 < n && fi < 0; b0 += BLK) {
      uint32_t cj[KPL], lc = 0;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        const int i = b0 + KPL * lane + j;
        cj[j] = (i < n) ? cnt[i] : 0u;
        lc += cj[j];
      }
      const uint32_t ic = warp_incl_scan_u32(lc);
      uint32_t rc = carry + ic - lc;
      int f = -1;
      uint32_t fc = 0;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        if (f < 0 && rc < static_cast<uint32_t>(k) && rc + cj[j] >= static_cast<uint32_t>(k)) {
          f = b0 + KPL * lane + j;
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
      for (int j = 0; j < KPL; ++j) {
        const int i = b0 + KPL * lane + j;
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
    uint32_t cj[KPL], lc = 0;
    unsigned long long mj[KPL], lm = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      const int i = b0 + KPL * lane + j;
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
    for (int j = 0; j < KPL; ++j) {
      const int i = b0 + KPL * lane + j;
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

// ------------------------------------------------------------ backward

// The gradient of g_full * full + g_restr * restr at column j of a resolved
// row is  -e_j * (key_j >= min_key ? a_in : a_out) + (j == t ? b : 0)  with
// e_j = exp((x_j - M) / tau), a_out = g_full / (Z tau), a_in = a_out +
// g_restr / (Z_S tau) and b = (g_full + g_restr) / tau, the restricted terms
// dropped when the target is outside the support (inv_z_support == 0).
// Products and sums are explicitly rounded (no contraction), so every kernel
// that forms a gradient from the same record gets the same bits.
enum : uint32_t { GRAD_VALUES = 0u, GRAD_ZERO = 1u, GRAD_NAN = 2u };
struct GradCoeffs {
  float M, c, a_in, a_out, b;
  int min_key;
  uint32_t mode;
};

__device__ __forceinline__ rlk_row_stats nan_stats() {
  rlk_row_stats st;
  st.max_logit = __int_as_float(0x7fc00000);
  st.inv_z = __int_as_float(0x7fc00000);
  st.inv_z_support = 0.0f;
  st.min_key = 0;
  return st;
}

__device__ __forceinline__ GradCoeffs nan_coeffs() {
  GradCoeffs g{};
  g.mode = GRAD_NAN;
  return g;
}

__device__ __forceinline__ GradCoeffs grad_coeffs(const rlk_row_stats& st, float tau, float gf,
                                                  float gr) {
  GradCoeffs g{};
  if (st.inv_z != st.inv_z) {
    g.mode = GRAD_NAN;
  } else if (tau == 0.0f) {
    g.mode = GRAD_ZERO;               // greedy: the logprobs are piecewise constant
  } else {
    const float rt = __fdiv_rn(1.0f, tau);
    const float grs = st.inv_z_support != 0.0f ? gr : 0.0f;
    g.mode = GRAD_VALUES;
    g.M = st.max_logit;
    g.c = __fdiv_rn(LOG2E, tau);
    g.a_out = __fmul_rn(__fmul_rn(gf, st.inv_z), rt);
    g.a_in = __fadd_rn(g.a_out, __fmul_rn(__fmul_rn(grs, st.inv_z_support), rt));
    g.b = __fmul_rn(__fadd_rn(gf, grs), rt);
    g.min_key = st.min_key;
  }
  return g;
}

// Store 8 gradient values of chunk ch (columns 8ch .. 8ch+7 of the shard),
// streaming (evict-first) stores.
__device__ __forceinline__ void store_grad8(char* gshard, int ch, bool f32, const float (&g)[8]) {
  if (f32) {
    uint4* dst = reinterpret_cast<uint4*>(gshard + static_cast<int64_t>(ch) * 32);
    __stcs(dst, make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                           __float_as_uint(g[3])));
    __stcs(dst + 1, make_uint4(__float_as_uint(g[4]), __float_as_uint(g[5]), __float_as_uint(g[6]),
                               __float_as_uint(g[7])));
  } else {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * j], g[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    __stcs(reinterpret_cast<uint4*>(gshard + static_cast<int64_t>(ch) * 16),
           make_uint4(w[0], w[1], w[2], w[3]));
  }
}

// One shard of a gradient row: the shard's real columns from its logits
// (shared memory, or global memory when src_global), zeros on the padded
// columns of the last shard.  col0 is the shard's first vocabulary column.
__device__ __forceinline__ void write_grad_shard(const uint4* src, bool src_global, int nchunks,
                                                 int col0, int t, const GradCoeffs& m,
                                                 char* gshard, bool f32) {
  const uint64_t nxm2 = pack2(-m.M, -m.M);
  const uint64_t c2 = pack2(m.c, m.c);
  for (int ch = threadIdx.x; ch < SHARD_CHUNKS; ch += NTHR) {
    float g[8];
    if (ch >= nchunks || m.mode == GRAD_ZERO) {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = 0.0f;
    } else if (m.mode == GRAD_NAN) {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = __int_as_float(0x7fc00000);
    } else {
      const uint4 v = src_global ? __ldg(src + ch) : src[ch];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t a = mul2(add2(pack2(bf16_lo(w[j]), bf16_hi(w[j])), nxm2), c2);
        float a0, a1;
        unpack2(a, a0, a1);
        const float k0 = okey(w[j] & 0xFFFFu) >= m.min_key ? m.a_in : m.a_out;
        const float k1 = okey(w[j] >> 16) >= m.min_key ? m.a_in : m.a_out;
        g[2 * j] = __fmul_rn(-ex2(a0), k0);
        g[2 * j + 1] = __fmul_rn(-ex2(a1), k1);
      }
      const int lt = t - col0 - ch * 8;
      if (lt >= 0 && lt < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j == lt) g[j] = __fadd_rn(g[j], m.b);
      }
    }
    store_grad8(gshard, ch, f32, g);
  }
}

// ------------------------------------------------------------ sampling

// Word 0 of Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011): key (seed low, seed high),
// counter (ctr low, ctr high, 0, 0).  Each round multiplies words 0 and 2 by
// the round constants, xors the high halves with words 1 and 3 and the round
// key, and the key steps by the Weyl increments between rounds.
__device__ __forceinline__ uint32_t philox_word0(unsigned long long seed, unsigned long long ctr) {
  uint32_t c0 = static_cast<uint32_t>(ctr), c1 = static_cast<uint32_t>(ctr >> 32), c2 = 0u, c3 = 0u;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  return c0;
}

// floor(u * z / 2^32) for a 32-bit draw u and a fixed-point mass z < 2^63.
__device__ __forceinline__ unsigned long long scale_draw(uint32_t u, unsigned long long z) {
  const unsigned long long lo = z * static_cast<unsigned long long>(u);
  const unsigned long long hi = __umul64hi(z, static_cast<unsigned long long>(u));
  return (hi << 32) | (lo >> 32);
}

// Support elements of one 16-byte chunk: those >= vmin (the value of the
// support's lowest key; -inf when the support is the whole vocabulary), as a
// mask with bit j for column 2j and bit 16 + j for column 2j + 1 of the chunk.
__device__ __forceinline__ uint32_t chunk_support_bits(uint4 v, __nv_bfloat162 vmin2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) bits |= (__hge2_mask(as_bf2(w[j]), vmin2) & 0x00010001u) << j;
  return bits;
}

// Fixed-point mass (2^-44 units, the selection's per-key values) of a chunk's
// support elements; the exponentials are evaluated for those elements only.
__device__ __forceinline__ unsigned long long chunk_support_mass(uint4 v, __nv_bfloat162 vmin2, float M,
                                                                 float c) {
  uint32_t bits = chunk_support_bits(v, vmin2);
  unsigned long long m = 0;
  if (bits == 0x000F000Fu) {
    // every element in the support: the same per-element values as qfx (IEEE
    // round-to-nearest subtract and multiply, ex2.approx, exact 2^44 scaling),
    // two columns at a time
    const uint64_t nm2 = pack2(-M, -M), c2 = pack2(c, c), s2 = pack2(FX_SCALE, FX_SCALE);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a0, a1, q0, q1;
      unpack2(mul2(add2(pack2(bf16_lo(w[j]), bf16_hi(w[j])), nm2), c2), a0, a1);
      unpack2(mul2(pack2(ex2(a0), ex2(a1)), s2), q0, q1);
      m += fx_round(q0) + fx_round(q1);
    }
    return m;
  }
  while (bits) {
    const int pos = __ffs(bits) - 1;
    bits &= bits - 1;
    const int j = pos & 3;
    const uint32_t wj = (j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w;
    const uint32_t b = (pos & 16) ? (wj >> 16) : (wj & 0xFFFFu);
    m += qfx(__uint_as_float(b << 16), M, c);
  }
  return m;
}

}  // namespace rlk
