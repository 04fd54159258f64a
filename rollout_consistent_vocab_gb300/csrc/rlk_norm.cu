// rlk_norm.cu -- deterministic gradient L2 norm for GB300 (sm_103a): the
// exact sum of the FP32 squares of the elements, gathered in integer bins
// keyed by exponent ("H100 canonical CP backward validation", section
// "Change": Megatron's L2 norm sums FP32 gradient squares in integer
// exponent bins before the distributed reduction).  Integers add exactly in
// any order, so the sum depends neither on element order, nor on the launch
// shape, nor on how the elements are split across ranks.
//
// A square q = M 2^(E-150) (M < 2^24) is an integer multiple of 2^(E-150).
// Instead of one shared-memory add per element, each thread keeps a 128-bit
// fixed-point accumulator whose unit is 2^(eb-150).  A square with
// eb <= E <= eb + 31 adds M << (E - eb) (< 2^55) to a 64-bit batch sum,
// folded into the 128-bit value after every batch of at most 32 squares.  A
// square above that window moves the window up, to 8 binades above it: the
// accumulator's low bits that would fall out are first written to the bins
// in 24-bit pieces.  A
// square below it goes straight to its own bin.  At the end the thread writes
// its accumulator to the bins in 24-bit pieces.  Every step is exact, so the
// bins hold the exact sum of the squares; only how that value is split over
// the entries depends on the order.  A block's bins live in shared memory and
// reach the caller's bins with one global atomic add per nonzero entry.
//
// BF16 and FP16 inputs take a shorter route (sqnorm16_kernel): a block counts
// the 32768 possible magnitudes and converts the counts into bin
// contributions at the end.
//
// The finalize kernel forms the exact sum as a multi-word integer, rounds it
// once to float64 (nearest even) and takes the correctly rounded square root.

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "rlk_norm.h"
#include "rlk_host.h"

namespace rlk {
namespace {

constexpr int NB = RLK_NORM_BINS;
constexpr int NAN_BIN = 0;
constexpr int INF_BIN = NB - 1;
constexpr int WIN_BINADES = 31;    // window of a thread accumulator: M << 31 < 2^55
constexpr int HEADROOM = 8;        // binades left above a new largest square when the window moves
constexpr int PIECE = 24;          // bits per piece written to a bin (each increment < 2^24)
constexpr int NORM_THREADS = 256;
#ifndef NORM_MIN_BLOCKS
#define NORM_MIN_BLOCKS 4     // 64 registers: 4 blocks of 256 threads per SM
#endif
// 16-byte loads per batch (two batches in flight): measured best at 4 for
// FP32 and 2 for the 16-bit types, whose 8 squares per vector make the loop
// longer.  A batch sum takes at most 32 terms of < 2^55 (plus a remainder of
// fewer) before it is folded.
template <int DT>
__host__ __device__ constexpr int norm_unroll() { return DT == RLK_DT_F32 ? 4 : 2; }
static_assert(4 * 4 <= 128 && 2 * 8 <= 128, "batch sum capacity");

struct Acc {
  int eb;                          // the accumulator's unit is 2^(eb - 150)
  unsigned long long lo, hi;       // its 128-bit value
  unsigned long long s;            // batch sum in the same unit (at most 255 terms < 2^55)
  uint32_t nan, inf;               // NaN and infinite squares seen
};

__device__ __forceinline__ void add128(unsigned long long& lo, unsigned long long& hi,
                                       unsigned long long v) {
  asm("add.cc.u64 %0, %0, %2;\n\taddc.u64 %1, %1, 0;" : "+l"(lo), "+l"(hi) : "l"(v));
}

// The batch sum into the 128-bit value.
__device__ __forceinline__ void acc_fold(Acc& a) {
  add128(a.lo, a.hi, a.s);
  a.s = 0ull;
}

__device__ __forceinline__ void bin_add(unsigned long long* sb, int e, unsigned long long v) {
  if (v) atomicAdd(&sb[e], v);
}

// Bits [at, at + n) of the 128-bit value (0 <= at < 128, 1 <= n <= 24).
__device__ __forceinline__ unsigned long long bits128(unsigned long long lo, unsigned long long hi,
                                                      int at, int n) {
  unsigned long long w;
  if (at == 0) w = lo;
  else if (at < 64) w = (lo >> at) | (hi << (64 - at));
  else w = hi >> (at - 64);
  return w & ((1ull << n) - 1ull);
}

// Write the accumulator's low k bits to the bins (pieces of PIECE bits at
// entries eb, eb + PIECE, ...) and shift them out: the unit becomes
// 2^(eb + k - 150).  Entries stay below eb + 128 <= 350 < INF_BIN.  Inlined:
// an out-of-line call anywhere in the element loop made the loop several
// times slower.
struct Acc128 { int eb; unsigned long long lo, hi; };

__device__ __forceinline__ Acc128 acc_spill_low(Acc128 a, int k, unsigned long long* sb) {
  for (int at = 0; at < k && at < 128; at += PIECE)
    bin_add(sb, a.eb + at, bits128(a.lo, a.hi, at, min(PIECE, k - at)));
  if (k >= 128) {
    a.lo = 0ull;
    a.hi = 0ull;
  } else if (k >= 64) {
    a.lo = a.hi >> (k - 64);
    a.hi = 0ull;
  } else if (k > 0) {
    a.lo = (a.lo >> k) | (a.hi << (64 - k));
    a.hi >>= k;
  }
  a.eb += k;
  return a;
}

__device__ __forceinline__ void acc_spill(Acc& a, int k, unsigned long long* sb) {
  const Acc128 r = acc_spill_low(Acc128{a.eb, a.lo, a.hi}, k, sb);
  a.eb = r.eb;
  a.lo = r.lo;
  a.hi = r.hi;
}

// One FP32 square, by its bits u: every case (the batch sum is folded
// first if the window moves).
__device__ __forceinline__ void acc_add(Acc& a, uint32_t u, unsigned long long* sb) {
  const int E = static_cast<int>((u >> 23) & 0xFFu);
  const uint32_t f = u & 0x7FFFFFu;
  if (E == 0xFF) {                 // NaN or infinite square
    if (f) ++a.nan;
    else ++a.inf;
    return;
  }
  const int e = max(E, 1);         // a subnormal square: unit 2^-149, as for E == 1
  const uint32_t M = E ? (f | 0x800000u) : f;
  int d = e - a.eb;
  if (static_cast<unsigned>(d) > static_cast<unsigned>(WIN_BINADES)) {
    if (d < 0) {                   // below the window: straight to its bin
      bin_add(sb, e, M);
      return;
    }
    // a new largest square: move the window up, leaving HEADROOM binades above
    // it, but never past eb = 254 - 31, so that an exponent field of 255 (NaN,
    // infinity) stays outside the window
    acc_fold(a);
    acc_spill(a, min(e - (WIN_BINADES - HEADROOM), 254 - WIN_BINADES) - a.eb, sb);
    d = e - a.eb;
  }
  add128(a.lo, a.hi, static_cast<unsigned long long>(M) << d);
}

// The common case, without branches: a square inside the window joins the
// batch sum.  Returns true for a square it leaves to acc_add: nonzero and
// outside the window (including NaN and infinite squares, whose exponent
// field is above eb + 31 because eb <= 254 - 31).
__device__ __forceinline__ bool acc_fast(Acc& a, uint32_t u) {
  const uint32_t d = (u >> 23) - static_cast<uint32_t>(a.eb);   // a NaN's sign bit makes d large
  // 2^d, or 0 outside the window: the shift amount is clamped at 32, and
  // the window is d <= 31 (WIN_BINADES)
  uint32_t p2;
  asm("shl.b32 %0, 1, %1;" : "=r"(p2) : "r"(d));
  // M 2^d joins the batch sum as one widening multiply-add
  asm("mad.wide.u32 %0, %1, %2, %0;" : "+l"(a.s) : "r"((u & 0x7FFFFFu) | 0x800000u), "r"(p2));
  return p2 == 0u && u != 0u;
}
static_assert(WIN_BINADES == 31, "acc_fast's window is the range of a 32-bit shift");

// The FP32 square of one element, rounded to nearest even.
template <int DT>
__device__ __forceinline__ uint32_t square_bits(uint32_t raw) {
  float g;
  if (DT == RLK_DT_F32) g = __uint_as_float(raw);
  else if (DT == RLK_DT_BF16) g = __uint_as_float(raw << 16);
  else g = __half2float(__ushort_as_half(static_cast<unsigned short>(raw)));
  return __float_as_uint(__fmul_rn(g, g));
}

// The FP32 squares of two FP32 elements (raw bits), one packed product
// rounded to nearest even in each lane.
__device__ __forceinline__ void square2(uint32_t x0, uint32_t x1, uint32_t& q0, uint32_t& q1) {
  unsigned long long p;
  asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tmul.rn.f32x2 %0, t, t;\n\t}"
      : "=l"(p) : "r"(x0), "r"(x1));
  q0 = static_cast<uint32_t>(p);
  q1 = static_cast<uint32_t>(p >> 32);
}

// Element j of a 16-byte vector (raw bits; j may be a runtime value).
template <int DT>
__device__ __forceinline__ uint32_t vec_elem(const uint4& v, int j) {
  const int wi = DT == RLK_DT_F32 ? j : (j >> 1);
  const uint32_t w = wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
  if (DT == RLK_DT_F32) return w;
  return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}

template <int DT>
__device__ __forceinline__ void acc_vec(Acc& a, const uint4& v, unsigned long long* sb) {
  constexpr int NQ = DT == RLK_DT_F32 ? 4 : 8;
  const int eb0 = a.eb;
  bool rest = false;
  if (DT == RLK_DT_F32) {
    // the four squares as two packed products (each lane rounded as a scalar product)
    uint32_t q[4];
    square2(v.x, v.y, q[0], q[1]);
    square2(v.z, v.w, q[2], q[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) rest |= acc_fast(a, q[j]);
  } else {
#pragma unroll
    for (int j = 0; j < NQ; ++j) rest |= acc_fast(a, square_bits<DT>(vec_elem<DT>(v, j)));
  }
  if (rest) {                      // rare: the squares acc_fast left, by its own test at eb0
#pragma unroll 1
    for (int j = 0; j < NQ; ++j) {
      const uint32_t u = square_bits<DT>(vec_elem<DT>(v, j));
      if ((u >> 23) - static_cast<uint32_t>(eb0) > static_cast<uint32_t>(WIN_BINADES) && u != 0u)
        acc_add(a, u, sb);
    }
  }
}

template <int DT>
__device__ __forceinline__ uint32_t load_elem(const char* x, int64_t i) {
  if (DT == RLK_DT_F32) return __ldg(reinterpret_cast<const uint32_t*>(x) + i);
  return __ldg(reinterpret_cast<const unsigned short*>(x) + i);
}

// x: the elements; the first `head` of them precede a 16-byte boundary, then
// nvec 16-byte vectors, then the rest up to n.  Block 0 also takes the head
// and the tail.
template <int DT>
__global__ void __launch_bounds__(NORM_THREADS, NORM_MIN_BLOCKS) sqnorm_kernel(const char* x, int64_t head,
                                                              int64_t nvec, int64_t n,
                                                              unsigned long long* bins) {
  __shared__ unsigned long long sb[NB];
  for (int i = threadIdx.x; i < NB; i += NORM_THREADS) sb[i] = 0ull;
  __syncthreads();

  constexpr int ES = DT == RLK_DT_F32 ? 4 : 2;
  constexpr int PER = 16 / ES;
  constexpr int NORM_UNROLL = norm_unroll<DT>();
  Acc a{1, 0ull, 0ull, 0ull, 0u, 0u};
  const uint4* vx = reinterpret_cast<const uint4*>(x + head * ES);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * NORM_THREADS;
  int64_t i = static_cast<int64_t>(blockIdx.x) * NORM_THREADS + threadIdx.x;
  // batches of NORM_UNROLL vectors; the next batch's loads go out before the
  // current batch is summed
  uint4 v[NORM_UNROLL];
  bool have = i + (NORM_UNROLL - 1) * stride < nvec;
  if (have) {
#pragma unroll
    for (int u = 0; u < NORM_UNROLL; ++u) v[u] = __ldg(vx + i + u * stride);
  }
  while (have) {
    const int64_t j = i + NORM_UNROLL * stride;
    const bool more = j + (NORM_UNROLL - 1) * stride < nvec;
    uint4 w[NORM_UNROLL];
    if (more) {
#pragma unroll
      for (int u = 0; u < NORM_UNROLL; ++u) w[u] = __ldg(vx + j + u * stride);
    }
#pragma unroll
    for (int u = 0; u < NORM_UNROLL; ++u) acc_vec<DT>(a, v[u], sb);
    acc_fold(a);                   // at most 32 terms since the last fold
    if (more) {
#pragma unroll
      for (int u = 0; u < NORM_UNROLL; ++u) v[u] = w[u];
    }
    i = j;
    have = more;
  }
  for (; i < nvec; i += stride) acc_vec<DT>(a, __ldg(vx + i), sb);
  if (blockIdx.x == 0) {
    const int64_t tail0 = head + nvec * PER;
    const int64_t nrest = head + (n - tail0);
    for (int64_t j = threadIdx.x; j < nrest; j += NORM_THREADS)
      acc_add(a, square_bits<DT>(load_elem<DT>(x, j < head ? j : tail0 + (j - head))), sb);
  }

  acc_fold(a);
  acc_spill(a, 128, sb);
  if (a.nan) atomicAdd(&sb[NAN_BIN], static_cast<unsigned long long>(a.nan));
  if (a.inf) atomicAdd(&sb[INF_BIN], static_cast<unsigned long long>(a.inf));
  __syncthreads();
  for (int e = threadIdx.x; e < NB; e += NORM_THREADS) {
    const unsigned long long v = sb[e];
    if (v) atomicAdd(&bins[e], v);
  }
}

// ---------------------------------------------------------------- 16-bit types
//
// A BF16 or FP16 square depends only on the element's 15 magnitude bits, so
// a block counts each of the 32768 magnitudes in shared memory (one add per
// element; zeros add nothing) and at the end adds, for every magnitude
// present, count x its FP32 square's significand to the square's bin (NaN
// and infinite squares to their counters): the same exact sum, with no
// per-element arithmetic beyond the add.

// Both 15-bit magnitudes of a 32-bit word add one to their counters at byte
// address base + 4 m, each add a predicated instruction (zero magnitudes add
// nothing and issue nothing): no branch per element.
__device__ __forceinline__ void count_mag_pair(uint32_t w, uint32_t base) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b32 m0, m1, a0, a1;\n\t"
      "and.b32 m0, %0, 32767;\n\t"
      "shr.b32 m1, %0, 16;\n\t"
      "and.b32 m1, m1, 32767;\n\t"
      "setp.ne.u32 p0, m0, 0;\n\t"
      "setp.ne.u32 p1, m1, 0;\n\t"
      "mad.lo.u32 a0, m0, 4, %1;\n\t"
      "mad.lo.u32 a1, m1, 4, %1;\n\t"
      "@p0 red.shared.add.u32 [a0], 1;\n\t"
      "@p1 red.shared.add.u32 [a1], 1;\n\t}"
      :: "r"(w), "r"(base) : "memory");
}

constexpr int H16_THREADS = 1024;
constexpr int H16_MIN_VEC = 8;    // 16-byte vectors per thread below which fewer blocks run
constexpr int NPAT = 32768;
constexpr uint32_t H16_SMEM = NPAT * 4u;

template <int DT>
__global__ void __launch_bounds__(H16_THREADS, 1) sqnorm16_kernel(const char* x, int64_t head,
                                                                  int64_t nvec, int64_t n,
                                                                  unsigned long long* bins) {
  extern __shared__ __align__(16) uint32_t cnt[];   // [NPAT] counts per magnitude
  __shared__ unsigned long long sb[NB];
  const int tid = threadIdx.x;
  for (int i = tid; i < NPAT / 4; i += H16_THREADS) reinterpret_cast<uint4*>(cnt)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < NB; i += H16_THREADS) sb[i] = 0ull;
  __syncthreads();
  const uint32_t cbase = static_cast<uint32_t>(__cvta_generic_to_shared(cnt));
  auto add2 = [&](uint32_t w) { count_mag_pair(w, cbase); };   // the two elements of a word
  const uint4* vx = reinterpret_cast<const uint4*>(x + head * 2);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * H16_THREADS;
  int64_t i = static_cast<int64_t>(blockIdx.x) * H16_THREADS + tid;
  for (; i + 3 * stride < nvec; i += 4 * stride) {  // four vectors in flight
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(vx + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      add2(v[u].x);
      add2(v[u].y);
      add2(v[u].z);
      add2(v[u].w);
    }
  }
  for (; i < nvec; i += stride) {
    const uint4 v = __ldg(vx + i);
    add2(v.x);
    add2(v.y);
    add2(v.z);
    add2(v.w);
  }
  if (blockIdx.x == 0) {
    const int64_t tail0 = head + nvec * 8;
    const int64_t nrest = head + (n - tail0);
    for (int64_t j = tid; j < nrest; j += H16_THREADS) {
      const uint32_t m = load_elem<DT>(x, j < head ? j : tail0 + (j - head)) & 0x7FFFu;
      if (m) atomicAdd(&cnt[m], 1u);
    }
  }
  __syncthreads();
  unsigned long long nan_c = 0ull, inf_c = 0ull;
  for (int m = tid; m < NPAT; m += H16_THREADS) {
    const uint32_t c = cnt[m];
    if (!c) continue;
    const uint32_t u = square_bits<DT>(static_cast<uint32_t>(m));
    const int E = static_cast<int>((u >> 23) & 0xFFu);
    const uint32_t f = u & 0x7FFFFFu;
    if (E == 0xFF) {
      if (f) nan_c += c;
      else inf_c += c;
      continue;
    }
    const uint32_t M = E ? (f | 0x800000u) : f;    // a subnormal square: unit 2^-149, as E = 1
    if (M) atomicAdd(&sb[max(E, 1)], static_cast<unsigned long long>(c) * M);
  }
  if (nan_c) atomicAdd(&sb[NAN_BIN], nan_c);
  if (inf_c) atomicAdd(&sb[INF_BIN], inf_c);
  __syncthreads();
  for (int e = tid; e < NB; e += H16_THREADS) {
    const unsigned long long v = sb[e];
    if (v) atomicAdd(&bins[e], v);
  }
}

// ---------------------------------------------------------------- finalize

constexpr int ND = 16;             // 32-bit digits: 512 bits > 381 + 64

// Bits [at, at + 53) of the digit string (at + 64 <= 32 * ND).
__device__ __forceinline__ unsigned long long digits53(const uint32_t* D, int at) {
  const int i = at >> 5, o = at & 31;
  unsigned long long w = static_cast<unsigned long long>(D[i]) |
                         (static_cast<unsigned long long>(D[i + 1]) << 32);
  if (o) w = (w >> o) | (static_cast<unsigned long long>(D[i + 2]) << (64 - o));
  return w & ((1ull << 53) - 1ull);
}

// Any of bits [0, at) set.
__device__ __forceinline__ bool digits_below(const uint32_t* D, int at) {
  const int i = at >> 5, o = at & 31;
  for (int j = 0; j < i; ++j)
    if (D[j]) return true;
  return o && (D[i] & ((1u << o) - 1u));
}

// One warp.  N = sum_e bins[e] 2^(e-1) is the exact sum in units of 2^-149;
// lanes add the bins into 32-bit digits kept with headroom in 64-bit words,
// lane 0 propagates the carries, rounds N 2^-149 to float64 and takes the
// square root.
__global__ void sqnorm_finalize_kernel(const unsigned long long* bins, double* out) {
  __shared__ unsigned long long dig[ND];
  const int lane = threadIdx.x;
  if (lane < ND) dig[lane] = 0ull;
  // every load first (independent), then the adds
  constexpr int PER_LANE = (INF_BIN - 1 + 31) / 32;
  unsigned long long vb[PER_LANE];
#pragma unroll
  for (int q = 0; q < PER_LANE; ++q) {
    const int e = 1 + lane + 32 * q;
    vb[q] = e < INF_BIN ? bins[e] : 0ull;
  }
  const unsigned long long nan_b = bins[NAN_BIN], inf_b = bins[INF_BIN];
  __syncwarp();
#pragma unroll
  for (int q = 0; q < PER_LANE; ++q) {
    const int e = 1 + lane + 32 * q;
    const unsigned long long v = vb[q];
    if (!v) continue;
    const int s = e - 1, L = s >> 5, sh = s & 31;
    const unsigned long long lo = v << sh;
    const unsigned long long hi = sh ? (v >> (64 - sh)) : 0ull;
    atomicAdd(&dig[L], lo & 0xFFFFFFFFull);
    atomicAdd(&dig[L + 1], lo >> 32);
    if (hi) atomicAdd(&dig[L + 2], hi);
  }
  __syncwarp();
  if (lane != 0) return;
  if (nan_b) {
    out[0] = out[1] = __longlong_as_double(0x7ff8000000000000ll);
    return;
  }
  if (inf_b) {
    out[0] = out[1] = __longlong_as_double(0x7ff0000000000000ll);
    return;
  }
  uint32_t D[ND];
  unsigned long long c = 0ull;
#pragma unroll
  for (int i = 0; i < ND; ++i) {
    const unsigned long long t = dig[i] + c;
    D[i] = static_cast<uint32_t>(t);
    c = t >> 32;
  }
  int top = ND - 1;
  while (top >= 0 && D[top] == 0u) --top;
  double s = 0.0;
  if (top >= 0) {
    const int p = 32 * top + 31 - __clz(D[top]);      // leading bit of N
    unsigned long long m;
    int b0 = 0;                                       // N rounded = m 2^b0
    if (p <= 52) {
      m = static_cast<unsigned long long>(D[0]) | (static_cast<unsigned long long>(D[1]) << 32);
    } else {
      b0 = p - 52;
      m = digits53(D, b0);
      const bool r = (D[(b0 - 1) >> 5] >> ((b0 - 1) & 31)) & 1u;
      if (r && (digits_below(D, b0 - 1) || (m & 1ull))) {
        ++m;
        if (m >> 53) {
          m >>= 1;
          ++b0;
        }
      }
    }
    // m < 2^53 converts exactly; the result is far inside the normal range
    s = scalbn(static_cast<double>(m), b0 - 149);
  }
  out[0] = s;
  out[1] = __dsqrt_rn(s);
}

int norm_grid(int64_t nvec) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  int& slots = cached[dev & 63];
  if (slots == 0) {
    int sms = 0, per = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, sqnorm_kernel<RLK_DT_F32>, NORM_THREADS, 0);
    slots = std::max(1, sms) * std::max(1, per);
  }
  const int64_t want = (nvec + NORM_THREADS * 8 - 1) / (NORM_THREADS * 8);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, slots)));
}

}  // namespace
}  // namespace rlk

using namespace rlk;

extern "C" rlk_status rlk_sqnorm_accumulate(const void* x, int64_t n, int32_t dtype, uint64_t* bins,
                                            void* stream) {
  if (dtype != RLK_DT_F32 && dtype != RLK_DT_BF16 && dtype != RLK_DT_F16)
    return fail(RLK_EINVAL, "dtype %d is not RLK_DT_F32, RLK_DT_BF16 or RLK_DT_F16", dtype);
  if (n < 0 || n > (int64_t(1) << 36)) return fail(RLK_EINVAL, "n = %lld must be in [0, 2^36]", (long long)n);
  if (!bins) return fail(RLK_EINVAL, "bins is NULL");
  if (!aligned(bins, 8)) return fail(RLK_EALIGN, "bins is not 8-byte aligned");
  if (n == 0) return RLK_OK;
  if (!x) return fail(RLK_EINVAL, "x is NULL");
  const int es = dtype == RLK_DT_F32 ? 4 : 2;
  if (!aligned(x, es)) return fail(RLK_EALIGN, "x is not aligned to its %d-byte elements", es);
  const int64_t head = std::min<int64_t>(n, ((16 - (reinterpret_cast<uintptr_t>(x) & 15)) & 15) / es);
  const int64_t nvec = (n - head) / (16 / es);
  const int grid = norm_grid(nvec);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* xc = static_cast<const char*>(x);
  unsigned long long* b = reinterpret_cast<unsigned long long*>(bins);
  if (dtype == RLK_DT_F32) {
    sqnorm_kernel<RLK_DT_F32><<<grid, NORM_THREADS, 0, st>>>(xc, head, nvec, n, b);
  } else {
    // one block per SM (128 KB of counts each), fewer for small inputs
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    if (!configured[dev & 63]) {
      cudaError_t e = cudaFuncSetAttribute(sqnorm16_kernel<RLK_DT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(H16_SMEM));
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sqnorm16_kernel<RLK_DT_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(H16_SMEM));
      if (e != cudaSuccess) return fail(RLK_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      configured[dev & 63] = true;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (nvec + H16_THREADS * H16_MIN_VEC - 1) / (H16_THREADS * H16_MIN_VEC);
    const unsigned g16 = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(want, std::max(1, sms))));
    if (dtype == RLK_DT_BF16) sqnorm16_kernel<RLK_DT_BF16><<<g16, H16_THREADS, H16_SMEM, st>>>(xc, head, nvec, n, b);
    else sqnorm16_kernel<RLK_DT_F16><<<g16, H16_THREADS, H16_SMEM, st>>>(xc, head, nvec, n, b);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

extern "C" rlk_status rlk_sqnorm_finalize(const uint64_t* bins, double* out, void* stream) {
  if (!bins || !out) return fail(RLK_EINVAL, "bins and out are required");
  if (!aligned(bins, 8) || !aligned(out, 8)) return fail(RLK_EALIGN, "bins and out must be 8-byte aligned");
  sqnorm_finalize_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const unsigned long long*>(bins), out);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(RLK_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
  return RLK_OK;
}

extern "C" rlk_status rlk_grad_norm(const void* x, int64_t n, int32_t dtype, uint64_t* bins, double* out,
                                    void* stream) {
  if (!bins || !out) return fail(RLK_EINVAL, "bins and out are required");
  if (!aligned(bins, 8) || !aligned(out, 8)) return fail(RLK_EALIGN, "bins and out must be 8-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(bins, 0, NB * sizeof(uint64_t), st) != cudaSuccess)
    return fail(RLK_ECUDA, "clearing the bins: %s", cudaGetErrorString(cudaGetLastError()));
  rlk_status s = rlk_sqnorm_accumulate(x, n, dtype, bins, stream);
  if (s != RLK_OK) return s;
  return rlk_sqnorm_finalize(bins, out, stream);
}
