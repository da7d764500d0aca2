// topk.cu -- the indexer's top-k selection: per query row, the k largest of
// its logits over the request's causal prefix, as request-local positions in
// ascending order (-1 padded), the index list the sparse attention reads.
//
// "[Feat][NVIDIA] DeepSeek-V4.1: Prefill support CP with multistream forward
// prepare (4/N)" (the indexer: mqa_logits scores, topk_v2 selects); the
// selection rule: values ordered by the IEEE total order of non-NaN binary32
// (-0 below +0), ties to the smaller column, a row with at most k candidates
// returning all of them.
//
// HBM-bound: a row of n > k logits is read once (4n bytes) and 4k bytes of
// indices are written.  Persistent CTAs take rows in turn, longest first; a
// bulk L2 prefetch of a CTA's next row is issued as soon as its current row
// has been filtered, so HBM streams while the selection runs on chip.  Per
// row:
//   1. threshold c: extrapolated from the CTA's previous row (its threshold,
//      the candidates that kept and its k-th largest value give the count of
//      the tail as a function of the threshold; the count scales with the
//      row's length), aiming at k + 4 sqrt(k) candidates; or, for a CTA's
//      first row, when the extrapolation reaches too far, or when its count
//      misses, a sample: 256 groups of 8 consecutive logits spread over the
//      row, c its r-th largest, r chosen so that about k + 3 standard
//      deviations of the row are expected at or above it.  Rows of at most C
//      logits skip this (c = -inf).
//   2. filter: one coalesced pass keeps every logit >= c, with its column,
//      as a candidate in shared memory (warp-aggregated appends).
//   3. exact selection over the candidates when there are between k and C of
//      them (then every logit below c ranks below the k-th largest): the k-th
//      largest key tau, how many keys exceed it and how many equal it, from
//      one histogram pass over a bracket around tau's estimate, else from a
//      radix select over the candidates' key range.
//   4. a bitmap over the row's columns marks the keys above tau and, cut in
//      column order, the ties; a scan of its words writes the k columns in
//      ascending order.
// An extrapolated threshold that fails the count (fewer than k or more than C
// logits at or above it) is replaced by the sample's, and the row filtered
// again; when the sample's fails too, steps 3-4 run over the row in global
// memory instead: slower, the same result.
#include <algorithm>
#include <cmath>

#include "cpmla_internal.cuh"

namespace cpmla {
namespace {

constexpr int kTkThreads = 256;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kSample = 2048;     // sampled logits: one group of 8 per thread
// float4 loads per thread in flight in the filter pass: with the lean appends
// three fit the 40 registers of six CTAs per SM (2, 3, 4: 0.981, 0.954, 0.989
// ms on the 32768-row case)
constexpr int kFilterUnroll = 3;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kRankDirect = 64;   // a bin this small is finished by direct ranking
constexpr int kDigitBits = 8;     // radix digit: 256 bins, one per thread in the scan
constexpr int kBins = 1 << kDigitBits;
constexpr int kPrefetchChunk = 32768;
// Six CTAs per SM (the candidate arrays sized k + k/2 + 512): 1.279 ms on the
// 32768-row case against 1.302 with four (2k + 1024, four loads), when the
// filter kept two loads in flight; five were no faster then, nor now (three
// loads: 0.958 against 0.954 ms).
constexpr int kTkMinBlocks = 6;
// A row's threshold is extrapolated from the CTA's previous row when it lies
// within this many times the previous row's (c, tau) span of counts (2, 4, 8,
// 16 spans: 1.121, 1.100, 1.095, 1.095 ms on the 32768-row case; the sampled
// threshold alone 1.279 ms).
constexpr int kExtrapSpans = 8;
// The candidates' kth-largest is first looked for by one histogram pass over
// +-kRangeHalf candidates around its estimate (the row's own count at its
// threshold and the previous row's slope), then the radix select over the
// whole candidate range if it is not there (+-32, 64, 128, 256, 512: 1.068,
// 1.060, 1.055, 1.056, 1.060 ms on the 32768-row case; radix select alone
// 1.069).
constexpr int kRangeHalf = 128;
// An extrapolated threshold aims at k + kTargetSigmas sqrt(k) + 8 candidates
// (2, 3, 4, 5: 1.035, 0.984, 0.955, 0.958 ms on the 32768-row case; below 4
// the misses' second filter passes cost more than the fewer candidates save).
constexpr int kTargetSigmas = 4;

static_assert(kSample == 8 * kTkThreads, "one sample group of 8 logits per thread");
static_assert(kBins == kTkThreads, "one histogram bin per thread when clearing");

// order-preserving image of a binary32 value: unsigned compare of keys is the
// IEEE total order (-0 below +0)
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v);
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// Starts streaming a row's logits into L2 (in-bounds: the row's allocation
// holds its length rounded up to a multiple of 4 floats).
__device__ __forceinline__ void prefetch_row_l2(const float *x, int n) {
  const int64_t bytes = (((int64_t)n * 4) + 15) & ~(int64_t)15;
  for (int64_t off = 0; off < bytes; off += kPrefetchChunk) {
    const int64_t left = bytes - off;
    const uint32_t sz = (uint32_t)(left < kPrefetchChunk ? left : kPrefetchChunk);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                     reinterpret_cast<const char *>(x) + off),
                 "r"(sz)
                 : "memory");
  }
}

struct TkScratch {
  int hist[2][kBins];  // double-buffered: one is cleared while the other is scanned
  int wsum[kTkWarps];
  uint32_t rlo[kTkWarps], rhi[kTkWarps];
  int cnt;       // candidates appended by the filter pass
  int bin, above, in_bin;  // the bin holding the wanted rank, counts above and in it
  int cut;       // last tie column kept
  int total;     // columns marked in the bitmap
  int n_small;   // keys gathered for direct ranking
  uint32_t tau;  // direct ranking result: key, elements above and equal
  int gt, eq;
  uint32_t small[kRankDirect];
};

struct Selection {
  uint32_t tau;  // key of the kth-largest element
  int n_gt;      // elements with key > tau (< kth)
  int n_eq;      // elements with key == tau (n_gt + n_eq >= kth)
};

// A CTA's last filtered row (every thread holds the same copy): the threshold
// c its filter used, the candidates that kept (cnt, of a row of n logits) and
// the row's kth-largest value tau.  c and tau are two points of the row's
// upper tail, from which the next row's threshold is extrapolated.
struct TkPrev {
  float c, tau;
  int cnt, n;
  bool ok;
};

// Inclusive scan of one int per thread over the block.
__device__ __forceinline__ int block_incl_scan(int v, TkScratch &sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) sc.wsum[warp] = v;
  __syncthreads();
  int add = 0;
  for (int w = 0; w < warp; ++w) add += sc.wsum[w];
  __syncthreads();
  return v + add;
}

// Smallest and largest of each thread's (lo, hi) over the block.  One
// barrier: the per-warp slots are written again only by a later call, after
// further barriers.
__device__ __forceinline__ void block_minmax(uint32_t &lo, uint32_t &hi, TkScratch &sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sc.rlo[warp] = lo;
    sc.rhi[warp] = hi;
  }
  __syncthreads();
  lo = sc.rlo[0];
  hi = sc.rhi[0];
  for (int w = 1; w < kTkWarps; ++w) {
    lo = min(lo, sc.rlo[w]);
    hi = max(hi, sc.rhi[w]);
  }
}

// Radix select of the kth-largest key (1 <= kth <= count) among
// key_at(0 .. count-1); (lo, hi) is each thread's smallest and largest of
// the keys (the block's are taken here).  Digits of kDigitBits are taken from
// the top of the keys' range (key - min), so the first histogram already
// spreads over it; warp 0 scans each histogram while the other warps clear
// the next one.  Once the bin holding the wanted rank has at most
// kRankDirect keys they are gathered and ranked against each other.  Called
// by every thread; ends with a barrier.
template <class KeyAt>
__device__ Selection block_select(const KeyAt &key_at, int count, int kth, uint32_t lo,
                                  uint32_t hi, TkScratch &sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  sc.hist[0][tid] = 0;  // kTkThreads == kBins
  sc.hist[1][tid] = 0;
  if (tid == 0) sc.n_small = 0;
  block_minmax(lo, hi, sc);
  const uint32_t kmin = lo, kmax = hi;
  if (kmin == kmax) return {kmax, 0, count};

  int hib = 32 - __clz((int)(kmax - kmin));  // bits hib.. of (key - kmin) are zero
  uint32_t fixed = 0;                          // (key - kmin) >> hib of the wanted element
  int krem = kth, n_gt = 0, in_bin = count;
  for (int pass = 0; in_bin > kRankDirect; ++pass) {
    int *hist = sc.hist[pass & 1];
    const int lob = max(hib - kDigitBits, 0), nb = 1 << (hib - lob);
    for (int i = tid; i < count; i += kTkThreads) {
      const uint32_t u = key_at(i) - kmin;
      const uint32_t high = hib >= 32 ? 0u : (u >> hib);
      if (high == fixed) atomicAdd(&hist[(u >> lob) & (uint32_t)(nb - 1)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // bins from the top, 8 consecutive ones per lane (bins >= nb are 0)
      constexpr int kPer = kBins / 32;
      int h[kPer], sum = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        h[j] = hist[kBins - 1 - kPer * lane - j];
        sum += h[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (incl - sum < krem && krem <= incl) {
        int above = incl - sum;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          if (above < krem && krem <= above + h[j]) {
            sc.bin = kBins - 1 - kPer * lane - j;
            sc.above = above;
            sc.in_bin = h[j];
          }
          above += h[j];
        }
      }
    } else {
      // the other buffer was scanned in the previous pass and is next used
      // after the barrier below
      for (int i = tid - 32; i < kBins; i += kTkThreads - 32) sc.hist[(pass + 1) & 1][i] = 0;
    }
    __syncthreads();
    const int bin = sc.bin, above = sc.above;
    in_bin = sc.in_bin;
    krem -= above;
    n_gt += above;
    fixed = (fixed << (hib - lob)) | (uint32_t)bin;
    hib = lob;
    if (hib == 0) return {kmin + fixed, n_gt, in_bin};  // the bin is one key
  }
  // at most kRankDirect keys left in the bin: gather them and rank each
  // against the others
  for (int i = tid; i < count; i += kTkThreads) {
    const uint32_t key = key_at(i), u = key - kmin;
    const uint32_t high = hib >= 32 ? 0u : (u >> hib);
    if (high == fixed) sc.small[atomicAdd(&sc.n_small, 1)] = key;
  }
  __syncthreads();
  if (tid < in_bin) {
    const uint32_t e = sc.small[tid];
    int gt = 0, eq = 0;
    for (int j = 0; j < in_bin; ++j) {
      const uint32_t o = sc.small[j];
      gt += o > e;
      eq += o == e;
    }
    if (gt < krem && krem <= gt + eq) {  // every holder of the wanted key writes the same
      sc.tau = e;
      sc.gt = gt;
      sc.eq = eq;
    }
  }
  __syncthreads();
  return {sc.tau, n_gt + sc.gt, sc.eq};
}

// The kth-largest of key_at(0 .. count-1) when it lies in [klo, khi]: one
// pass counts the keys above khi and takes a histogram of those inside (the
// range's top kDigitBits bits), warp 0 finds the wanted bin, and that bin's
// keys (at most kRankDirect) are ranked against each other.  Returns false
// (s untouched) when the wanted rank is outside the range or its bin holds
// more keys.  Called by every thread; ends with a barrier.
template <class KeyAt>
__device__ bool range_select(const KeyAt &key_at, int count, int kth, uint32_t klo,
                             uint32_t khi, TkScratch &sc, Selection &s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int *hist = sc.hist[0];
  hist[tid] = 0;  // kTkThreads == kBins
  if (tid == 0) sc.n_small = 0;
  __syncthreads();
  const uint32_t width = khi - klo;
  const int hib = 32 - __clz((int)width);  // (key - klo) >> hib == 0 inside the range
  const int lob = hib > kDigitBits ? hib - kDigitBits : 0;
  int above = 0;
  for (int i = tid; i < count; i += kTkThreads) {
    const uint32_t key = key_at(i);
    if (key > khi)
      ++above;
    else if (key >= klo)
      atomicAdd(&hist[(key - klo) >> lob], 1);
  }
  above = __reduce_add_sync(0xffffffffu, above);
  if (lane == 0) sc.wsum[warp] = above;
  __syncthreads();
  above = 0;
#pragma unroll
  for (int w = 0; w < kTkWarps; ++w) above += sc.wsum[w];
  const int krem = kth - above;
  if (warp == 0) {
    // bins from the top, 8 consecutive ones per lane
    constexpr int kPer = kBins / 32;
    int h[kPer], sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      h[j] = hist[kBins - 1 - kPer * lane - j];
      sum += h[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 0) sc.bin = -1;
    __syncwarp();
    if (krem >= 1 && incl - sum < krem && krem <= incl) {
      int ab = incl - sum;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (ab < krem && krem <= ab + h[j]) {
          sc.bin = kBins - 1 - kPer * lane - j;
          sc.above = ab;
          sc.in_bin = h[j];
        }
        ab += h[j];
      }
    }
  }
  __syncthreads();
  const int bin = sc.bin;
  if (bin < 0 || sc.in_bin > kRankDirect) {
    __syncthreads();  // the scratch is reused by the caller's next step
    return false;
  }
  const int kb = krem - sc.above, in_bin = sc.in_bin, ab_in = sc.above;
  for (int i = tid; i < count; i += kTkThreads) {
    const uint32_t key = key_at(i);
    if (key >= klo && key <= khi && (int)((key - klo) >> lob) == bin)
      sc.small[atomicAdd(&sc.n_small, 1)] = key;
  }
  __syncthreads();
  if (tid < in_bin) {
    const uint32_t e = sc.small[tid];
    int gt = 0, eq = 0;
    for (int j = 0; j < in_bin; ++j) {
      const uint32_t o = sc.small[j];
      gt += o > e;
      eq += o == e;
    }
    if (gt < kb && kb <= gt + eq) {  // every holder of the wanted key writes the same
      sc.tau = e;
      sc.gt = gt;
      sc.eq = eq;
    }
  }
  __syncthreads();
  s = {sc.tau, above + ab_in + sc.gt, sc.eq};
  return true;
}

// Marks the k selected columns of the row in the bitmap bm (zeroed, n bits)
// and writes them in ascending order to orow.  elem(i) -> (key, column) for
// i < count enumerates a set holding every element with key >= s.tau.
template <class Elem>
__device__ void emit_selection(const Elem &elem, int count, const Selection &s, int k, int n,
                               uint32_t *bm, int32_t *orow, TkScratch &sc) {
  const int tid = threadIdx.x;
  const int need = k - s.n_gt;  // ties to keep, 1..s.n_eq
  const int nw = (n + 31) >> 5;
  const int per = (nw + kTkThreads - 1) / kTkThreads;  // contiguous words per thread
  const int w0 = min(tid * per, nw), w1 = min(w0 + per, nw);
  if (s.n_eq > need) {
    // the ties first, cut after the need-th in column order
    for (int i = tid; i < count; i += kTkThreads) {
      uint32_t key;
      int col;
      elem(i, key, col);
      if (key == s.tau) atomicOr(&bm[col >> 5], 1u << (col & 31));
    }
    __syncthreads();
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bm[w]);
    const int incl = block_incl_scan(c, sc);
    if (incl - c < need && need <= incl) {
      int r = need - 1 - (incl - c);  // rank of the last kept tie among this thread's bits
      for (int w = w0; w < w1; ++w) {
        uint32_t m = bm[w];
        const int pc = __popc(m);
        if (r < pc) {
          for (int j = 0; j < r; ++j) m &= m - 1;
          sc.cut = 32 * w + __ffs(m) - 1;
          break;
        }
        r -= pc;
      }
    }
    __syncthreads();
    const int cut = sc.cut;
    for (int w = w0; w < w1; ++w) {
      const int d = cut - 32 * w;  // bits 0..d of word w are kept
      if (d < 0)
        bm[w] = 0u;
      else if (d < 31)
        bm[w] &= (2u << d) - 1u;
    }
    __syncthreads();
    for (int i = tid; i < count; i += kTkThreads) {
      uint32_t key;
      int col;
      elem(i, key, col);
      if (key > s.tau) atomicOr(&bm[col >> 5], 1u << (col & 31));
    }
  } else {
    for (int i = tid; i < count; i += kTkThreads) {
      uint32_t key;
      int col;
      elem(i, key, col);
      if (key >= s.tau) atomicOr(&bm[col >> 5], 1u << (col & 31));
    }
  }
  __syncthreads();
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bm[w]);
  const int incl = block_incl_scan(c, sc);
  if (tid == kTkThreads - 1) sc.total = incl;
  int pos = incl - c;
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bm[w];
    while (m) {
      if (pos < k) orow[pos] = 32 * w + __ffs(m) - 1;
      ++pos;
      m &= m - 1;
    }
  }
  __syncthreads();
  // exactly k columns are marked; the padding only keeps the row defined if
  // NaN logits broke the count
  for (int j = sc.total + tid; j < k; j += kTkThreads) orow[j] = -1;
}

// One row of the selection (every thread of the block).  next_x / next_n: the
// CTA's next row, prefetched into L2 once this row no longer needs the
// filter pass (nullptr: none).
__device__ __forceinline__ void select_row(const float *__restrict__ x, int n, int k, int cap,
                                           int32_t *__restrict__ orow, uint32_t *cand,
                                           uint32_t *bm, TkScratch &sc,
                                           const float *next_x, int next_n, TkPrev &prev) {
  const int tid = threadIdx.x, lane = tid & 31;
  const float4 *x4 = reinterpret_cast<const float4 *>(x);
  const int nw = (n + 31) >> 5;
  for (int w = tid; w < nw; w += kTkThreads) bm[w] = 0u;

  bool try_candidates = cap >= k;
  float c = -INFINITY;
  // 1. the sample: group tid at a float4 boundary, 8 logits, inside the row;
  // c = the sample's r-th largest, r chosen so that about k + 3 standard
  // deviations of the row are expected at or above it
  auto sample_threshold = [&]() -> float {
    const int64_t off = ((int64_t)tid * (n - 8) / (kTkThreads - 1)) & ~(int64_t)3;
    const float4 a = __ldg(x4 + off / 4), b = __ldg(x4 + off / 4 + 1);
    const uint32_t sk[8] = {order_key(a.x), order_key(a.y), order_key(a.z), order_key(a.w),
                            order_key(b.x), order_key(b.y), order_key(b.z), order_key(b.w)};
    uint32_t lo = sk[0], hi = sk[0];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cand[j * kTkThreads + tid] = sk[j];  // (the select ignores the order)
      lo = min(lo, sk[j]);
      hi = max(hi, sk[j]);
    }
    const float p = (float)k / (float)n;
    const float want = (float)kSample * p + 3.f * sqrtf((float)kSample * p * (1.f - p)) + 2.f;
    const int r = min(kSample, max(1, (int)ceilf(want)));
    const Selection s = block_select([&](int i) { return cand[i]; }, kSample, r, lo, hi, sc);
    return key_value(s.tau);
  };
  // 1'. or, cheaper, the threshold extrapolated from the CTA's last row: its
  // count is linear in the threshold between (c, cnt) and (tau, k), and scales
  // with the row's length; aim at k + 4 sqrt(k) candidates.  The filter's
  // count verifies it; a miss takes the sample's threshold and filters again.
  bool predicted = false;
  // the previous row's tail slope (value per candidate), -1 when unknown
  const float slope =
      (prev.ok && prev.cnt > k) ? (prev.tau - prev.c) / (float)(prev.cnt - k) : -1.f;
  if (try_candidates && n > cap) {
    if (prev.ok && prev.cnt > k) {
      const float target = (float)k + (float)kTargetSigmas * sqrtf((float)k) + 8.f;
      const float span = (float)(prev.cnt - k);
      const float extra = target * (float)prev.n / (float)n - (float)prev.cnt;
      if (fabsf(extra) <= (float)kExtrapSpans * span) {
        c = prev.c - (prev.tau - prev.c) / span * extra;
        predicted = true;
      }
    }
    if (!predicted) {
      if (n >= kSample)
        c = sample_threshold();
      else
        try_candidates = false;
    }
    prev.ok = false;  // set again by a row that passes the check below
  }

  for (int attempt = 0; try_candidates && attempt < 2; ++attempt) {
    // 2. the filter pass
    if (tid == 0) sc.cnt = 0;
    __syncthreads();
    const int nv = (n + 3) >> 2;
    for (int base = 0; base < nv; base += kTkThreads * kFilterUnroll) {
      float4 v[kFilterUnroll];
      const bool whole = 4 * (base + kTkThreads * kFilterUnroll) <= n;
      {
        // logits past the row's end read as NaN, which no threshold passes,
        // so the tests below need no bounds checks (0.982 ms against 0.997
        // with a check on each element)
        const float nan = __int_as_float(0x7fc00000);
#pragma unroll
        for (int u = 0; u < kFilterUnroll; ++u) {
          const int vi = base + u * kTkThreads + tid;
          v[u] = vi < nv ? __ldcs(x4 + vi) : make_float4(nan, nan, nan, nan);
        }
        if (!whole) {
#pragma unroll
          for (int u = 0; u < kFilterUnroll; ++u) {
            const int j = 4 * (base + u * kTkThreads + tid);
            if (j + 1 >= n) v[u].y = nan;
            if (j + 2 >= n) v[u].z = nan;
            if (j + 3 >= n) v[u].w = nan;
          }
        }
      }
      // this thread's candidates
      int q = 0;
#pragma unroll
      for (int u = 0; u < kFilterUnroll; ++u)
        q += (int)(v[u].x >= c) + (int)(v[u].y >= c) + (int)(v[u].z >= c) + (int)(v[u].w >= c);
      const int total = __reduce_add_sync(0xffffffffu, q);
      int wbase = 0;
      if (lane == 0 && total) wbase = atomicAdd(&sc.cnt, total);
      int p = __shfl_sync(0xffffffffu, wbase, 0);
      // one ballot per (load, component): the warp's candidates of a slot go to
      // consecutive entries (lane order), one shared-memory append per warp;
      // a warp whose candidates would pass the buffer's end appends none (the
      // row then fails the count check below)
      if (total && p + total <= cap) {
        uint32_t lt;
        asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
#pragma unroll
        for (int u = 0; u < kFilterUnroll; ++u) {
          const int j = 4 * (base + u * kTkThreads + tid);
          const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const bool pass = e[t] >= c;
            const uint32_t bal = __ballot_sync(0xffffffffu, pass);
            if (pass) {
              const uint32_t key = order_key(e[t]);
              const int at = p + __popc(bal & lt);
              *reinterpret_cast<uint2 *>(cand + 2 * at) = make_uint2(key, (uint32_t)(j + t));
            }
            p += __popc(bal);
          }
        }
      }
    }
    __syncthreads();
    const int cnt = sc.cnt;
    // every logit below c ranks below every candidate, so with at least k
    // candidates the row's top k are among them
    if (cnt >= k && cnt <= cap) {
      if (tid == 0 && next_x) prefetch_row_l2(next_x, next_n);
      // 3.-4. exact selection over the candidates
      Selection s;
      bool found = false;
      if (slope >= 0.f) {
        // tau's estimate: the row's own count at c, the previous row's slope
        const float t_hat = c + slope * (float)(cnt - k);
        const float d = slope * (float)kRangeHalf;
        found = range_select([&](int i) { return cand[2 * i]; }, cnt, k, order_key(t_hat - d),
                             order_key(t_hat + d), sc, s);
      }
      if (!found) {
        // the candidates' key range, for the radix select (taken here rather
        // than in every append of the filter: 0.997 ms against 1.057 on the
        // 32768-row case, with the capacity checked once per warp slot)
        uint32_t lo = 0xFFFFFFFFu, hi = 0u;
        for (int i = tid; i < cnt; i += kTkThreads) {
          lo = min(lo, cand[2 * i]);
          hi = max(hi, cand[2 * i]);
        }
        s = block_select([&](int i) { return cand[2 * i]; }, cnt, k, lo, hi, sc);
      }
      emit_selection(
          [&](int i, uint32_t &key, int &col) {
            const uint2 kc = *reinterpret_cast<const uint2 *>(cand + 2 * i);
            key = kc.x;
            col = (int)kc.y;
          },
          cnt, s, k, n, bm, orow, sc);
      if (n > cap) prev = {c, key_value(s.tau), cnt, n, true};
      return;
    }
    if (!predicted) break;
    // the extrapolated threshold missed: the sample's, and a second pass
    predicted = false;
    if (n >= kSample)
      c = sample_threshold();
    else
      break;
  }
  // the same exact selection over the whole row in global memory
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = tid; i < n; i += kTkThreads) {
    const uint32_t key = order_key(__ldg(x + i));
    lo = min(lo, key);
    hi = max(hi, key);
  }
  const Selection s =
      block_select([&](int i) { return order_key(__ldg(x + i)); }, n, k, lo, hi, sc);
  if (tid == 0 && next_x) prefetch_row_l2(next_x, next_n);
  emit_selection(
      [&](int i, uint32_t &key, int &col) {
        key = order_key(__ldg(x + i));
        col = i;
      },
      n, s, k, n, bm, orow, sc);
}

__global__ void __launch_bounds__(kTkThreads, kTkMinBlocks)
    topk_select_kernel(const float *__restrict__ logits, int64_t stride, int n_rows,
                       const int32_t *__restrict__ row_len, int max_len, int k, int cap,
                       int32_t *__restrict__ out, int *status) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  __shared__ TkScratch sc;
  // candidates as (key, column) pairs, cap of them (a row's filter appends one
  // 8-byte store per candidate: 1.068 ms on the 32768-row case against 1.093
  // with separate key and column arrays); the sample's kSample keys use the
  // same words
  uint32_t *cand = reinterpret_cast<uint32_t *>(tk_smem);
  uint32_t *bm = cand + max(cap, kSample) + cap;  // ceil(max_len / 32) words
  const int tid = threadIdx.x;

  // a row's length, -1 for none; out-of-range lengths are recorded and read as 0
  auto length_of = [&](int i) -> int {
    if (i >= n_rows) return -1;
    const int n = row_len[n_rows - 1 - i];
    if (n < 0 || n > max_len) {
      if (tid == 0) record_status(status, CPMLA_ERR_INDEX);
      return 0;
    }
    return n;
  };
  // rows in reverse (long causal rows sit at the end), in turn over the CTAs
  int i = blockIdx.x;
  int n = length_of(i);
  TkPrev prev{0.f, 0.f, 0, 0, false};
  if (tid == 0 && n > k) prefetch_row_l2(logits + (int64_t)(n_rows - 1 - i) * stride, n);
  for (; i < n_rows; i += gridDim.x) {
    const int row = n_rows - 1 - i;
    int32_t *orow = out + (int64_t)row * k;
    const int i_next = i + gridDim.x;
    const int n_next = length_of(i_next);
    if (n <= k) {
      for (int j = tid; j < k; j += kTkThreads) orow[j] = j < n ? j : -1;
    } else {
      const float *next_x =
          n_next > k ? logits + (int64_t)(n_rows - 1 - i_next) * stride : nullptr;
      select_row(logits + (int64_t)row * stride, n, k, cap, orow, cand, bm, sc, next_x,
                 n_next, prev);
    }
    if (n <= k && n_next > k && tid == 0)
      prefetch_row_l2(logits + (int64_t)(n_rows - 1 - i_next) * stride, n_next);
    n = n_next;
    __syncthreads();  // shared memory is reused by the next row
  }
}

}  // namespace
}  // namespace cpmla

extern "C" int mla_topk_select(const float *logits, int64_t logits_row_stride, int n_rows,
                               const int32_t *row_len, int max_row_len, int k,
                               int32_t *topk_idx, void *stream) {
  using namespace cpmla;
  const char *fn = "mla_topk_select";
  CPMLA_CHECK_ARG(n_rows >= 0, "%s: n_rows=%d < 0", fn, n_rows);
  CPMLA_CHECK_ARG(k >= 1 && k <= CPMLA_TOPK_MAX, "%s: k=%d outside 1..%d", fn, k, CPMLA_TOPK_MAX);
  CPMLA_CHECK_ARG(max_row_len >= 0 && max_row_len <= CPMLA_TOPK_MAX_ROW,
                  "%s: max_row_len=%d outside 0..%d", fn, max_row_len, CPMLA_TOPK_MAX_ROW);
  CPMLA_CHECK_ARG(logits_row_stride >= max_row_len && logits_row_stride % 4 == 0,
                  "%s: logits_row_stride=%lld must be >= max_row_len and a multiple of 4", fn,
                  (long long)logits_row_stride);
  if (n_rows == 0) return CPMLA_OK;
  CPMLA_CHECK_ARG(row_len && topk_idx, "%s: row_len and topk_idx are required", fn);
  CPMLA_CHECK_ARG(max_row_len <= k || (logits && ((uintptr_t)logits & 15) == 0),
                  "%s: logits must be non-NULL and 16-byte aligned", fn);
  int *status = status_word();
  if (!status) return fail(CPMLA_ERR_CUDA, "%s: status word unavailable", fn);

  // candidate capacity: room for the expected k + a few standard deviations
  const int64_t bm_bytes = 4 * (((int64_t)max_row_len + 31) / 32);
  // (at least the sample's size, so that every row too short to sample is
  // taken whole)
  int64_t cap = std::min<int64_t>(std::max<int64_t>((int64_t)k + k / 2 + 512, kSample),
                                  (kSmemBudget - bm_bytes) / 8);
  if (cap < kSample)  // the key array still holds the sample
    cap = std::max<int64_t>(0, std::min<int64_t>(cap, (kSmemBudget - bm_bytes - 4 * kSample) / 4));
  const size_t smem = 4 * (size_t)std::max<int64_t>(cap, kSample) + 4 * (size_t)cap + (size_t)bm_bytes;
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "mla_topk_select: shared memory attribute");
  // persistent CTAs: as many as fit on the device at once
  int dev = 0, n_sm = 0, per_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_select_kernel, kTkThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "mla_topk_select: occupancy");
  const int64_t grid = std::min<int64_t>(n_rows, (int64_t)std::max(1, n_sm * per_sm));
  topk_select_kernel<<<(unsigned)grid, kTkThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      logits, logits_row_stride, n_rows, row_len, max_row_len, k, (int)cap, topk_idx, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "mla_topk_select: launch");
  return CPMLA_OK;
}
