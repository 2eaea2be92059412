// cambi.cu — CAMBI c-values and top-K pooling on the device (ss2_cambi_* in
// include/ss2.h).
//
// Source: "ADR-1357: Run the SYCL CAMBI extractor entirely on the device"
// (vmafx documentation), Decision: per-pixel window counts of 10-bit levels
// (window^2 < 4226, so at most 65 x 65) kept as commuting modular uint16
// histogram updates, the value w p0 pm / (p0 + pm) formed as (float)(w p0
// pm) times the reciprocal, and top-K pooling by a three-pass radix select
// over the IEEE bit patterns with the exact sum in units of 2^-24.
// Readings where the page is silent (as the oracle takes them): centred
// windows clipped to the plane, an optional mask, a table of up to four
// (d, w) pairs with the largest term taken, the reciprocal 1/n rounded to
// nearest (a table of 1.0f / n built by the host's IEEE division), the pool
// the mean of the exact sum.
//
//   k_cambi_present  the levels that occur in each plane (1024-bit maps).
//   k_cambi_cvalues  one warp per 32 columns of a plane; lane = column.  Each
//                    step the warp stages the leaving and entering row
//                    segments in shared memory (fetched one step ahead).  A
//                    window's count is split in two: the columns that all
//                    four lanes of a lane group share go to the group's
//                    core histogram (16-bit bins, two to a 32-bit word,
//                    shared-memory atomics, the columns dealt out among the
//                    four lanes); the three columns left to each lane go to
//                    its own histogram (8-bit bins interleaved by lane so
//                    each lane owns its elements, plain loads and stores).
//                    A column whose leaving and entering pixels agree is
//                    skipped.  At 65 x 65 a pixel costs about 37 bin
//                    updates instead of 130.  Planes with at most 256
//                    distinct levels (8-bit video as 10-bit levels) index
//                    bins by the level's rank among those present (a 2 KB
//                    table per warp): 12 KB of bins per warp instead of
//                    48 KB.
//   k_cambi_hist     radix histogram of one 11/11/10-bit digit of the values
//                    that match the digits chosen so far.
//   k_cambi_select   one block per plane: the digit holding the k-th largest
//                    value and the rank left inside it.
//   k_cambi_sum      the values above the threshold, exact, in 2^-24 units
//                    (a value is below 2^14, so below 2^38 units; a block's
//                    sum fits 64 bits).
//   k_cambi_final    per plane: block sums in index order into 128 bits,
//                    plus rank * threshold; the mean.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/ss2.h"
#include "ss2_host.h"

#define SS2_API extern "C" __attribute__((visibility("default")))

namespace {

using namespace ss2;

constexpr int kLevels = 1024;
constexpr int kMaxWin2 = 4225;
constexpr int kGroup = 4;                          // lanes sharing a core histogram
constexpr int kGroups = 32 / kGroup;
constexpr int kOwnMax = kGroup - 1;                // columns a lane counts alone (at most)
// per warp: 32 lanes' own 16-bit bins, then the groups' core bins (16-bit,
// two to a 32-bit word)
constexpr int cv_smem(int bins) { return bins * 32 * 1 + kGroups * bins * 2; }
constexpr int kCvSmem = cv_smem(1024);             // 48 KB
constexpr int kCvSmemCompact = cv_smem(256);       // 12 KB: the compact histograms
constexpr int kMaxCount = 2 * kMaxWin2;            // p0 + pm <= 8450: the reciprocal table's range
constexpr int kErrLevel = 2;                       // a level >= 1024 was seen
constexpr int kErrValue = 4;                       // a value off the 2^-24 grid or >= 2^14
constexpr int kSumThreads = 256;
constexpr int kSumPerBlock = 16384;                // values per sum block (fits 64-bit sums)

struct CGeom {
  int w, h, window, ndiff;
  int diffs[4], weights[4];
  long long plane;          // w * h
  int sum_blocks;           // per plane
};

constexpr int kSeg = 32 + 64;                      // a row's window columns for 32 lanes
constexpr unsigned kSkip = 0xFFFFu;                // outside the plane or not counted
constexpr int kCompactBins = 256;                  // the compact histogram's bins

// Which of the 1024 levels occur in each plane (a 1024-bit map per plane,
// levels >= 1024 ignored: the c-value kernel reports them).
__global__ void __launch_bounds__(256)
    k_cambi_present(CGeom g, const uint16_t *__restrict__ levels, unsigned *__restrict__ present) {
  __shared__ unsigned bits[kLevels / 32];
  const int t = threadIdx.x;
  if (t < kLevels / 32) bits[t] = 0u;
  __syncthreads();
  const uint16_t *L = levels + (long long)blockIdx.y * g.plane;
  for (long long i = (long long)blockIdx.x * blockDim.x + t; i < g.plane;
       i += (long long)gridDim.x * blockDim.x) {
    const unsigned v = __ldg(L + i);
    if (v < kLevels) atomicOr(&bits[v >> 5], 1u << (v & 31));
  }
  __syncthreads();
  if (t < kLevels / 32 && bits[t]) atomicOr(&present[blockIdx.y * (kLevels / 32) + t], bits[t]);
}

// k_cambi_cvalues<BINS>: one warp per 32 output columns of a plane; lane =
// column.  Lane l's window covers segment columns l .. l + 2r.  The four
// lanes of group q (lanes 4q .. 4q+3) all cover columns 4q+3 .. 4q+2r: the
// group's core, counted once in a histogram of BINS 16-bit bins packed two
// to a 32-bit word, which the group's lanes update with 32-bit shared-memory
// atomics (+-1 or +-2^16), each taking every fourth core column.  The steps'
// updates commute and every final count lies in 0..4030, so the packed word
// holds both counts exactly once a step's updates are all in, whatever the
// borrows and carries between the halves along the way.  The rest of a
// lane's window (2-j columns on the left and j on the right for lane 4q+j,
// three in all) goes to the lane's own histogram of BINS 8-bit bins
// (element bin * 32 + lane, plain loads and stores; a count stays in
// 0..195).  A window narrower than a group has no core: each lane counts
// its whole window (at most 3 x 3 pixels) alone.  A count is the core bin
// plus the own bin.  Groups of four rather than eight cost more core
// updates per pixel (2 x 62 / 4 against 2 x 58 / 8) but let the own bins
// be 8-bit: 14.7 KB of shared memory per warp instead of 20.7 KB, 14
// resident warps per SM instead of 10, and the kernel waits on its step
// chains more than it issues.  With BINS = 256 a level is replaced by its
// rank among the levels present in the plane (8-bit video as 10-bit levels
// has at most 256); planes with more levels run the BINS = 1024 variant,
// which uses the levels themselves.  Both variants are launched; a block
// whose plane belongs to the other one returns at once.  Each step the warp
// stages the leaving and entering row segments in shared memory (fetched
// one step ahead); a column whose two pixels agree is skipped.
template <int BINS>
__global__ void __launch_bounds__(32)
    k_cambi_cvalues(CGeom g, const uint16_t *__restrict__ levels, const uint8_t *__restrict__ mask,
                    const unsigned *__restrict__ present, const float *__restrict__ recip,
                    float *__restrict__ out, int *__restrict__ err) {
  extern __shared__ __align__(16) uint8_t cv_hist[];   // own 8-bit bins (BINS x 32 lanes), then the cores
  __shared__ uint16_t seg[2][kSeg];
  __shared__ unsigned pbits[kLevels / 32];         // levels present in the plane
  __shared__ unsigned prank[kLevels / 32];         // present levels below each word
  __shared__ uint16_t rank_of[BINS == kLevels ? 1 : kLevels];   // compact bin of each level
  const int lane = threadIdx.x;
  const unsigned *pp = present + blockIdx.y * (kLevels / 32);
  {
    const unsigned b = pp[lane];
    unsigned r = __popc(b);
    // exclusive prefix of the popcounts over the 32 words, in lane order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned u = __shfl_up_sync(0xffffffffu, r, o);
      if (lane >= o) r += u;
    }
    pbits[lane] = b;
    prank[lane] = r - __popc(b);
    const unsigned total = __shfl_sync(0xffffffffu, r, 31);
    if ((BINS == kCompactBins) != (total <= (unsigned)kCompactBins)) return;   // the other variant's
  }
  __syncwarp();
  if (BINS != kLevels) {
    for (int v = lane; v < kLevels; v += 32) {
      const unsigned w = pbits[v >> 5], m = 1u << (v & 31);
      rank_of[v] = (uint16_t)((w & m) ? prank[v >> 5] + __popc(w & (m - 1u)) : kSkip);
    }
    __syncwarp();
  }
  // histogram index of level v (v < 1024): its rank among the present
  // levels (BINS = 256) or v itself; kSkip when v does not occur
  auto bin = [&](unsigned v) -> unsigned {
    if (BINS == kLevels) return v;
    return rank_of[v];
  };
  const int x0 = blockIdx.x * 32, x = x0 + lane;
  const long long base = (long long)blockIdx.y * g.plane;
  const uint16_t *L = levels + base;
  const uint8_t *M = mask ? mask + base : nullptr;
  unsigned *cores = reinterpret_cast<unsigned *>(cv_hist + BINS * 32);
  for (int i = lane; i < BINS * 8; i += 32) reinterpret_cast<unsigned *>(cv_hist)[i] = 0u;
  for (int i = lane; i < kGroups * BINS / 2; i += 32) cores[i] = 0u;
  const int r = g.window / 2;
  const int nseg = 32 + 2 * r;
  const bool col = x < g.w;
  bool bad = false;
  // the lane's group, its core columns [ca, cz] and the lane's own columns:
  // own column t is lane + t for t < nleft, then cz + 1 + (t - nleft)
  const int jl = lane % kGroup;
  unsigned *core = cores + (lane / kGroup) * (BINS / 2);
  // the core count of bin b: half b & 1 of word b >> 1
  auto core_count = [&](unsigned b) -> unsigned { return (core[b >> 1] >> ((b & 1u) * 16)) & 0xFFFFu; };
  const bool has_core = g.window >= kGroup;           // the same for every lane
  const int ca = lane - jl + kGroup - 1, cz = lane - jl + 2 * r;
  const int nown = has_core ? kGroup - 1 : 2 * r + 1;
  const int nleft = has_core ? kGroup - 1 - jl : 2 * r + 1;
  const int ncore = has_core ? (cz - ca) / kGroup + 1 : 0;   // the first lane's count
  auto fetch = [&](int yy, unsigned (&v)[3]) {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int i = lane + 32 * j, xx = x0 - r + i;
      v[j] = kSkip;
      if (i < nseg && yy >= 0 && yy < g.h && xx >= 0 && xx < g.w) {
        const long long at = (long long)yy * g.w + xx;
        if (!M || __ldg(M + at)) {
          const unsigned lv = __ldg(L + at);
          if (lv >= kLevels) bad = true;        // skipped; the call reports -EINVAL
          else v[j] = bin(lv);
        }
      }
    }
  };
  auto put = [&](int s_, const unsigned (&v)[3]) {
#pragma unroll
    for (int j = 0; j < 3; ++j)
      if (lane + 32 * j < kSeg) seg[s_][lane + 32 * j] = (uint16_t)v[j];
  };
  // remove seg[0] and add seg[1] over the lane's own columns (indices read
  // before the updates) and the lane's share of its group's core columns
  auto apply = [&](bool remove) {
    unsigned a[kOwnMax], b[kOwnMax];
#pragma unroll
    for (int t = 0; t < kOwnMax; ++t) {
      const int i = t < nleft ? lane + t : cz + 1 + (t - nleft);
      a[t] = (remove && t < nown) ? seg[0][i] : kSkip;
      b[t] = t < nown ? seg[1][i] : kSkip;
    }
#pragma unroll
    for (int t = 0; t < kOwnMax; ++t) {
      if (a[t] == b[t]) continue;                   // the column's count does not change
      // a != b: two different bins, both read before either is written
      const unsigned ca_ = a[t] != kSkip ? cv_hist[a[t] * 32 + lane] : 0u;
      const unsigned cb_ = b[t] != kSkip ? cv_hist[b[t] * 32 + lane] : 0u;
      if (a[t] != kSkip) cv_hist[a[t] * 32 + lane] = (uint8_t)(ca_ - 1u);
      if (b[t] != kSkip) cv_hist[b[t] * 32 + lane] = (uint8_t)(cb_ + 1u);
    }
    for (int t = 0; t < ncore; ++t) {
      const int i = ca + jl + t * kGroup;
      if (i > cz) break;
      const unsigned av = remove ? seg[0][i] : kSkip, bv = seg[1][i];
      if (av == bv) continue;
      // commuting +-1 on a packed bin: both halves are exact once the
      // step's updates are all in
      if (av != kSkip) atomicAdd(&core[av >> 1], 0u - (1u << ((av & 1u) * 16)));
      if (bv != kSkip) atomicAdd(&core[bv >> 1], 1u << ((bv & 1u) * 16));
    }
  };
  __syncwarp();
  // the first window: rows 0 .. r added
  for (int yy = 0; yy <= min(r, g.h - 1); ++yy) {
    unsigned v[3];
    fetch(yy, v);
    put(1, v);
    __syncwarp();
    apply(false);                                   // every lane: the cores are shared
    __syncwarp();
  }
  // step y moves the window from rows y-1-r .. y-1+r to y-r .. y+r; the
  // rows of step y + 1 are fetched while step y is applied
  unsigned nout[3], nin[3];
  fetch(-r, nout);                                  // step 1: leaving row -r, entering row 1 + r
  fetch(1 + r, nin);
  for (int y = 0; y < g.h; ++y) {
    if (y > 0) {
      put(0, nout);
      put(1, nin);
      __syncwarp();
      fetch(y - r, nout);                           // rows of step y + 1
      fetch(y + 1 + r, nin);
      apply(true);
      __syncwarp();                                 // the cores are complete
    }
    if (col) {
      const long long at = (long long)y * g.w + x;
      float best = 0.0f;
      if (!M || __ldg(M + at)) {
        const unsigned lv = __ldg(L + at);
        if (lv >= kLevels) {
          bad = true;
        } else {
          const unsigned b0 = bin(lv);               // the pixel's own level occurs
          const unsigned p0 = cv_hist[b0 * 32 + lane] + (has_core ? core_count(b0) : 0u);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i >= g.ndiff || lv + g.diffs[i] >= kLevels) continue;
            const unsigned bm = bin(lv + g.diffs[i]);
            if (bm == kSkip) continue;
            const unsigned pm = cv_hist[bm * 32 + lane] + (has_core ? core_count(bm) : 0u);
            if (pm == 0u) continue;
            const float c = __fmul_rn((float)((unsigned)g.weights[i] * p0 * pm),
                                      __ldg(recip + p0 + pm));
            best = fmaxf(best, c);
          }
        }
      }
      out[base + at] = best;
    }
    __syncwarp();                                   // seg is rewritten next step
  }
  if (bad) atomicOr(err, kErrLevel);
}

// Radix state per plane: prefix bits chosen so far, their mask, the rank k
// still to find inside them.
struct RState {
  unsigned prefix, mask;
  long long k;
};

// radix digits of a value's 32 bits, most significant first: 11, 11, 10
__host__ __device__ constexpr int digit_bits(int pass) { return pass < 2 ? 11 : 10; }
__host__ __device__ constexpr int digit_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }

// A value the exact sum can take: +0, or finite, below 2^14 and a multiple
// of 2^-24 (every fp32 in [0.5, 2^14) is; below 0.5 the low significand bits
// must be zero).
__device__ __forceinline__ bool on_grid(unsigned b) {
  if (b == 0u) return true;
  if (b >= 0x46800000u) return false;                 // >= 2^14, inf, NaN or negative
  if (b >= 0x3F000000u) return true;                  // [0.5, 2^14)
  const unsigned e = b >> 23;
  const unsigned m = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  const int drop = 126 - (int)(e ? e : 1u);           // bits below 2^-24
  return drop <= 23 && (m & ((1u << drop) - 1u)) == 0u;
}

__global__ void k_cambi_init(RState *__restrict__ st, long long k) {
  st[threadIdx.x] = RState{0u, 0u, k};
}

__global__ void __launch_bounds__(256)
    k_cambi_hist(CGeom g, const float *__restrict__ c, const RState *__restrict__ st, int pass,
                 unsigned *__restrict__ hist, int *__restrict__ err) {
  __shared__ unsigned h[2048];
  const int plane = blockIdx.y;
  const int nb = 1 << digit_bits(pass), sh = digit_shift(pass);
  for (int i = threadIdx.x; i < nb; i += blockDim.x) h[i] = 0u;
  __syncthreads();
  const RState s = st[plane];
  const unsigned *v = reinterpret_cast<const unsigned *>(c + (long long)plane * g.plane);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < g.plane;
       i += (long long)gridDim.x * blockDim.x) {
    const unsigned b = __ldg(v + i);
    if (pass == 0 && !on_grid(b)) atomicOr(err, kErrValue);
    if ((b & s.mask) == s.prefix) atomicAdd(&h[(b >> sh) & (nb - 1)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nb; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[(long long)plane * 2048 + i], h[i]);
}

// One block of 1024 threads per plane: suffix counts over the digit's bins
// (largest bin first) locate the bin holding the k-th largest value.
__global__ void __launch_bounds__(1024)
    k_cambi_select(RState *__restrict__ st, int pass, unsigned *__restrict__ hist) {
  __shared__ unsigned long long suf[2048];
  const int plane = blockIdx.x, t = threadIdx.x;
  const int nb = 1 << digit_bits(pass), sh = digit_shift(pass);
  unsigned *hp = hist + (long long)plane * 2048;
  // suf[i] = sum of bins i .. nb-1, by a block scan over reversed order
  for (int i = t; i < nb; i += 1024) suf[i] = hp[i];
  __syncthreads();
  for (int off = 1; off < nb; off <<= 1) {
    unsigned long long a[2] = {0, 0};
    for (int j = 0; j < 2; ++j) {
      const int i = t + 1024 * j;
      if (i < nb) a[j] = suf[i] + (i + off < nb ? suf[i + off] : 0ull);
    }
    __syncthreads();
    for (int j = 0; j < 2; ++j) {
      const int i = t + 1024 * j;
      if (i < nb) suf[i] = a[j];
    }
    __syncthreads();
  }
  const long long k = st[plane].k;
  for (int j = 0; j < 2; ++j) {
    const int i = t + 1024 * j;
    if (i < nb) {
      const unsigned long long above = i + 1 < nb ? suf[i + 1] : 0ull;
      if ((long long)above < k && k <= (long long)suf[i]) {   // exactly one bin matches
        RState s = st[plane];
        s.prefix |= (unsigned)i << sh;
        s.mask |= (unsigned)(nb - 1) << sh;
        s.k = k - (long long)above;
        st[plane] = s;
      }
    }
  }
  __syncthreads();
  for (int i = t; i < nb; i += 1024) hp[i] = 0u;     // ready for the next pass
}

__global__ void __launch_bounds__(kSumThreads)
    k_cambi_sum(CGeom g, const float *__restrict__ c, const RState *__restrict__ st,
                unsigned long long *__restrict__ part) {
  __shared__ unsigned long long red[kSumThreads];
  const int plane = blockIdx.y, t = threadIdx.x;
  const unsigned T = st[plane].prefix;              // the threshold's bits
  const unsigned *v = reinterpret_cast<const unsigned *>(c + (long long)plane * g.plane);
  const long long i0 = (long long)blockIdx.x * kSumPerBlock;
  const long long i1 = min((long long)g.plane, i0 + kSumPerBlock);
  unsigned long long s = 0;
  for (long long i = i0 + t; i < i1; i += kSumThreads) {
    const unsigned b = __ldg(v + i);
    if (b > T) {   // non-negative floats order as their bit patterns
      const float f = __uint_as_float(b);
      s += (unsigned long long)__float2ull_rn(__fmul_rn(f, 16777216.0f));   // exact: on the 2^-24 grid
    }
  }
  red[t] = s;
  __syncthreads();
  for (int o = kSumThreads / 2; o > 0; o >>= 1) {
    if (t < o) red[t] += red[t + o];
    __syncthreads();
  }
  if (t == 0) part[(long long)plane * g.sum_blocks + blockIdx.x] = red[0];
}

__global__ void k_cambi_final(CGeom g, const RState *__restrict__ st,
                              const unsigned long long *__restrict__ part, long long k,
                              unsigned long long *__restrict__ sums, float *__restrict__ thr,
                              double *__restrict__ means) {
  const int plane = blockIdx.x;
  if (threadIdx.x != 0) return;
  unsigned long long lo = 0, hi = 0;
  for (int b = 0; b < g.sum_blocks; ++b) {
    const unsigned long long a = part[(long long)plane * g.sum_blocks + b];
    lo += a;
    hi += lo < a ? 1ull : 0ull;
  }
  const RState s = st[plane];
  const float T = __uint_as_float(s.prefix);
  const unsigned long long tu = __float2ull_rn(__fmul_rn(T, 16777216.0f));
  // + rank * T units: rank <= 2^31, T units < 2^38 -> the product < 2^69
  const unsigned long long r = (unsigned long long)s.k;
  const unsigned long long p_lo = r * tu, p_hi = __umul64hi(r, tu);
  lo += p_lo;
  hi += p_hi + (lo < p_lo ? 1ull : 0ull);
  sums[2 * plane] = lo;
  sums[2 * plane + 1] = hi;
  thr[plane] = T;
  means[plane] = ((double)hi * 18446744073709551616.0 + (double)lo) / 16777216.0 / (double)k;
}

}  // namespace

struct ss2_cambi {
  CGeom g;
  int batch, device;
  float *d_c = nullptr;                     // c-values of a batch (pool-only calls use the caller's)
  RState *d_st = nullptr;
  unsigned *d_hist = nullptr;
  unsigned long long *d_part = nullptr, *d_sums = nullptr;
  float *d_thr = nullptr;
  double *d_means = nullptr;
  int *d_err = nullptr, *h_err = nullptr;
  unsigned *d_present = nullptr;            // levels present, a 1024-bit map per plane
  float *d_recip = nullptr;                 // 1.0f / n for n = 0 .. kMaxCount (entry 0 unused)
  unsigned long long *h_sums = nullptr;
  float *h_thr = nullptr;
  double *h_means = nullptr;
  size_t h_cap = 0;
  KernelTimer timer;                         // per-kernel event timing
};

static void cambi_free(ss2_cambi *c) {
  if (!c) return;
  cudaFree(c->d_c);
  cudaFree(c->d_st);
  cudaFree(c->d_hist);
  cudaFree(c->d_part);
  cudaFree(c->d_sums);
  cudaFree(c->d_thr);
  cudaFree(c->d_means);
  cudaFree(c->d_err);
  cudaFree(c->d_present);
  cudaFree(c->d_recip);
  if (c->h_err) cudaFreeHost(c->h_err);
  if (c->h_sums) cudaFreeHost(c->h_sums);
  if (c->h_thr) cudaFreeHost(c->h_thr);
  if (c->h_means) cudaFreeHost(c->h_means);
  delete c;
}

SS2_API ss2_cambi *ss2_cambi_create(int width, int height, int window, int ndiff,
                                    const int *diffs, const int *weights, int max_batch) {
  if (width < 1 || height < 1 || width > SS2_MAX_DIM || height > SS2_MAX_DIM) {
    fail(SS2_EINVAL, "plane %dx%d is outside 1..%d", width, height, SS2_MAX_DIM);
    return nullptr;
  }
  if (window < 1 || !(window & 1) || window * window > kMaxWin2) {
    fail(SS2_EINVAL, "cambi: window %d must be odd with window^2 <= %d", window, kMaxWin2);
    return nullptr;
  }
  if (ndiff < 1 || ndiff > 4 || !diffs || !weights) {
    fail(SS2_EINVAL, "cambi: 1 to 4 (diff, weight) pairs");
    return nullptr;
  }
  CGeom g;
  std::memset(&g, 0, sizeof(g));
  for (int i = 0; i < ndiff; ++i) {
    if (diffs[i] < 1 || diffs[i] >= kLevels || weights[i] < 1 || weights[i] > 9) {
      fail(SS2_EINVAL, "cambi: diff %d must be 1..1023 and weight %d 1..9", diffs[i], weights[i]);
      return nullptr;
    }
    g.diffs[i] = diffs[i];
    g.weights[i] = weights[i];
  }
  if (max_batch < 0 || max_batch > 1024) {
    fail(SS2_EINVAL, "batch %d is outside 0..1024", max_batch);
    return nullptr;
  }
  g.w = width; g.h = height; g.window = window; g.ndiff = ndiff;
  g.plane = (long long)width * height;
  g.sum_blocks = (int)((g.plane + kSumPerBlock - 1) / kSumPerBlock);
  int dev = 0;
  if (check_device(&dev)) return nullptr;
  ss2_cambi *c = new (std::nothrow) ss2_cambi();
  if (!c) {
    fail(SS2_ENOMEM, "host allocation failed");
    return nullptr;
  }
  c->g = g;
  c->device = dev;
  // default: as many planes as 2 GB of c-values hold, 1 to 64
  c->batch = max_batch ? max_batch
                       : (int)std::max<long long>(1, std::min<long long>(64, (2LL << 30) / (g.plane * 4)));
  const size_t B = (size_t)c->batch;
  if (cudaFuncSetAttribute(k_cambi_cvalues<kLevels>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kCvSmem) != cudaSuccess ||
      cudaMalloc(&c->d_present, B * (kLevels / 32) * sizeof(unsigned)) != cudaSuccess ||
      cudaMalloc(&c->d_recip, (kMaxCount + 1) * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&c->d_c, B * g.plane * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&c->d_st, B * sizeof(RState)) != cudaSuccess ||
      cudaMalloc(&c->d_hist, B * 2048 * sizeof(unsigned)) != cudaSuccess ||
      cudaMalloc(&c->d_part, B * g.sum_blocks * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMalloc(&c->d_sums, B * 2 * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMalloc(&c->d_thr, B * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&c->d_means, B * sizeof(double)) != cudaSuccess ||
      cudaMalloc(&c->d_err, sizeof(int)) != cudaSuccess ||
      cudaMallocHost(&c->h_err, sizeof(int)) != cudaSuccess ||
      cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess ||
      cudaMemset(c->d_hist, 0, B * 2048 * sizeof(unsigned)) != cudaSuccess) {
    cudaGetLastError();
    fail(SS2_ENOMEM, "cambi workspace allocation failed");
    cambi_free(c);
    return nullptr;
  }
  *c->h_err = 0;
  {
    // the reciprocal table: IEEE single division on the host rounds to
    // nearest, so entry n is 1/n correctly rounded
    std::vector<float> r(kMaxCount + 1, 0.0f);
    for (int n = 1; n <= kMaxCount; ++n) r[n] = 1.0f / (float)n;
    // the copy and the memsets above are ordered on the legacy stream only
    // (a pageable copy may still be in flight when cudaMemcpy returns):
    // wait for them before any call on a non-blocking stream
    if (cudaMemcpy(c->d_recip, r.data(), r.size() * sizeof(float), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      fail(SS2_EIO, "cambi reciprocal table upload failed");
      cambi_free(c);
      return nullptr;
    }
  }
  return c;
}

SS2_API void ss2_cambi_destroy(ss2_cambi *ctx) { cambi_free(ctx); }

SS2_API int ss2_cambi_profile_begin(ss2_cambi *ctx) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  ctx->timer.begin();
  return 0;
}

SS2_API int ss2_cambi_profile_end(ss2_cambi *ctx, double *ms, int *launches) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  const cudaError_t e = ctx->timer.finish(2, ms, launches);
  return e == cudaSuccess ? 0 : cuda_fail(e, "cambi profile events");
}

static cudaError_t cambi_cv_launch(ss2_cambi *c, const uint16_t *levels, const uint8_t *mask,
                                   float *out, int nb, cudaStream_t st) {
  const CGeom &g = c->g;
  cudaError_t e = c->timer.mark(0, true, st);
  if (e != cudaSuccess) return e;
  // which levels occur, then both histogram variants (each block keeps or
  // leaves its plane by the count of levels present)
  e = cudaMemsetAsync(c->d_present, 0, (size_t)nb * (kLevels / 32) * sizeof(unsigned), st);
  if (e == cudaSuccess) {
    const int pblocks = std::max(1, std::min(64, (int)((g.plane + 8191) / 8192)));
    k_cambi_present<<<dim3(pblocks, nb), 256, 0, st>>>(g, levels, c->d_present);
    e = cudaGetLastError();
  }
  const dim3 grid((g.w + 31) / 32, nb);
  if (e == cudaSuccess) {
    k_cambi_cvalues<kCompactBins><<<grid, 32, kCvSmemCompact, st>>>(
        g, levels, mask, c->d_present, c->d_recip, out, c->d_err);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    k_cambi_cvalues<kLevels><<<grid, 32, kCvSmem, st>>>(g, levels, mask, c->d_present,
                                                       c->d_recip, out, c->d_err);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = c->timer.mark(0, false, st);
  return e;
}

static cudaError_t cambi_pool_launch(ss2_cambi *c, const float *cv, int nb, long long k,
                                     cudaStream_t st) {
  const CGeom &g = c->g;
  cudaError_t e = c->timer.mark(1, true, st);
  if (e == cudaSuccess) {
    k_cambi_init<<<1, nb, 0, st>>>(c->d_st, k);
    e = cudaGetLastError();
  }
  const int hblocks = std::max(1, std::min(256, (int)((g.plane + 4095) / 4096)));
  for (int pass = 0; pass < 3 && e == cudaSuccess; ++pass) {
    k_cambi_hist<<<dim3(hblocks, nb), 256, 0, st>>>(g, cv, c->d_st, pass, c->d_hist, c->d_err);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
      k_cambi_select<<<nb, 1024, 0, st>>>(c->d_st, pass, c->d_hist);
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess) {
    k_cambi_sum<<<dim3(g.sum_blocks, nb), kSumThreads, 0, st>>>(g, cv, c->d_st, c->d_part);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    k_cambi_final<<<nb, 32, 0, st>>>(g, c->d_st, c->d_part, k, c->d_sums, c->d_thr, c->d_means);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = c->timer.mark(1, false, st);
  return e;
}

static int cambi_grow(ss2_cambi *c, int n) {
  if ((size_t)n <= c->h_cap) return 0;
  if (c->h_sums) cudaFreeHost(c->h_sums);
  if (c->h_thr) cudaFreeHost(c->h_thr);
  if (c->h_means) cudaFreeHost(c->h_means);
  c->h_sums = nullptr;
  c->h_thr = nullptr;
  c->h_means = nullptr;
  c->h_cap = 0;
  if (cudaMallocHost(&c->h_sums, (size_t)n * 2 * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMallocHost(&c->h_thr, (size_t)n * sizeof(float)) != cudaSuccess ||
      cudaMallocHost(&c->h_means, (size_t)n * sizeof(double)) != cudaSuccess) {
    cudaGetLastError();
    return fail(SS2_ENOMEM, "pinned allocation failed");
  }
  c->h_cap = (size_t)n;
  return 0;
}

static int cambi_finish(ss2_cambi *c, cudaStream_t st) {
  cudaError_t e = cudaMemcpyAsync(c->h_err, c->d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (*c->h_err) {
    const int bits = *c->h_err;
    *c->h_err = 0;
    cudaMemsetAsync(c->d_err, 0, sizeof(int), st);
    cudaStreamSynchronize(st);
    if (bits & kErrLevel) return fail(SS2_EINVAL, "cambi: a level is 1024 or more");
    if (bits & kErrValue)
      return fail(SS2_EINVAL, "cambi: a c-value is negative, not finite, 2^14 or more, or off "
                              "the 2^-24 grid");
    return fail(SS2_EIO, "cambi: kernel error bits %#x", bits);
  }
  return 0;
}

// Copies the pooled results of nb planes to the caller's arrays at plane f0.
static cudaError_t cambi_readback(ss2_cambi *c, int f0, int nb, cudaStream_t st) {
  cudaError_t e = cudaMemcpyAsync(c->h_sums + 2 * (size_t)f0, c->d_sums,
                                  (size_t)nb * 2 * sizeof(unsigned long long),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->h_thr + f0, c->d_thr, nb * sizeof(float), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->h_means + f0, c->d_means, nb * sizeof(double), cudaMemcpyDeviceToHost,
                        st);
  return e;
}

static void cambi_copy_out(ss2_cambi *c, int n, uint64_t *sums, float *thr, double *means) {
  if (sums) std::memcpy(sums, c->h_sums, (size_t)n * 2 * sizeof(uint64_t));
  if (thr) std::memcpy(thr, c->h_thr, (size_t)n * sizeof(float));
  if (means) std::memcpy(means, c->h_means, (size_t)n * sizeof(double));
}

SS2_API int ss2_cambi_cvalues(ss2_cambi *ctx, const uint16_t *levels, const uint8_t *mask,
                              int n_planes, float *cvalues, void *stream) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  if (n_planes < 0) return fail(SS2_EINVAL, "negative plane count %d", n_planes);
  if (n_planes == 0) return 0;
  if (!levels || !cvalues) return fail(SS2_EINVAL, "NULL pointer");
  cudaStream_t st = (cudaStream_t)stream;
  const long long P = ctx->g.plane;
  for (int f0 = 0; f0 < n_planes; f0 += ctx->batch) {
    const int nb = std::min(ctx->batch, n_planes - f0);
    cudaError_t e = cambi_cv_launch(ctx, levels + f0 * P, mask ? mask + f0 * P : nullptr,
                                    cvalues + f0 * P, nb, st);
    if (e != cudaSuccess) return cuda_fail(e, "cambi c-values launch");
  }
  return cambi_finish(ctx, st);
}

SS2_API int ss2_cambi_topk(ss2_cambi *ctx, const float *cvalues, int n_planes, long long k,
                           uint64_t *sums, float *thresholds, double *means, void *stream) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  if (n_planes < 0) return fail(SS2_EINVAL, "negative plane count %d", n_planes);
  if (n_planes == 0) return 0;
  if (!cvalues) return fail(SS2_EINVAL, "NULL pointer");
  if (k < 1 || k > ctx->g.plane) return fail(SS2_EINVAL, "k %lld is outside 1..%lld", k, ctx->g.plane);
  if (int rc = cambi_grow(ctx, n_planes)) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const long long P = ctx->g.plane;
  for (int f0 = 0; f0 < n_planes; f0 += ctx->batch) {
    const int nb = std::min(ctx->batch, n_planes - f0);
    cudaError_t e = cambi_pool_launch(ctx, cvalues + f0 * P, nb, k, st);
    if (e == cudaSuccess) e = cambi_readback(ctx, f0, nb, st);
    if (e != cudaSuccess) return cuda_fail(e, "cambi top-k launch");
  }
  if (int rc = cambi_finish(ctx, st)) return rc;
  cambi_copy_out(ctx, n_planes, sums, thresholds, means);
  return 0;
}

SS2_API int ss2_cambi_pool(ss2_cambi *ctx, const uint16_t *levels, const uint8_t *mask,
                           int n_planes, long long k, uint64_t *sums, float *thresholds,
                           double *means, void *stream) {
  if (!ctx) return fail(SS2_EINVAL, "NULL context");
  if (n_planes < 0) return fail(SS2_EINVAL, "negative plane count %d", n_planes);
  if (n_planes == 0) return 0;
  if (!levels) return fail(SS2_EINVAL, "NULL pointer");
  if (k < 1 || k > ctx->g.plane) return fail(SS2_EINVAL, "k %lld is outside 1..%lld", k, ctx->g.plane);
  if (int rc = cambi_grow(ctx, n_planes)) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const long long P = ctx->g.plane;
  for (int f0 = 0; f0 < n_planes; f0 += ctx->batch) {
    const int nb = std::min(ctx->batch, n_planes - f0);
    cudaError_t e = cambi_cv_launch(ctx, levels + f0 * P, mask ? mask + f0 * P : nullptr,
                                    ctx->d_c, nb, st);
    if (e == cudaSuccess) e = cambi_pool_launch(ctx, ctx->d_c, nb, k, st);
    if (e == cudaSuccess) e = cambi_readback(ctx, f0, nb, st);
    if (e != cudaSuccess) return cuda_fail(e, "cambi launch");
  }
  if (int rc = cambi_finish(ctx, st)) return rc;
  cambi_copy_out(ctx, n_planes, sums, thresholds, means);
  return 0;
}
