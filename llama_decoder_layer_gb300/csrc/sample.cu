// Sampling beyond greedy: temperature, top-k, top-p, an inverse-CDF draw at a
// caller-supplied uniform, and the raw logprob of the sampled token.
//
//   greedy (temperature < 1e-5): token = argmax of the raw logits (lowest index)
//   otherwise, with w_i = exp((l_i - max l) / T):
//     top-k keeps every token whose logit is >= the k-th largest (ties kept),
//     top-p keeps, inside that set, every token whose w_i >= tau, tau the
//       largest value whose kept mass reaches p times the top-k mass (ties kept),
//     the token is the first kept one, in index order, at which the running
//       kept mass exceeds u times the total kept mass
//   logprob = l_token - log(sum_j exp(l_j))   (the unscaled logits)
//
// A row is split over a thread-block cluster of up to 8 CTAs.  Thresholds are
// found on the logits' order-preserving 32-bit keys (dividing by T > 0 keeps
// the order).  Masses are 64-bit fixed point (w_i * 2^40, w_i in (0, 1]), so
// every histogram, sum and scan is exact integer arithmetic: the result does
// not depend on the order of the atomic adds, and the same call always returns
// the same tokens.
//
// Rows without truncation (top-k off, top-p >= 1): after the first pass, each
// warp sums the weights of a contiguous segment of its CTA's slice, the cluster
// exchanges its CTAs' sums, and the warp whose segment holds the draw finds
// the token with 32-wide scans.  Top-p without top-k: a radix descent on mass
// (histograms summed over the cluster) gives the threshold, then the same
// draw over the keys above it.
//
// Top-k rows with k <= 1024 (the fast path): one pass gives the row maximum,
// its index, the log-normaliser (an online sum) and a histogram of the keys'
// top 12 bits; the cluster sums its CTAs' histograms through distributed
// shared memory.  Once the keys at or above the bin holding the k-th largest
// number at most 1024, one more pass gathers them (else the next 12 and 8
// bits refine the bin first), and the k-th largest key, the top-p threshold
// and the inverse-CDF draw are taken exactly over those candidates.  Other
// rows (k > 1024, or more than 1024 keys tied at the k-th value) take the
// general path in the cluster's first CTA: a radix select on counts for top-k
// and a radix descent on mass for top-p over the whole row.
//
// Sources: [LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B", Sampler
// (sample(): greedy rows take the argmax; temperature scaling; the top-k /
// top-p sampler; greedy results merged below a temperature threshold;
// gather_logprobs of the sampled token from the raw logprobs).
#include <float.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace llama {

namespace {

constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;
constexpr float kGreedyTemperature = 1e-5f;
constexpr float kFixedScale = 1099511627776.0f;  // 2^40

// monotone map of a float to an unsigned key (larger float -> larger key,
// equal floats -> equal keys: -0 is taken as +0, as float comparison does)
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// w = exp((l - lmax) * inv_t) in [0, 1], as fixed point with 40 fraction bits
__device__ __forceinline__ unsigned long long fixed_weight(float l, float lmax, float inv_t) {
  return __float2ull_rz(expf((l - lmax) * inv_t) * kFixedScale);
}

template <class T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// block sums in a fixed order (lanes, then warps): deterministic for floats too
__device__ __forceinline__ float block_sum_f(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < kSampWarps ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;  // every warp holds the total
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  unsigned long long t = lane < kSampWarps ? red[lane] : 0ull;
  return warp_sum(t);
}

// exclusive prefix sum over the threads of the block (thread order)
__device__ __forceinline__ unsigned long long block_exclusive_scan_u64(unsigned long long v, unsigned long long* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  __syncthreads();
  if (lane == 31) red[w] = inc;
  __syncthreads();
  if (w == 0) {
    unsigned long long x = lane < kSampWarps ? red[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += t;
    }
    red[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  return (w > 0 ? red[w - 1] : 0ull) + inc - v;
}

constexpr int kBinsMax = 4096;  // 12-bit digits

constexpr int kCandMax = 1024;  // candidates of the fast path (one per thread)
constexpr int kMaxCluster = 8;  // CTAs per row

struct Cand {
  int idx;
  float logit;
};

// hist doubles as the fast path's storage: 4096 uint32 counts in its first
// half and this CTA's candidate list (up to 2048) in its second half; after
// the last histogram the first CTA assembles the cluster's candidates (index,
// key, weight) in the first half.
struct SampleShared {
  unsigned long long hist[kBinsMax];
  unsigned long long red_u[kSampWarps];
  float red_f[kSampWarps];
  float best_v[kSampWarps];
  int best_i[kSampWarps];
  uint32_t red_k[kSampWarps];
  uint32_t digit;
  unsigned long long acc;
  unsigned long long bin_count;
  unsigned long long need;
  int token;
  // this CTA's pass-one partials, read by the cluster: max, its index, and the
  // online log-sum (m, s) with sum_i exp(x_i - m) = s
  float part_best, part_m, part_s;
  int part_bi;
  int cand_n;
  // the cluster's merged values
  float lmax, log_z;
  int amax;
  // rows without truncation: the mass of each warp's segment and of this CTA
  unsigned long long warp_mass[kSampWarps];
  unsigned long long part_mass;
  unsigned long long target;  // the draw, as a mass offset inside this CTA's slice
  int owner;                  // 1 when the draw falls in this CTA's slice
};

// Every pass over a row goes through for_row: each thread loads kUnroll
// elements (stride kSampThreads) before it uses any of them, so a thread keeps
// that many L2 requests in flight (one CTA per row is all the parallelism a
// 34-row head gives).
constexpr int kUnroll = 8;

template <class F>
__device__ __forceinline__ void for_range(const float* __restrict__ row, int i0, int i1, F&& f) {
  for (int base = i0 + static_cast<int>(threadIdx.x); base < i1; base += kSampThreads * kUnroll) {
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kSampThreads;
      x[u] = i < i1 ? __ldg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kSampThreads;
      if (i < i1) f(i, x[u]);
    }
  }
}

template <class F>
__device__ __forceinline__ void for_row(const float* __restrict__ row, int V, F&& f) {
  for_range(row, 0, V, f);
}

// Largest key t with S(key >= t) >= need, where S counts the tokens (MASS
// false) or sums their fixed-point weights (MASS true), by digits of 12, 12
// and 8 bits from the top.  The first digit holds the sign, the exponent and
// three mantissa bits, so the logits of a row spread over many bins (an 8-bit
// first digit put nearly all of them in two or three, and the shared-memory
// atomics on those bins serialised).  The bin where the running sum from the
// top reaches `need` is found by a block-wide scan.  Keys below floor_key are
// left out: the answer is known to be >= floor_key, and S(key >= t) for
// t >= floor_key does not depend on them.
template <bool MASS>
__device__ uint32_t threshold_key(const float* row, int V, float lmax, float inv_t, unsigned long long need,
                                  uint32_t floor_key, SampleShared& sh) {
  uint32_t prefix = 0, mask = 0;
  unsigned long long above = 0;  // S of the keys above the current prefix range
#pragma unroll 1
  for (int level = 0; level < 3; ++level) {
    const int bits = level < 2 ? 12 : 8;
    const int shift = level == 0 ? 20 : (level == 1 ? 8 : 0);
    const int nb = 1 << bits;
    for (int i = threadIdx.x; i < nb; i += kSampThreads) sh.hist[i] = 0;
    __syncthreads();
    for_row(row, V, [&](int, float l) {
      const uint32_t key = order_key(l);
      if (key >= floor_key && (key & mask) == prefix)
        atomicAdd(&sh.hist[(key >> shift) & static_cast<uint32_t>(nb - 1)], MASS ? fixed_weight(l, lmax, inv_t) : 1ull);
    });
    __syncthreads();
    // thread t owns the bins j = nb-1-t*per .. nb-1-(t+1)*per+1 (descending)
    const int per = nb >= kSampThreads ? nb / kSampThreads : 1;
    const int j0 = threadIdx.x * per;
    unsigned long long local = 0;
    if (j0 < nb)
      for (int q = 0; q < per; ++q) local += sh.hist[nb - 1 - (j0 + q)];
    const unsigned long long excl = above + block_exclusive_scan_u64(local, sh.red_u);
    if (j0 < nb && excl < need && need <= excl + local) {
      unsigned long long run = excl;
      for (int q = 0; q < per; ++q) {
        const int bin = nb - 1 - (j0 + q);
        if (run + sh.hist[bin] >= need) {
          sh.digit = static_cast<uint32_t>(bin);
          sh.acc = run;
          break;
        }
        run += sh.hist[bin];
      }
    }
    __syncthreads();
    above = sh.acc;
    prefix |= sh.digit << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
  }
  return prefix;
}

__device__ __forceinline__ unsigned long long kept_mass(const float* row, int V, float lmax, float inv_t,
                                                        uint32_t t_key, SampleShared& sh) {
  unsigned long long m = 0;
  for_row(row, V, [&](int, float l) {
    if (order_key(l) >= t_key) m += fixed_weight(l, lmax, inv_t);
  });
  return block_sum_u64(m, sh.red_u);
}

// (m, s) <- (m, s) + (m2, s2) for online log-sums: sum exp(x - m) = s
__device__ __forceinline__ void lse_add(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * expf(m - m2) + s2;  // m = -inf: s is 0
    m = m2;
  } else if (m2 > -INFINITY) {
    s += s2 * expf(m2 - m);
  }
}

__device__ __forceinline__ void best_add(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  return __reduce_max_sync(0xffffffffu, lane < kSampWarps ? red[lane] : 0u);
}

__device__ __forceinline__ uint32_t ld_cluster_val(uint32_t addr, uint32_t rank, uint32_t) {
  return ld_cluster_u32(mapa_shared(addr, rank));
}

__device__ __forceinline__ unsigned long long ld_cluster_val(uint32_t addr, uint32_t rank, unsigned long long) {
  const uint2 v = ld_cluster_u32x2(mapa_shared(addr, rank));
  return (static_cast<unsigned long long>(v.y) << 32) | v.x;
}

// The bin of `bits` bits where the sum of the histogram (counts of keys, or
// their fixed-point masses) from the top reaches `need`, over the cluster's
// summed histograms; `above` is the sum above the current prefix range.  With
// p_frac >= 0 the need is max(1, floor(p_frac * total)) of this histogram's
// total (left in sh.need).  Sets sh.digit, sh.acc (the sum above the bin) and
// sh.bin_count (the bin's own sum).
template <class T>
__device__ void select_bin(const T* hist, int bits, unsigned long long above, unsigned long long need, uint32_t C,
                           SampleShared& sh, float p_frac = -1.f) {
  const int nb = 1 << bits;
  const int per = nb >= kSampThreads ? nb / kSampThreads : 1;
  const int j0 = threadIdx.x * per;
  unsigned long long mine[kBinsMax / kSampThreads];
  unsigned long long local = 0;
  const uint32_t base = smem_u32(hist);
  // a bin's remote loads (one per CTA) are all issued before they are summed
#pragma unroll
  for (int q = 0; q < kBinsMax / kSampThreads; ++q) {
    T v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      v[r] = q < per && j0 < nb && r < static_cast<int>(C)
                 ? ld_cluster_val(base + static_cast<uint32_t>(sizeof(T)) * (nb - 1 - (j0 + q)),
                                  static_cast<uint32_t>(r), T{})
                 : T{};
    unsigned long long c = 0;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) c += v[r];
    mine[q] = c;
    local += c;
  }
  if (p_frac >= 0.f) {
    const unsigned long long total = block_sum_u64(local, sh.red_u);
    const double pc = p_frac > 0.f ? static_cast<double>(p_frac) : 0.0;
    need = static_cast<unsigned long long>(pc * static_cast<double>(total));
    if (need < 1) need = 1;  // at least one unit: the threshold is the key of a token with weight
    if (threadIdx.x == 0) sh.need = need;
  }
  const unsigned long long excl = above + block_exclusive_scan_u64(local, sh.red_u);
  if (j0 < nb && excl < need && need <= excl + local) {
    unsigned long long run = excl;
#pragma unroll
    for (int q = 0; q < kBinsMax / kSampThreads; ++q) {
      if (q >= per) break;
      if (run + mine[q] >= need) {
        sh.digit = static_cast<uint32_t>(nb - 1 - (j0 + q));
        sh.acc = run;
        sh.bin_count = mine[q];
        break;
      }
      run += mine[q];
    }
  }
  __syncthreads();
}

// The inverse-CDF draw over the keys >= t_key of the whole row, on the
// cluster: every warp sums the weights of a contiguous segment of its CTA's
// slice (so rank, warp and lane order is index order), the CTAs exchange their
// sums, and the warp whose segment holds the draw finds the token with
// 32-wide scans and writes the outputs.  Every CTA of the cluster calls it.
__device__ void draw_segmented(const float* row, int s0, int s1, float lmax, float inv_t, uint32_t t_key, float u_in,
                               uint32_t C, uint32_t rank, float log_z, int32_t* out_token, float* out_logprob,
                               SampleShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (s1 - s0 + kSampWarps - 1) / kSampWarps;
  const int w0 = min(s1, s0 + warp * seg), w1 = min(s1, w0 + seg);
  auto weight = [&](float x) { return order_key(x) >= t_key ? fixed_weight(x, lmax, inv_t) : 0ull; };
  unsigned long long wm = 0;
  for (int i0 = w0; i0 < w1; i0 += 32 * kUnroll) {
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * 32 + lane;
      x[u] = i < w1 ? __ldg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i0 + u * 32 + lane < w1) wm += weight(x[u]);
  }
  wm = warp_sum(wm);
  if (lane == 0) sh.warp_mass[warp] = wm;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0;
    for (int w = 0; w < kSampWarps; ++w) m += sh.warp_mass[w];
    sh.part_mass = m;
  }
  cluster_sync();  // every CTA's mass is complete
  if (warp == 0) {  // lane r reads CTA r's mass
    unsigned long long m = 0;
    if (lane < static_cast<int>(C))
      m = ld_cluster_val(smem_u32(&sh.part_mass), static_cast<uint32_t>(lane), 0ull);
    unsigned long long incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
    const unsigned long long excl = __shfl_sync(0xffffffffu, incl - m, static_cast<int>(rank));
    const unsigned long long mine = __shfl_sync(0xffffffffu, m, static_cast<int>(rank));
    const float u = u_in > 0.f ? (u_in < 1.f ? u_in : 0.99999994f) : 0.f;
    const unsigned long long target =
        static_cast<unsigned long long>(static_cast<double>(u) * static_cast<double>(total));
    if (lane == 0) {
      sh.owner = excl <= target && target < excl + mine ? 1 : 0;
      sh.target = target - excl;
    }
  }
  __syncthreads();
  cluster_sync();  // the cluster has read every CTA's mass
  if (!sh.owner) return;
  const unsigned long long tgt = sh.target;
  unsigned long long wex = 0;
  for (int w = 0; w < warp; ++w) wex += sh.warp_mass[w];
  if (!(wex <= tgt && tgt < wex + sh.warp_mass[warp])) return;
  unsigned long long acc = wex;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const unsigned long long wi = i < w1 ? weight(row[i]) : 0ull;
    unsigned long long incl = wi;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned int hit = __ballot_sync(0xffffffffu, acc + incl > tgt);
    if (hit != 0u) {
      if (lane == __ffs(hit) - 1) {
        *out_token = i;
        if (out_logprob != nullptr) *out_logprob = row[i] - log_z;
      }
      return;
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// The general path over the whole row, by one CTA: top-k threshold key (0 for
// none), top-p by a radix descent on mass above it, and the inverse-CDF draw in
// index order.  Returns the token.
__device__ int sample_general(const float* row, int V, float lmax, float inv_t, int k, float p, float u_in,
                              int amax, SampleShared& sh) {
  uint32_t t_key = 0;  // keep everything
  if (k > 0 && k < V) t_key = threshold_key<false>(row, V, lmax, inv_t, static_cast<unsigned long long>(k), 0u, sh);
  if (p < 1.f) {
    const unsigned long long mass_k = kept_mass(row, V, lmax, inv_t, t_key, sh);
    const double pc = p > 0.f ? static_cast<double>(p) : 0.0;
    // at least one unit, so the threshold is the key of a token that has
    // weight (p -> 0 keeps the maximum and its ties)
    unsigned long long target = static_cast<unsigned long long>(pc * static_cast<double>(mass_k));
    if (target < 1) target = 1;
    const uint32_t t_p = threshold_key<true>(row, V, lmax, inv_t, target, t_key, sh);
    if (t_p > t_key) t_key = t_p;
  }
  const unsigned long long total = kept_mass(row, V, lmax, inv_t, t_key, sh);
  const float u = u_in > 0.f ? (u_in < 1.f ? u_in : 0.99999994f) : 0.f;
  const unsigned long long target = static_cast<unsigned long long>(static_cast<double>(u) *
                                                                    static_cast<double>(total));
  // inverse CDF in index order: contiguous chunks per thread, block scan
  const int chunk = (V + kSampThreads - 1) / kSampThreads;
  const int c0 = threadIdx.x * chunk;
  const int c1 = min(V, c0 + chunk);
  unsigned long long cm = 0;
  for (int i = c0; i < c1; ++i) {
    const float l = row[i];
    if (order_key(l) >= t_key) cm += fixed_weight(l, lmax, inv_t);
  }
  if (threadIdx.x == 0) sh.token = amax;
  const unsigned long long excl = block_exclusive_scan_u64(cm, sh.red_u);
  if (cm > 0 && excl <= target && target < excl + cm) {
    unsigned long long acc = excl;
    for (int i = c0; i < c1; ++i) {
      const float l = row[i];
      if (order_key(l) < t_key) continue;
      acc += fixed_weight(l, lmax, inv_t);
      if (acc > target) {
        sh.token = i;
        break;
      }
    }
  }
  __syncthreads();
  return sh.token;
}

// The fast path's selection over n <= kCandMax candidates that include every
// key >= the row's k-th largest (thread j owns candidate j): the exact top-k
// threshold, top-p above it, and the inverse-CDF draw in index order.
__device__ int sample_candidates(const int* idx_s, const uint32_t* key_s, const unsigned long long* w_s, int n, int k,
                                 float p, float u_in, int amax, SampleShared& sh) {
  const int j = threadIdx.x;
  const bool mine = j < n;
  const uint32_t kj = mine ? key_s[j] : 0u;
  const unsigned long long wj = mine ? w_s[j] : 0ull;
  // the k-th largest key: the largest key with at least k keys >= it
  int ge = 0;
  if (mine)
    for (int i = 0; i < n; ++i) ge += key_s[i] >= kj;
  uint32_t t_key = block_max_u32(mine && ge >= k ? kj : 0u, sh.red_k);
  bool kept = mine && kj >= t_key;
  if (p < 1.f) {
    const unsigned long long mass_k = block_sum_u64(kept ? wj : 0ull, sh.red_u);
    const double pc = p > 0.f ? static_cast<double>(p) : 0.0;
    unsigned long long target = static_cast<unsigned long long>(pc * static_cast<double>(mass_k));
    if (target < 1) target = 1;
    // the largest kept key whose mass of kept keys >= it reaches the target
    unsigned long long s_ge = 0;
    if (kept)
      for (int i = 0; i < n; ++i)
        if (key_s[i] >= kj && key_s[i] >= t_key) s_ge += w_s[i];
    const uint32_t t_p = block_max_u32(kept && s_ge >= target ? kj : 0u, sh.red_k);
    if (t_p > t_key) t_key = t_p;
    kept = mine && kj >= t_key;
  }
  const unsigned long long total = block_sum_u64(kept ? wj : 0ull, sh.red_u);
  const float u = u_in > 0.f ? (u_in < 1.f ? u_in : 0.99999994f) : 0.f;
  const unsigned long long target = static_cast<unsigned long long>(static_cast<double>(u) *
                                                                    static_cast<double>(total));
  if (threadIdx.x == 0) sh.token = amax;
  __syncthreads();
  if (kept && wj > 0) {  // inclusive running mass in index order
    const int ij = idx_s[j];
    unsigned long long run = 0;
    for (int i = 0; i < n; ++i)
      if (key_s[i] >= t_key && idx_s[i] <= ij) run += w_s[i];
    if (run > target && run - wj <= target) sh.token = ij;
  }
  __syncthreads();
  return sh.token;
}

__global__ void __launch_bounds__(kSampThreads, 1) k_sample(const float* __restrict__ logits, int V,
                                                          const float* __restrict__ temperature,
                                                          const int32_t* __restrict__ top_k,
                                                          const float* __restrict__ top_p,
                                                          const float* __restrict__ uniform,
                                                          int32_t* __restrict__ out_tokens,
                                                          float* __restrict__ out_logprobs) {
  __shared__ SampleShared sh;
  pdl_wait();
  const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
  const int b = blockIdx.x / static_cast<int>(C);
  const float* row = logits + static_cast<size_t>(b) * V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_cta = (V + static_cast<int>(C) - 1) / static_cast<int>(C);
  const int s0 = min(V, static_cast<int>(rank) * per_cta), s1 = min(V, s0 + per_cta);

  const float t = temperature[b];
  const bool greedy = !(t >= kGreedyTemperature);  // (a NaN temperature samples greedily)
  const int k = top_k[b];
  const float p = top_p[b];
  const bool fast = !greedy && k > 0 && k < V && k <= kCandMax;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(sh.hist);
  Cand* cand = reinterpret_cast<Cand*>(sh.hist + kBinsMax / 2);
  if (fast)
    for (int i = threadIdx.x; i < kBinsMax; i += kSampThreads) cnt[i] = 0;
  if (threadIdx.x == 0) sh.cand_n = 0;
  __syncthreads();

  // pass one over this CTA's slice: maximum (lowest index), online log-sum,
  // and the histogram of the keys' top 12 bits
  float best = -FLT_MAX, m = -INFINITY, se = 0.f;
  int bi = 0x7fffffff;
  for_range(row, s0, s1, [&](int i, float x) {  // i increases within a thread: strict > keeps the lowest
    if (x > best) {
      best = x;
      bi = i;
    }
    if (x > m) {
      se = se * expf(m - x) + 1.f;
      m = x;
    } else if (x > -INFINITY) {
      se += expf(x - m);
    }
    if (fast) atomicAdd(&cnt[order_key(x) >> 20], 1u);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    best_add(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
    lse_add(m, se, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, se, o));
  }
  if (lane == 0) {
    sh.best_v[warp] = best;
    sh.best_i[warp] = bi;
    sh.red_f[warp] = m;
    sh.red_u[warp] = __float_as_uint(se);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv = -FLT_MAX, mm = -INFINITY, ss = 0.f;
    int bj = 0x7fffffff;
    for (int w = 0; w < kSampWarps; ++w) {
      best_add(bv, bj, sh.best_v[w], sh.best_i[w]);
      lse_add(mm, ss, sh.red_f[w], __uint_as_float(static_cast<uint32_t>(sh.red_u[w])));
    }
    sh.part_best = bv;
    sh.part_bi = bj;
    sh.part_m = mm;
    sh.part_s = ss;
  }
  cluster_sync();  // every CTA's partials and histogram are complete
  if (warp == 0) {  // lane r reads CTA r's partials; a fixed shuffle tree merges them
    float bv = -FLT_MAX, mm = -INFINITY, ss = 0.f;
    int bj = 0x7fffffff;
    if (lane < static_cast<int>(C)) {
      const uint32_t r = static_cast<uint32_t>(lane);
      bv = __uint_as_float(ld_cluster_u32(mapa_shared(smem_u32(&sh.part_best), r)));
      bj = static_cast<int>(ld_cluster_u32(mapa_shared(smem_u32(&sh.part_bi), r)));
      mm = __uint_as_float(ld_cluster_u32(mapa_shared(smem_u32(&sh.part_m), r)));
      ss = __uint_as_float(ld_cluster_u32(mapa_shared(smem_u32(&sh.part_s), r)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      best_add(bv, bj, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bj, o));
      lse_add(mm, ss, __shfl_xor_sync(0xffffffffu, mm, o), __shfl_xor_sync(0xffffffffu, ss, o));
    }
    if (lane == 0) {
      sh.lmax = bv;
      sh.amax = bj == 0x7fffffff ? 0 : bj;
      sh.log_z = mm + logf(ss);
    }
  }
  if (fast) select_bin(cnt, 12, 0ull, static_cast<unsigned long long>(k), C, sh);
  __syncthreads();
  cluster_sync();  // the cluster has read every CTA's pass-one results
  const float lmax = sh.lmax;
  const int amax = sh.amax;
  const float log_z = sh.log_z;

  int token = amax;
  const bool topk_on = k > 0 && k < V;
  // no truncation (top-k off or >= V, top-p >= 1): the draw over the whole row
  const bool full = !greedy && !topk_on && !(p < 1.f);
  // top-p alone: a radix descent on mass over the cluster, then the draw
  const bool topp = !greedy && !topk_on && p < 1.f;
  bool general = !greedy && !fast && !full && !topp;
  if (full) {
    draw_segmented(row, s0, s1, lmax, 1.f / t, 0u, uniform[b], C, rank, log_z, out_tokens + b,
                   out_logprobs != nullptr ? out_logprobs + b : nullptr, sh);
    return;
  }
  if (topp) {
    // tau = the largest key whose mass of keys >= it reaches max(1, p * the
    // row's mass), by 12, 12 and 8 bits of the key, the CTAs' mass histograms
    // summed through distributed shared memory
    const float inv_t = 1.f / t;
    unsigned long long* mh = sh.hist;
    uint32_t prefix = 0, mask = 0;
    unsigned long long above = 0, need = 0;
#pragma unroll 1
    for (int level = 0; level < 3; ++level) {
      const int bits = level < 2 ? 12 : 8;
      const int shift = level == 0 ? 20 : (level == 1 ? 8 : 0);
      const uint32_t nbm = (1u << bits) - 1u;
      for (int i = threadIdx.x; i < kBinsMax; i += kSampThreads) mh[i] = 0;
      __syncthreads();
      for_range(row, s0, s1, [&](int, float x) {
        const uint32_t key = order_key(x);
        if ((key & mask) == prefix) atomicAdd(&mh[(key >> shift) & nbm], fixed_weight(x, lmax, inv_t));
      });
      __syncthreads();
      cluster_sync();  // every CTA's histogram is complete
      select_bin(mh, bits, above, need, C, sh, level == 0 ? p : -1.f);
      cluster_sync();  // the cluster has read every histogram
      if (level == 0) need = sh.need;
      prefix |= sh.digit << shift;
      mask |= nbm << shift;
      above = sh.acc;
    }
    draw_segmented(row, s0, s1, lmax, inv_t, prefix, uniform[b], C, rank, log_z, out_tokens + b,
                   out_logprobs != nullptr ? out_logprobs + b : nullptr, sh);
    return;
  }
  if (fast) {
    // refine the bin of the k-th largest key until the keys at or above it
    // fit the candidate list (all CTAs take the same decisions)
    uint32_t prefix = sh.digit << 20, mask = 0xFFF00000u;
    unsigned long long above = sh.acc;
    unsigned long long n_ge = sh.acc + sh.bin_count;
#pragma unroll 1
    for (int level = 1; level < 3 && n_ge > static_cast<unsigned long long>(kCandMax); ++level) {
      const int bits = level == 1 ? 12 : 8;
      const int shift = level == 1 ? 8 : 0;
      for (int i = threadIdx.x; i < kBinsMax; i += kSampThreads) cnt[i] = 0;
      __syncthreads();
      for_range(row, s0, s1, [&](int, float x) {
        const uint32_t key = order_key(x);
        if ((key & mask) == prefix) atomicAdd(&cnt[(key >> shift) & ((1u << bits) - 1u)], 1u);
      });
      __syncthreads();
      cluster_sync();
      select_bin(cnt, bits, above, static_cast<unsigned long long>(k), C, sh);
      cluster_sync();
      prefix |= sh.digit << shift;
      mask |= ((1u << bits) - 1u) << shift;
      above = sh.acc;
      n_ge = sh.acc + sh.bin_count;
    }
    if (n_ge > static_cast<unsigned long long>(kCandMax)) {
      general = true;  // more than kCandMax keys tie at the k-th value
    } else {
      // gather every key >= prefix (the top-k and the rest of its bin)
      for_range(row, s0, s1, [&](int i, float x) {
        if (order_key(x) >= prefix) {
          const int at = atomicAdd(&sh.cand_n, 1);
          cand[at] = Cand{i, x};
        }
      });
      __syncthreads();
      cluster_sync();  // every candidate list is complete
      int* idx_s = reinterpret_cast<int*>(sh.hist);
      uint32_t* key_s = reinterpret_cast<uint32_t*>(idx_s + kCandMax);
      unsigned long long* w_s = sh.hist + kCandMax;  // bytes 8 KB .. 16 KB, after idx_s and key_s
      int n = 0;
      if (rank == 0) {
        // candidate j of the cluster: thread j reads it from its CTA's list
        int nr[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          nr[r] = r < static_cast<int>(C)
                      ? static_cast<int>(ld_cluster_u32(mapa_shared(smem_u32(&sh.cand_n), static_cast<uint32_t>(r))))
                      : 0;
        int base = 0, src = -1, at = 0;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
          if (src < 0 && static_cast<int>(threadIdx.x) < base + nr[r]) {
            src = r;
            at = threadIdx.x - base;
          }
          base += nr[r];
        }
        n = base;
        const float inv_t = 1.f / t;
        if (src >= 0) {
          const uint2 c = ld_cluster_u32x2(mapa_shared(smem_u32(&cand[at]), static_cast<uint32_t>(src)));
          const float x = __uint_as_float(c.y);
          idx_s[threadIdx.x] = static_cast<int>(c.x);
          key_s[threadIdx.x] = order_key(x);
          w_s[threadIdx.x] = fixed_weight(x, lmax, inv_t);
        }
      }
      cluster_sync();  // the first CTA has copied every list; the others may leave
      if (rank == 0) token = sample_candidates(idx_s, key_s, w_s, n, k, p, uniform[b], amax, sh);
    }
  }
  if (rank != 0) return;
  if (general) token = sample_general(row, V, lmax, 1.f / t, k, p, uniform[b], amax, sh);
  if (threadIdx.x == 0) {
    out_tokens[b] = token;
    if (out_logprobs != nullptr) out_logprobs[b] = row[token] - log_z;
  }
}

}  // namespace

int sample_launch(const float* logits, int rows, int vocab, const float* temperature, const int32_t* top_k,
                  const float* top_p, const float* uniform, int32_t* out_tokens, float* out_logprobs, bool pdl,
                  cudaStream_t s) {
  if (rows <= 0) return 0;
  // CTAs per row: a power of two up to 8 while the rows' clusters fit the SMs
  // once, and none for short rows
  int C = 1;
  const int sms = num_sms();
  while (C < 8 && vocab >= 16384 * C && static_cast<long long>(rows) * C * 2 <= sms) C *= 2;
  return launch_kernel_cluster(k_sample, dim3(rows * C), dim3(kSampThreads), 0, s, pdl, C, logits, vocab,
                               temperature, top_k, top_p, uniform, out_tokens, out_logprobs);
}

}  // namespace llama
