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
// One CTA per row.  Thresholds are found on the logits' order-preserving
// 32-bit keys (dividing by T > 0 keeps the order): top-k by a radix select on
// counts, top-p by a radix descent on mass, digits of 12, 12 and 8 bits.  Masses are
// 64-bit fixed point (w_i * 2^40, w_i in (0, 1]), so every histogram, sum and
// scan is exact integer arithmetic: the result does not depend on the order of
// the atomic adds, and the same call always returns the same tokens.
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

struct SampleShared {
  unsigned long long hist[kBinsMax];
  unsigned long long red_u[kSampWarps];
  float red_f[kSampWarps];
  float best_v[kSampWarps];
  int best_i[kSampWarps];
  uint32_t digit;
  unsigned long long acc;
  int token;
};

// Every pass over a row goes through for_row: each thread loads kUnroll
// elements (stride kSampThreads) before it uses any of them, so a thread keeps
// that many L2 requests in flight (one CTA per row is all the parallelism a
// 34-row head gives).
constexpr int kUnroll = 8;

template <class F>
__device__ __forceinline__ void for_row(const float* __restrict__ row, int V, F&& f) {
  for (int base = threadIdx.x; base < V; base += kSampThreads * kUnroll) {
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kSampThreads;
      x[u] = i < V ? __ldg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kSampThreads;
      if (i < V) f(i, x[u]);
    }
  }
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

__global__ void __launch_bounds__(kSampThreads, 1) k_sample(const float* __restrict__ logits, int V,
                                                          const float* __restrict__ temperature,
                                                          const int32_t* __restrict__ top_k,
                                                          const float* __restrict__ top_p,
                                                          const float* __restrict__ uniform,
                                                          int32_t* __restrict__ out_tokens,
                                                          float* __restrict__ out_logprobs) {
  __shared__ SampleShared sh;
  pdl_wait();
  const int b = blockIdx.x;
  const float* row = logits + static_cast<size_t>(b) * V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // maximum and its lowest index
  float best = -FLT_MAX;
  int bi = 0x7fffffff;
  for_row(row, V, [&](int i, float x) {  // i increases within a thread: strict > keeps the lowest
    if (x > best) {
      best = x;
      bi = i;
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    sh.best_v[warp] = best;
    sh.best_i[warp] = bi;
  }
  __syncthreads();
  best = lane < kSampWarps ? sh.best_v[lane] : -FLT_MAX;
  bi = lane < kSampWarps ? sh.best_i[lane] : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  const float lmax = best;
  const int amax = bi == 0x7fffffff ? 0 : bi;

  // log of the raw normaliser
  float se = 0.f;
  for_row(row, V, [&](int, float x) { se += expf(x - lmax); });
  const float log_z = lmax + logf(block_sum_f(se, sh.red_f));

  const float t = temperature[b];
  int token = amax;
  if (t >= kGreedyTemperature) {  // (a NaN temperature samples greedily)
    const float inv_t = 1.f / t;
    const int k = top_k[b];
    uint32_t t_key = 0;  // keep everything
    if (k > 0 && k < V)
      t_key = threshold_key<false>(row, V, lmax, inv_t, static_cast<unsigned long long>(k), 0u, sh);
    const float p = top_p[b];
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
    float u = uniform[b];
    u = u > 0.f ? (u < 1.f ? u : 0.99999994f) : 0.f;
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
    token = sh.token;
  }
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
  return launch_kernel(k_sample, dim3(rows), dim3(kSampThreads), 0, s, pdl, logits, vocab, temperature, top_k, top_p,
                       uniform, out_tokens, out_logprobs);
}

}  // namespace llama
