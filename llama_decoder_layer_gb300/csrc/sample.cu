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
// counts, top-p by a radix descent on mass, four 8-bit digits each.  Masses are
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

struct SampleShared {
  unsigned int count[256];
  unsigned long long mass[256];
  unsigned long long red_u[kSampWarps];
  float red_f[kSampWarps];
  float best_v[kSampWarps];
  int best_i[kSampWarps];
  uint32_t digit;
  unsigned long long acc;
  int token;
};

// Largest key t with count(key >= t) >= k (the k-th largest key), by four
// 8-bit digits from the top.
__device__ uint32_t kth_largest_key(const float* row, int V, int k, SampleShared& sh) {
  uint32_t prefix = 0, mask = 0;
  unsigned int need = static_cast<unsigned int>(k);
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kSampThreads) sh.count[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < V; i += kSampThreads) {
      const uint32_t key = order_key(row[i]);
      if ((key & mask) == prefix) atomicAdd(&sh.count[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int above = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (above + sh.count[d] >= need) break;
        above += sh.count[d];
      }
      sh.digit = static_cast<uint32_t>(d);
      sh.acc = need - above;
    }
    __syncthreads();
    need = static_cast<unsigned int>(sh.acc);
    prefix |= sh.digit << shift;
    mask |= 255u << shift;
  }
  return prefix;
}

// Largest key t with mass(key >= t) >= target, by four 8-bit digits from the
// top; mass in 40-bit fixed point.
__device__ uint32_t mass_threshold_key(const float* row, int V, float lmax, float inv_t, unsigned long long target,
                                       SampleShared& sh) {
  uint32_t prefix = 0, mask = 0;
  unsigned long long above_total = 0;  // mass of the keys above the current prefix range
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kSampThreads) sh.mass[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < V; i += kSampThreads) {
      const float l = row[i];
      const uint32_t key = order_key(l);
      if ((key & mask) == prefix) atomicAdd(&sh.mass[(key >> shift) & 255u], fixed_weight(l, lmax, inv_t));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long above = above_total;
      int d = 255;
      for (; d > 0; --d) {
        if (above + sh.mass[d] >= target) break;
        above += sh.mass[d];
      }
      sh.digit = static_cast<uint32_t>(d);
      sh.acc = above;
    }
    __syncthreads();
    above_total = sh.acc;
    prefix |= sh.digit << shift;
    mask |= 255u << shift;
  }
  return prefix;
}

__device__ __forceinline__ unsigned long long kept_mass(const float* row, int V, float lmax, float inv_t,
                                                        uint32_t t_key, SampleShared& sh) {
  unsigned long long m = 0;
  for (int i = threadIdx.x; i < V; i += kSampThreads) {
    const float l = row[i];
    if (order_key(l) >= t_key) m += fixed_weight(l, lmax, inv_t);
  }
  return block_sum_u64(m, sh.red_u);
}

__global__ void __launch_bounds__(kSampThreads) k_sample(const float* __restrict__ logits, int V,
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
  for (int i = threadIdx.x; i < V; i += kSampThreads) {
    const float x = row[i];
    if (x > best) {
      best = x;
      bi = i;
    }
  }
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
  for (int i = threadIdx.x; i < V; i += kSampThreads) se += expf(row[i] - lmax);
  const float log_z = lmax + logf(block_sum_f(se, sh.red_f));

  const float t = temperature[b];
  int token = amax;
  if (t >= kGreedyTemperature) {  // (a NaN temperature samples greedily)
    const float inv_t = 1.f / t;
    const int k = top_k[b];
    uint32_t t_key = 0;  // keep everything
    if (k > 0 && k < V) t_key = kth_largest_key(row, V, k, sh);
    const float p = top_p[b];
    if (p < 1.f) {
      const unsigned long long mass_k = kept_mass(row, V, lmax, inv_t, t_key, sh);
      const double pc = p > 0.f ? static_cast<double>(p) : 0.0;
      // at least one unit, so the threshold is the key of a token that has
      // weight (p -> 0 keeps the maximum and its ties)
      unsigned long long target = static_cast<unsigned long long>(pc * static_cast<double>(mass_k));
      if (target < 1) target = 1;
      const uint32_t t_p = mass_threshold_key(row, V, lmax, inv_t, target, sh);
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
