// Sparse MoE block (the Qwen3 MoE MLP): router logits, top-k routing with
// renormalised weights, the selected experts' SiluAndMul FFNs as two grouped
// tensor-core GEMMs, and the weighted combine.
//
//   logits  = h W_router^T                        (fp32, k_gemm_tc)
//   ids, w  = top-k of each row (ties to the lower expert), w = softmax of the
//             k selected logits                   (k_moe_topk)
//   rows    = every (token, slot) pair copied into its expert's segment of a
//             permuted activation matrix; each segment is padded to whole
//             128-row tiles, so a GEMM tile belongs to one expert (k_moe_plan,
//             k_moe_scatter)
//   act     = SiluAndMul(rows W13_e^T)            (grouped k_gemm_tc, SwiGLU)
//   y       = act W2_e^T                          (grouped k_gemm_tc, bf16)
//   out[t]  = sum_j w[t, j] y[row(t, j)]          (fp32 in routing order, bf16 out)
//
// Each permuted row is computed independently of its position, so the order in
// which the scatter's atomics place a token inside its expert's segment does
// not change any result.
//
// Sources: [LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B",
// Qwen3MoeSparseMoeBlock (router over 128 experts, top-8 per token, two-layer
// expert FFNs, sum weighted by the routing weights, no shared expert);
// [WALKTHROUGH] "模型库与算子层 — 代码走读", Fused MoE (w13 [E, 2I, H], w2 [E, H, I],
// router, torch.topk, fused_moe_kernel).
#include <float.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace llama {

namespace {

constexpr int kMoeTile = 128;          // rows of a GEMM tile = segment granularity
constexpr int kPlanThreads = 1024;

// One warp per token: k rounds of a warp-wide argmax over the expert logits
// (equal values go to the lower index), then the softmax of the k selected
// logits.  E <= kMoeMaxExperts, k <= 32.
template <int PER_LANE>
__global__ void __launch_bounds__(256) k_moe_topk(const float* __restrict__ logits, int T, int E, int K,
                                                  int32_t* __restrict__ ids, float* __restrict__ wts) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float v[PER_LANE];
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? logits[static_cast<size_t>(t) * E + e] : -FLT_MAX;
  }
  float sel_v = 0.f;  // lane j < K keeps the j-th selection
  int sel_i = 0;
  for (int k = 0; k < K; ++k) {
    float best = -FLT_MAX;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j;
      if (e < E && (v[j] > best || (v[j] == best && e < bi))) {
        best = v[j];
        bi = e;
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
    if (lane == k) {
      sel_v = best;
      sel_i = bi;
    }
    if ((bi & 31) == lane) {  // the owner drops the chosen expert from the next rounds
#pragma unroll
      for (int j = 0; j < PER_LANE; ++j)
        if (lane + 32 * j == bi) v[j] = -FLT_MAX;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, sel_v, 0);  // the first selection is the largest
  const float ex = lane < K ? expf(sel_v - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < K) {
    ids[static_cast<size_t>(t) * K + lane] = sel_i;
    wts[static_cast<size_t>(t) * K + lane] = ex / sum;
  }
}

// exclusive prefix sum over the threads of the block (thread order)
__device__ __forceinline__ int block_exclusive_scan(int v, int* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  __syncthreads();
  if (lane == 31) red[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += t;
    }
    red[lane] = x;
  }
  __syncthreads();
  return (w > 0 ? red[w - 1] : 0) + inc - v;
}

// Loads the expert ids of pairs [i0, i0 + 4 * kPlanBatch * kPlanThreads), every
// load of a thread issued before any is used; ids beyond `pairs` read as -1.
constexpr int kPlanBatch = 4;
__device__ __forceinline__ void plan_load_ids(const int32_t* __restrict__ ids, int pairs, int i0,
                                              int (&v)[kPlanBatch][4]) {
  const int4* ids4 = reinterpret_cast<const int4*>(ids);
#pragma unroll
  for (int b = 0; b < kPlanBatch; ++b) {
    const int i = i0 + 4 * (b * kPlanThreads + static_cast<int>(threadIdx.x));
    if (i + 3 < pairs) {
      const int4 q = ids4[i / 4];
      v[b][0] = q.x;
      v[b][1] = q.y;
      v[b][2] = q.z;
      v[b][3] = q.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[b][j] = i + j < pairs ? ids[i + j] : -1;
    }
  }
}

// One CTA: tokens per expert, the padded segment offsets, a zeroed fill
// counter per expert, and the tile lists of both grouped GEMMs, {A row, B base
// row of the expert, N tile, valid rows}; the list lengths go to counts[0..1].
__global__ void __launch_bounds__(kPlanThreads) k_moe_plan(const int32_t* __restrict__ ids, int pairs, int E,
                                                           int nt1, int b1_rows, int nt2, int b2_rows,
                                                           int32_t* __restrict__ offset, int32_t* __restrict__ fill,
                                                           int4* __restrict__ tiles1, int4* __restrict__ tiles2,
                                                           int32_t* __restrict__ counts, int* err) {
  __shared__ int cnt[kPlanThreads];
  __shared__ int red[32];
  pdl_wait();
  const int e = threadIdx.x;
  cnt[e] = 0;
  __syncthreads();
  for (int i0 = 0; i0 < pairs; i0 += 4 * kPlanBatch * kPlanThreads) {
    int v[kPlanBatch][4];
    plan_load_ids(ids, pairs, i0, v);
#pragma unroll
    for (int b = 0; b < kPlanBatch; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int x = v[b][j];
        if (x >= 0 && x < E) atomicAdd(&cnt[x], 1);
        else if (i0 + 4 * (b * kPlanThreads + e) + j < pairs) report_error(err, kErrGuard, kWhereMoe);
      }
  }
  __syncthreads();
  const int c = e < E ? cnt[e] : 0;
  const int mt = (c + kMoeTile - 1) / kMoeTile;
  const int row0 = block_exclusive_scan(mt * kMoeTile, red);
  const int t1 = block_exclusive_scan(mt * nt1, red);
  const int t2 = block_exclusive_scan(mt * nt2, red);
  if (e < E) {
    offset[e] = row0;
    fill[e] = 0;
    for (int m = 0; m < mt; ++m) {
      const int rows = min(kMoeTile, c - m * kMoeTile);
      for (int n = 0; n < nt1; ++n) tiles1[t1 + m * nt1 + n] = make_int4(row0 + m * kMoeTile, e * b1_rows, n, rows);
      for (int n = 0; n < nt2; ++n) tiles2[t2 + m * nt2 + n] = make_int4(row0 + m * kMoeTile, e * b2_rows, n, rows);
    }
  }
  if (e == kPlanThreads - 1) {  // the last thread's exclusive sums plus its own share are the totals
    counts[0] = t1 + mt * nt1;
    counts[1] = t2 + mt * nt2;
  }
}

// One warp per (token, slot): place the pair in its expert's segment and copy
// the token's row there, eight 16-byte loads in flight per lane.
constexpr int kScatterWarps = 8;
constexpr int kScatterUnroll = 8;
__global__ void __launch_bounds__(kScatterWarps * 32) k_moe_scatter(
    const uint4* __restrict__ h, const int32_t* __restrict__ ids, int pairs, int K, int E, int chunks,
    const int32_t* __restrict__ offset, int32_t* __restrict__ fill, int32_t* __restrict__ slot_row,
    uint4* __restrict__ x_perm) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kScatterWarps + (threadIdx.x >> 5);
  if (i >= pairs) return;
  const int e = ids[i];
  if (e < 0 || e >= E) return;  // reported by the planning kernel
  int row = 0;
  if (lane == 0) {
    row = offset[e] + atomicAdd(&fill[e], 1);
    slot_row[i] = row;
  }
  row = __shfl_sync(0xffffffffu, row, 0);
  const uint4* src = h + static_cast<size_t>(i / K) * chunks;
  uint4* dst = x_perm + static_cast<size_t>(row) * chunks;
  for (int c0 = 0; c0 < chunks; c0 += 32 * kScatterUnroll) {
    uint4 v[kScatterUnroll];
#pragma unroll
    for (int u = 0; u < kScatterUnroll; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < chunks) v[u] = src[c];
    }
#pragma unroll
    for (int u = 0; u < kScatterUnroll; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < chunks) dst[c] = v[u];
    }
  }
}

// out[t] = sum_j w[t, j] * y[row(t, j)], fp32 in routing order, bf16 out.
__global__ void __launch_bounds__(256) k_moe_combine(const uint4* __restrict__ y, const int32_t* __restrict__ ids,
                                                     const float* __restrict__ wts, const int32_t* __restrict__ slot_row,
                                                     int K, int E, int chunks, uint4* __restrict__ out) {
  pdl_wait();
  const int t = blockIdx.x;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < K; ++j) {
      const int i = t * K + j;
      const int e = ids[i];
      if (e < 0 || e >= E) continue;
      const float w = wts[i];
      const uint4 v = y[static_cast<size_t>(slot_row[i]) * chunks + c];
      acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
      acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
      acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
      acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
      acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
      acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
      acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
      acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    out[static_cast<size_t>(t) * chunks + c] = o;
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

MoeLayout moe_layout(int T, int H, int E, int K, int I, int sms) {
  MoeLayout L{};
  const size_t pairs = static_cast<size_t>(T > 0 ? T : 1) * K;
  L.rows = pairs + static_cast<size_t>(E) * (kMoeTile - 1);
  L.rows = (L.rows + kMoeTile - 1) / kMoeTile * kMoeTile;
  const size_t mtiles = L.rows / kMoeTile;
  const int nt1 = (I + kMoeTile - 1) / kMoeTile, nt2 = (H + 255) / 256;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.logits = take(static_cast<size_t>(T > 0 ? T : 1) * E * 4);
  L.ids = take(pairs * 4);
  L.wts = take(pairs * 4);
  L.slot_row = take(pairs * 4);
  L.offset = take(static_cast<size_t>(E) * 4);
  L.fill = take(static_cast<size_t>(E) * 4);
  L.counts = take(2 * 4);
  L.tiles1 = take(mtiles * nt1 * 16);
  L.tiles2 = take(mtiles * nt2 * 16);
  L.x_perm = take(L.rows * H * 2);
  L.act = take(L.rows * I * 2);
  L.y_perm = take(L.rows * H * 2);
  L.gpart = take(gemm_partials_bytes(sms));
  L.gpart_bytes = gemm_partials_bytes(sms);
  L.total = off + 256;
  return L;
}

int moe_launch(const MoeArgs& a, cudaStream_t s) {
  if (a.T <= 0) return 0;
  const MoeLayout L = moe_layout(a.T, a.H, a.E, a.K, a.I, num_sms());
  uint8_t* ws = a.ws;
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
  float* wts = reinterpret_cast<float*>(ws + L.wts);
  int32_t* slot_row = reinterpret_cast<int32_t*>(ws + L.slot_row);
  int32_t* offset = reinterpret_cast<int32_t*>(ws + L.offset);
  int32_t* fill = reinterpret_cast<int32_t*>(ws + L.fill);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int4* tiles1 = reinterpret_cast<int4*>(ws + L.tiles1);
  int4* tiles2 = reinterpret_cast<int4*>(ws + L.tiles2);
  void* x_perm = ws + L.x_perm;
  void* act = ws + L.act;
  void* y_perm = ws + L.y_perm;
  const int pairs = a.T * a.K;
  const int chunks = a.H / 8;

  // router logits (fp32), the first kernel of the call
  GemmArgs g{};
  g.epi = kEpiF32;
  g.A = a.h;
  g.B = a.w_router;
  g.M = a.T;
  g.N = a.E;
  g.K = a.H;
  g.out = logits;
  g.ldo = a.E;
  g.partials = reinterpret_cast<float*>(ws + L.gpart);
  g.partials_bytes = L.gpart_bytes;
  g.err = a.err;
  g.force_mode = -1;
  g.pdl = a.chain ? 1 : 0;
  int e = gemm_launch(g, s);
  if (e) return e;
  const int per_lane = (a.E + 31) / 32;
  const dim3 gt((a.T + 7) / 8);
  cudaError_t ce;
  if (per_lane <= 4)
    ce = launch_kernel(k_moe_topk<4>, gt, dim3(256), 0, s, true, logits, a.T, a.E, a.K, ids, wts);
  else if (per_lane <= 8)
    ce = launch_kernel(k_moe_topk<8>, gt, dim3(256), 0, s, true, logits, a.T, a.E, a.K, ids, wts);
  else
    ce = launch_kernel(k_moe_topk<16>, gt, dim3(256), 0, s, true, logits, a.T, a.E, a.K, ids, wts);
  if (ce != cudaSuccess) return ce;
  const int nt1 = (a.I + kMoeTile - 1) / kMoeTile, nt2 = (a.H + 255) / 256;
  ce = launch_kernel(k_moe_plan, dim3(1), dim3(kPlanThreads), 0, s, true, ids, pairs, a.E, nt1, 2 * a.I, nt2, a.H,
                     offset, fill, tiles1, tiles2, counts, a.err);
  if (ce != cudaSuccess) return ce;
  ce = launch_kernel(k_moe_scatter, dim3((pairs + kScatterWarps - 1) / kScatterWarps), dim3(kScatterWarps * 32), 0, s,
                     true, static_cast<const uint4*>(a.h), ids, pairs, a.K, a.E, chunks, offset, fill, slot_row,
                     static_cast<uint4*>(x_perm));
  if (ce != cudaSuccess) return ce;
  // experts' gate/up projections + SiluAndMul over the permuted rows
  GemmArgs g1{};
  g1.epi = kEpiSwiGlu;
  g1.A = x_perm;
  g1.B = a.w13;
  g1.M = static_cast<int>(L.rows);
  g1.N = 2 * a.I;
  g1.K = a.H;
  g1.out = act;
  g1.ldo = a.I;
  g1.err = a.err;
  g1.force_mode = 0;
  g1.pdl = 1;
  g1.group_tiles = tiles1;
  g1.group_count = counts;
  g1.b_rows = a.E * 2 * a.I;
  e = gemm_launch(g1, s);
  if (e) return e;
  // experts' down projections
  GemmArgs g2{};
  g2.epi = kEpiBf16;
  g2.A = act;
  g2.B = a.w2;
  g2.M = static_cast<int>(L.rows);
  g2.N = a.H;
  g2.K = a.I;
  g2.out = y_perm;
  g2.ldo = a.H;
  g2.err = a.err;
  g2.force_mode = 0;
  g2.pdl = 1;
  g2.group_tiles = tiles2;
  g2.group_count = counts + 1;
  g2.b_rows = a.E * a.H;
  e = gemm_launch(g2, s);
  if (e) return e;
  ce = launch_kernel(k_moe_combine, dim3(a.T), dim3(256), 0, s, true, static_cast<const uint4*>(y_perm), ids, wts,
                     slot_row, a.K, a.E, chunks, static_cast<uint4*>(a.out));
  if (ce != cudaSuccess) return ce;
  if (a.out_ids != nullptr)
    ce = cudaMemcpyAsync(a.out_ids, ids, static_cast<size_t>(pairs) * 4, cudaMemcpyDeviceToDevice, s);
  if (ce == cudaSuccess && a.out_wts != nullptr)
    ce = cudaMemcpyAsync(a.out_wts, wts, static_cast<size_t>(pairs) * 4, cudaMemcpyDeviceToDevice, s);
  return ce;
}

}  // namespace llama
