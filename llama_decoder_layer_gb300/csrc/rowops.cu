// Row-wise and indexing kernels: fused residual-add + RMSNorm (or, with the
// norm folded into the next projection, the add and each row's rsqrt), the
// folding of norm weights into a projection, cache slot mapping, the
// standalone paged-cache write, the embedding gather, the greedy argmax and
// the self-test of the bounded wait.  All are HBM-bound: 16-byte vector loads/stores, fp32
// arithmetic, warp-shuffle reductions.  They wait for the kernel before them
// (pdl_wait).  A norm over at most kEarlyTriggerRows rows (decode batches)
// lets the next kernel start at once, so the next GEMM sets up and requests its
// first weight tiles while the norm runs (70B decode layer 0.654 -> 0.650 ms,
// 8B 0.213 -> 0.208 ms from a CUDA graph, with the skip of accumulator rows
// past M in the GEMM epilogues).  Above that the next kernel starts when they
// complete: a norm over thousands of rows that let the following GEMM in early
// made the 70B prefill layer ~8% slower (measured).
//
// Sources: [LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B", §3
// input_layernorm (RMSNorm fused with the residual add; residual None on the
// first layer), the final RMSNorm and the Sampler (greedy = argmax);
// [WALKTHROUGH] "模型库与算子层 — 代码走读", Attention (_update_kv_cache into the
// block-paged cache) and LlamaModel (embed_tokens); [CODE-READING] "vLLM Llama
// 代码解析", §2.1 (final norm over hidden + residual).
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace llama {

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (warp == 0) {
    t = lane < (blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// The cache slot of token t: block_table[b][pos / bs] * bs + pos % bs, b the
// token's sequence (found in query_start_loc); -1 (and the error word) for a
// position outside its sequence or a block-table entry outside the cache.
__device__ __forceinline__ int32_t token_slot(const SlotMapArgs& m, int t) {
  int lo = 0, hi = m.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (m.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int pos = m.positions[t];
  const int j = pos / m.bs;
  if (pos < 0 || pos >= m.seq_lens[b] || j >= m.max_blocks) {
    report_error(m.err, kErrGuard, kWhereSlot);
    return -1;
  }
  const int blk = m.block_table[static_cast<size_t>(b) * m.max_blocks + j];
  if (blk < 0 || blk >= m.num_blocks) {
    report_error(m.err, kErrGuard, kWhereBlockTable);
    return -1;
  }
  return blk * m.bs + pos % m.bs;
}

// One CTA per output row.  Every thread holds up to MAXC 16-byte chunks of the
// row in registers, so the row is fully read before anything is written:
// res_out may alias x or res_in and h_out may alias x.  With sm.slots set (the
// input norm of a layer), the CTA of row t also writes token t's cache slot.
constexpr int kEarlyTriggerRows = 256;

template <int MAXC>
__global__ void __launch_bounds__(kNormThreads) k_add_rmsnorm(const uint4* __restrict__ x, const uint4* res_in,
                                                              uint4* res_out, uint4* h_out,
                                                              const uint4* __restrict__ gamma, int H, float eps,
                                                              const int32_t* __restrict__ qsl,
                                                              float* __restrict__ inv_out, const SlotMapArgs sm) {
  __shared__ float red[33];
  pdl_wait();
  if (gridDim.x <= kEarlyTriggerRows) pdl_trigger();
  const int out_row = blockIdx.x;
  if (sm.slots != nullptr && threadIdx.x == 0) sm.slots[out_row] = token_slot(sm, out_row);
  const int in_row = qsl != nullptr ? qsl[out_row + 1] - 1 : out_row;
  const int nch = H >> 3;
  const size_t ibase = static_cast<size_t>(in_row) * nch;
  const size_t obase = static_cast<size_t>(out_row) * nch;
  float v[MAXC][8];
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int i = threadIdx.x + c * kNormThreads;
    if (i < nch) {
      const uint4 a = x[ibase + i];
      v[c][0] = bf16_lo(a.x);
      v[c][1] = bf16_hi(a.x);
      v[c][2] = bf16_lo(a.y);
      v[c][3] = bf16_hi(a.y);
      v[c][4] = bf16_lo(a.z);
      v[c][5] = bf16_hi(a.z);
      v[c][6] = bf16_lo(a.w);
      v[c][7] = bf16_hi(a.w);
      if (res_in != nullptr) {
        const uint4 r = res_in[ibase + i];
        v[c][0] += bf16_lo(r.x);
        v[c][1] += bf16_hi(r.x);
        v[c][2] += bf16_lo(r.y);
        v[c][3] += bf16_hi(r.y);
        v[c][4] += bf16_lo(r.z);
        v[c][5] += bf16_hi(r.z);
        v[c][6] += bf16_lo(r.w);
        v[c][7] += bf16_hi(r.w);
      }
      // the new residual is a bf16 tensor; the norm is taken of that tensor
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[c][e] = round_bf16(v[c][e]);
        ss += v[c][e] * v[c][e];
      }
    }
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
  if (inv_out != nullptr && threadIdx.x == 0) inv_out[out_row] = inv;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int i = threadIdx.x + c * kNormThreads;
    if (i < nch) {
      if (res_out != nullptr) {
        uint4 r;
        r.x = pack_bf16x2(v[c][0], v[c][1]);
        r.y = pack_bf16x2(v[c][2], v[c][3]);
        r.z = pack_bf16x2(v[c][4], v[c][5]);
        r.w = pack_bf16x2(v[c][6], v[c][7]);
        res_out[obase + i] = r;
      }
      if (gamma == nullptr) continue;  // folded: the next GEMM applies inv (and gamma is in its weights)
      const uint4 g = gamma[i];
      uint4 h;
      h.x = pack_bf16x2(v[c][0] * inv * bf16_lo(g.x), v[c][1] * inv * bf16_hi(g.x));
      h.y = pack_bf16x2(v[c][2] * inv * bf16_lo(g.y), v[c][3] * inv * bf16_hi(g.y));
      h.z = pack_bf16x2(v[c][4] * inv * bf16_lo(g.z), v[c][5] * inv * bf16_hi(g.z));
      h.w = pack_bf16x2(v[c][6] * inv * bf16_lo(g.w), v[c][7] * inv * bf16_hi(g.w));
      h_out[obase + i] = h;
    }
  }
}

// The norm weights folded into the columns of the projection that follows the
// norm: w_folded[o, i] = bf16(w[o, i] * gamma[i]) (eight columns per thread).
__global__ void k_fold_norm(const uint4* __restrict__ gamma, const uint4* __restrict__ w, long long chunks,
                            int row_chunks, uint4* __restrict__ w_folded) {
  for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < chunks;
       c += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 a = w[c], g = gamma[c % row_chunks];
    uint4 o;
    o.x = pack_bf16x2(bf16_lo(a.x) * bf16_lo(g.x), bf16_hi(a.x) * bf16_hi(g.x));
    o.y = pack_bf16x2(bf16_lo(a.y) * bf16_lo(g.y), bf16_hi(a.y) * bf16_hi(g.y));
    o.z = pack_bf16x2(bf16_lo(a.z) * bf16_lo(g.z), bf16_hi(a.z) * bf16_hi(g.z));
    o.w = pack_bf16x2(bf16_lo(a.w) * bf16_lo(g.w), bf16_hi(a.w) * bf16_hi(g.w));
    w_folded[c] = o;
  }
}

// Self-test of the bounded wait: one thread waits on a shared-memory barrier
// that nothing arrives at.  The wait gives up after its wall-clock limit and
// the timeout is recorded in the error word, as in every kernel's waits.
__global__ void k_selftest_wait(int* err) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  if (!mbar_wait(b, 0, nullptr)) report_error(err, kErrTimeout, kWhereSelftest);
}

// Standalone cache write: one thread per 16-byte chunk of one (token, head)
// row of k and of v.
__global__ void k_kv_write(const uint4* __restrict__ k, const uint4* __restrict__ v, const int32_t* __restrict__ slots,
                           int T, int nkv, int d, int bs, int num_blocks, uint4* k_cache, uint4* v_cache, int* err) {
  const int cpr = d >> 3;  // chunks per head row
  const long long total = static_cast<long long>(T) * nkv * cpr;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % cpr);
    const int h = static_cast<int>((i / cpr) % nkv);
    const int t = static_cast<int>(i / (static_cast<long long>(cpr) * nkv));
    const int slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * bs) {
      report_error(err, kErrGuard, kWhereSlot);
      continue;
    }
    const size_t dst = ((static_cast<size_t>(slot / bs) * nkv + h) * bs + slot % bs) * cpr + c;
    k_cache[dst] = k[i];
    v_cache[dst] = v[i];
  }
}

__global__ void k_embed(const uint4* __restrict__ table, const int32_t* __restrict__ ids, int H, int vocab,
                        uint4* __restrict__ out, int* err) {
  pdl_wait();
  const int t = blockIdx.x;
  const int id = ids[t];
  const int nch = H >> 3;
  const bool ok = id >= 0 && id < vocab;
  if (!ok && threadIdx.x == 0) report_error(err, kErrGuard, kWhereTokenId);
  for (int i = threadIdx.x; i < nch; i += blockDim.x)
    out[static_cast<size_t>(t) * nch + i] = ok ? table[static_cast<size_t>(id) * nch + i] : make_uint4(0, 0, 0, 0);
}

// argmax over one row; ties resolve to the lowest index
__global__ void __launch_bounds__(1024) k_argmax(const float* __restrict__ logits, int vocab, int32_t* out) {
  __shared__ float sv[32];
  __shared__ int si[32];
  pdl_wait();
  const float* row = logits + static_cast<size_t>(blockIdx.x) * vocab;
  float best = -FLT_MAX;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < vocab; i += blockDim.x) {
    const float x = row[i];
    if (x > best) {  // indices increase along the loop: strict > keeps the lowest
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    best = lane < nw ? sv[lane] : -FLT_MAX;
    bi = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) {
        best = ov;
        bi = oi;
      }
    }
    if (lane == 0) out[blockIdx.x] = bi == 0x7fffffff ? 0 : bi;
  }
}

int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

int add_rmsnorm_launch(const void* x, const void* res_in, void* res_out, void* h_out, const void* gamma, int rows,
                       int H, float eps, const int32_t* row_index_qsl, bool pdl, cudaStream_t s, float* inv_out,
                       const SlotMapArgs* slot_map) {
  if (rows <= 0) return 0;
  const int nch = H / 8;
  const int per = (nch + kNormThreads - 1) / kNormThreads;
  auto X = static_cast<const uint4*>(x);
  auto R = static_cast<const uint4*>(res_in);
  auto RO = static_cast<uint4*>(res_out);
  auto HO = static_cast<uint4*>(h_out);
  auto G = static_cast<const uint4*>(gamma);
  SlotMapArgs sm{};
  if (slot_map != nullptr) sm = *slot_map;
  auto go = [&](auto kernel) {
    return launch_kernel(kernel, dim3(rows), dim3(kNormThreads), 0, s, pdl, X, R, RO, HO, G, H, eps, row_index_qsl,
                         inv_out, sm);
  };
  if (per <= 1) return go(k_add_rmsnorm<1>);
  if (per <= 2) return go(k_add_rmsnorm<2>);
  if (per <= 4) return go(k_add_rmsnorm<4>);
  if (per <= 8) return go(k_add_rmsnorm<8>);
  return cudaErrorInvalidValue;
}

int selftest_wait_launch(int* err, cudaStream_t s) {
  return launch_kernel(k_selftest_wait, dim3(1), dim3(1), 0, s, false, err);
}

int fold_norm_launch(const void* gamma, const void* w, int rows, int cols, void* w_folded, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return 0;
  const long long chunks = static_cast<long long>(rows) * (cols / 8);
  return launch_kernel(k_fold_norm, dim3(grid_for(chunks, 256)), dim3(256), 0, s, false,
                       static_cast<const uint4*>(gamma), static_cast<const uint4*>(w), chunks, cols / 8,
                       static_cast<uint4*>(w_folded));
}

int kv_write_launch(const void* k, const void* v, const int32_t* slots, int T, int n_kv, int head_dim,
                    int block_size, int num_blocks, void* k_cache, void* v_cache, int* err, cudaStream_t s) {
  if (T <= 0) return 0;
  const long long work = static_cast<long long>(T) * n_kv * (head_dim / 8);
  return launch_kernel(k_kv_write, dim3(grid_for(work, 256)), dim3(256), 0, s, false, static_cast<const uint4*>(k),
                       static_cast<const uint4*>(v), slots, T, n_kv, head_dim, block_size, num_blocks,
                       static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), err);
}

int embed_launch(const void* table, const int32_t* ids, int T, int H, int vocab, void* out, int* err, bool pdl,
                 cudaStream_t s) {
  if (T <= 0) return 0;
  return launch_kernel(k_embed, dim3(T), dim3(256), 0, s, pdl, static_cast<const uint4*>(table), ids, H, vocab,
                       static_cast<uint4*>(out), err);
}

int argmax_launch(const float* logits, int rows, int vocab, int32_t* out, bool pdl, cudaStream_t s) {
  if (rows <= 0) return 0;
  return launch_kernel(k_argmax, dim3(rows), dim3(1024), 0, s, pdl, logits, vocab, out);
}

}  // namespace llama
