// Paged, causal, grouped-query attention over the block-paged KV cache.
//
//   o[t, h] = sum_j softmax_j(q[t, h] . K[b, h / g, j] / sqrt(d)) V[b, h / g, j],
//   j = 0 .. position(t)  (the current tokens are already in the cache)
//
// The q heads sharing one KV head (g = n_heads / n_kv_heads of them) are
// processed together, so every K/V block is loaded from memory once per group.
// K/V blocks (16 tokens x head_dim of one KV head, contiguous in the cache) are
// fetched by TMA with 128-byte swizzle; softmax is online, in the exp2 domain.
//
// * decode (query length 1): split-KV, ldmatrix + mma.sync (bf16 in, fp32
//   accumulate: the group's q heads fill only 8 of 16 MMA rows, too few for
//   the 128-row tensor-memory MMA).  One CTA per (sequence, KV head, chunk of
//   up to 1536 keys); its 4 warps stream disjoint blocks of the chunk through
//   their own 3-stage TMA rings, merge in shared memory, and either write the
//   output (one chunk) or a partial (unnormalised o, running max, sum) that
//   k_attn_combine merges in chunk order.  (Merging in the decode kernel
//   itself, by the chunk CTA that completes a per-(sequence, KV head) arrival
//   count, was measured slower: the fence and atomic every chunk CTA then pays
//   hold its SM slot.)
// * prefill (query length >= 2), head_dim 128: k_attn_prefill_tc on the
//   tensor-memory MMA (S and O accumulate in TMEM, P goes back to TMEM as the
//   A operand of P V); other shapes: k_attn_prefill, one CTA per (sequence,
//   KV head, 16 query tokens), warp w owns q head w of the group, mma.sync.
// * In a batch with prefill sequences the decode kernels run on a side stream
//   beside the prefill kernel (HBM-bound next to tensor-bound work).
//
// Sources: [WALKTHROUGH] "模型库与算子层 — 代码走读", Attention
// (attn_backend.forward(q, k, v, kv_cache.block_table) after _update_kv_cache);
// [LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B", config.json and §4
// (grouped-query attention, 64 q heads over 8 kv heads).
#include <math.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace llama {

namespace {

constexpr int kBS = 16;             // tokens per cache block
constexpr int kDecWarps = 4;
constexpr int kDecStages = 3;
constexpr int kChunkBlocks = 96;    // a sequence splits into ceil(keys / 1536) split-KV chunks (sweep:
                                    // 512 -> 1536 keys took the 70B decode batch from 0.372 to 0.329 ms)
constexpr int kPreStages = 2;
constexpr int kPreKeys = 64;        // keys per prefill K/V tile (4 blocks)
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* positions;
  const int32_t* block_table;
  int max_blocks, num_blocks, nq, nkv, group, max_chunks;
  float scale_log2;
  float* part_o;
  float2* part_ml;
  uint32_t* pre_items;  // prefill work list: (sequence << 16) | q-tile, 0xFFFFFFFF past the end
  int* err;
};

constexpr uint32_t kNoItem = 0xFFFFFFFFu;

// number of prefill work items the host sizes the list for: at most
// ceil(q_len / tile) per sequence, tile >= 8 tokens, so at most T / 8 + B
__host__ __device__ __forceinline__ int max_prefill_items(int T, int B) { return (T + 7) / 8 + B; }

__host__ __device__ constexpr int tile_bytes(int D) { return kBS * D * 2; }

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// zero the bf16 halves of a V fragment register whose key is >= n_keys
__device__ __forceinline__ uint32_t mask_pair(uint32_t r, int key_lo, int n_keys) {
  if (key_lo >= n_keys) return 0u;
  if (key_lo + 1 >= n_keys) return r & 0x0000FFFFu;
  return r;
}

// number of context chunks of a decode sequence with nblk cache blocks
__host__ __device__ __forceinline__ int num_chunks(int nblk) { return (nblk + kChunkBlocks - 1) / kChunkBlocks; }

// Online-softmax update of one 16-key block for the two rows (g, g+8) this
// thread holds; s[n][c] are scores already scaled to the log2 domain and
// masked (-inf).  Returns the P fragment as an m16k16 A operand.
__device__ __forceinline__ void softmax_block(float (&s)[2][4], float& m0, float& m1, float& l0, float& l1,
                                              float& alpha0, float& alpha1, uint32_t (&pa)[4]) {
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = quad_max(mx0);
  mx1 = quad_max(mx1);
  const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
  const float b0 = n0 == -INFINITY ? 0.f : n0;
  const float b1 = n1 == -INFINITY ? 0.f : n1;
  alpha0 = exp2f(m0 - b0);
  alpha1 = exp2f(m1 - b1);
  m0 = n0;
  m1 = n1;
  float p[2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    p[n][0] = exp2f(s[n][0] - b0);
    p[n][1] = exp2f(s[n][1] - b0);
    p[n][2] = exp2f(s[n][2] - b1);
    p[n][3] = exp2f(s[n][3] - b1);
  }
  l0 = l0 * alpha0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
  l1 = l1 * alpha1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
  pa[0] = pack_bf16x2(p[0][0], p[0][1]);
  pa[1] = pack_bf16x2(p[0][2], p[0][3]);
  pa[2] = pack_bf16x2(p[1][0], p[1][1]);
  pa[3] = pack_bf16x2(p[1][2], p[1][3]);
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kDecWarps * 32)
    k_attn_decode(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnParams p) {
  constexpr int TB = tile_bytes(D);
  constexpr int QS = (D + 8) * 2;  // padded row stride of the q tile (bytes)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t ring = raw + pad;                                   // [warp][stage][K | V]
  uint8_t* qtile = smem + kDecWarps * kDecStages * 2 * TB;           // [16][D + 8] bf16
  uint64_t* bars = reinterpret_cast<uint64_t*>(qtile + 16 * QS);     // [warp][stage]

  // The batch metadata, the block table and every cache block but the one
  // holding the sequence's new token are inputs of the call: no kernel of the
  // chain writes them (the new token's K/V slot, in the last block, is
  // written by the qkv epilogue).  They are read, and the chunk's first
  // blocks requested, before waiting for the previous kernel; the q rows and
  // the last block after it, and so is every global write.
  const int b = blockIdx.x / p.nkv, kvh = blockIdx.x % p.nkv, chunk = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = p.qsl[b];
  int err_where = -1;  // reported once the previous kernel has completed
  bool work = p.qsl[b + 1] - t0 == 1;
  const int pos = work ? p.positions[t0] : 0;
  const int n_keys = pos + 1;
  if (work && (pos < 0 || n_keys > p.seq_lens[b] || (n_keys + kBS - 1) / kBS > p.max_blocks)) {
    err_where = kWhereQueryLen;
    work = false;
  }
  const int nblk = (n_keys + kBS - 1) / kBS;
  const int nch = work ? num_chunks(nblk) : 0;
  if (work && nch > p.max_chunks) {  // context longer than the launch's max_seq_len
    err_where = kWhereQueryLen;
    work = false;
  }
  if (!work || chunk >= nch) {
    pdl_wait();
    pdl_trigger();
    if (err_where >= 0 && chunk == 0 && kvh == 0 && threadIdx.x == 0) report_error(p.err, kErrGuard, err_where);
    return;
  }
  // Chunk c of nch covers a share of the sequence's blocks that falls with c
  // (8:1 for two chunks, nch + 1 - c for more), and the grid dispatches every
  // sequence's chunk 0 first, then every chunk 1, ..., so the last CTAs of
  // the launch are the shortest and fill the last wave more evenly.
  int wsum = 0, wpre = 0, wcur = 0;
  for (int c = 0; c < nch; ++c) {
    const int w = nch <= 2 ? (nch - c) * (nch - c) * (nch - c) : nch + 1 - c;
    if (c < chunk) wpre += w;
    if (c == chunk) wcur = w;
    wsum += w;
  }
  const int blk0 = static_cast<int>(static_cast<long long>(nblk) * wpre / wsum);
  const int blk1 = static_cast<int>(static_cast<long long>(nblk) * (wpre + wcur) / wsum);
  const int G = p.group;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecWarps * kDecStages; ++i) mbar_init(smem_u32(bars + i), 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int nb_w = blk0 + warp < blk1 ? (blk1 - blk0 - warp + kDecWarps - 1) / kDecWarps : 0;
  const uint32_t wring = ring + warp * kDecStages * 2 * TB;
  const uint32_t wbar = smem_u32(bars + warp * kDecStages);
  const uint64_t pol = policy_evict_first();
  const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks;

  auto issue_blk = [&](int i, int blk) {
    const int row = (blk * p.nkv + kvh) * kBS;
    const int st = i % kDecStages;
    const uint32_t dst = wring + st * 2 * TB;
    const uint32_t bar = wbar + 8 * st;
    mbar_arrive_expect_tx(bar, 2 * TB);
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx) {
      tma_load_2d(dst + bx * 2048, &tmK, bar, bx * 64, row, pol);
      tma_load_2d(dst + TB + bx * 2048, &tmV, bar, bx * 64, row, pol);
    }
  };
  auto issue = [&](int i) {  // after the wait: reports a bad block table entry
    int blk = bt[blk0 + warp + kDecWarps * i];
    if (blk < 0 || blk >= p.num_blocks) {
      report_error(p.err, kErrGuard, kWhereBlockTable);
      blk = 0;
    }
    issue_blk(i, blk);
  };

  // first stages before the wait: blocks other than the last, with valid entries
  int n_early = 0;
  if (lane == 0) {
    for (; n_early < kDecStages && n_early < nb_w; ++n_early) {
      const int jb = blk0 + warp + kDecWarps * n_early;
      const int blk = bt[jb];
      if (jb == nblk - 1 || blk < 0 || blk >= p.num_blocks) break;
      issue_blk(n_early, blk);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (lane == 0)
    for (int i = n_early; i < kDecStages && i < nb_w; ++i) issue(i);
  __syncwarp();

  // q rows of the group (rows >= G are zero padding)
  for (int i = threadIdx.x; i < 16 * (D / 8); i += blockDim.x) {
    const int r = i / (D / 8), c = i % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < G) v = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(t0) * p.nq + kvh * G + r) * D)[c];
    *reinterpret_cast<uint4*>(qtile + r * QS + c * 16) = v;
  }
  __syncthreads();

  // A fragments of q for all head_dim/16 k-steps
  uint32_t qa[D / 16][4];
  {
    const int m = lane >> 3;
    const int row = (m & 1) * 8 + (lane & 7);
    const uint32_t base = smem_u32(qtile) + row * QS + (m >> 1) * 16;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) ldsm_x4(base + kk * 32, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool ok = true;
  int done = 0;

  for (int i = 0; i < nb_w; ++i) {
    const int st = i % kDecStages;
    if (!mbar_wait(wbar + 8 * st, (i / kDecStages) & 1, nullptr)) {
      ok = false;
      break;
    }
    done = i + 1;
    const uint32_t kt = wring + st * 2 * TB;
    const uint32_t vt = kt + TB;
    const int key0 = (blk0 + warp + kDecWarps * i) * kBS;

    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int krow = (lane >> 4) * 8 + (lane & 7);
      const int csel = (lane >> 3) & 1;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int ch = 2 * kk + csel;
        uint32_t r0, r1, r2, r3;
        ldsm_x4(kt + (ch >> 3) * 2048 + sw128_offset(krow, ch & 7), r0, r1, r2, r3);
        mma_bf16_16816(s[0], qa[kk], r0, r1);
        mma_bf16_16816(s[1], qa[kk], r2, r3);
      }
    }
    const int kq = key0 + 2 * (lane & 3);
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = kq + n * 8 + (c & 1);
        s[n][c] = key < n_keys ? s[n][c] * p.scale_log2 : -INFINITY;
      }
    float a0, a1;
    uint32_t pa[4];
    softmax_block(s, m0, m1, l0, l1, a0, a1, pa);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= a0;
      o[n][1] *= a0;
      o[n][2] *= a1;
      o[n][3] *= a1;
    }
    {
      const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
      const int csel = lane >> 4;
      const bool tail = key0 + kBS > n_keys;
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        const int ch = 2 * nd + csel;
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(vt + (ch >> 3) * 2048 + sw128_offset(vrow, ch & 7), r0, r1, r2, r3);
        if (tail) {
          r0 = mask_pair(r0, kq, n_keys);
          r1 = mask_pair(r1, kq + 8, n_keys);
          r2 = mask_pair(r2, kq, n_keys);
          r3 = mask_pair(r3, kq + 8, n_keys);
        }
        mma_bf16_16816(o[2 * nd], pa, r0, r1);
        mma_bf16_16816(o[2 * nd + 1], pa, r2, r3);
      }
    }
    __syncwarp();
    fence_proxy_async_smem();
    if (lane == 0 && i + kDecStages < nb_w) issue(i + kDecStages);
    __syncwarp();
  }
  if (!ok) {
    if (lane == 0) report_error(p.err, kErrTimeout, kWhereAttnDecode);
    // let the loads still in flight land before the shared memory is reused
    for (int i = done; i < nb_w && i < done + kDecStages; ++i)
      mbar_wait(wbar + 8 * (i % kDecStages), (i / kDecStages) & 1, nullptr);
  }
  l0 = quad_sum(l0);
  l1 = quad_sum(l1);

  // merge the warps' partial softmax states in shared memory (ring reused)
  __syncthreads();
  float* mbuf = reinterpret_cast<float*>(smem);           // [warp][16]
  float* lbuf = mbuf + kDecWarps * 16;                     // [warp][16]
  float* obuf = lbuf + kDecWarps * 16;                     // [warp][16][D]
  {
    const int g = lane >> 2;
    if ((lane & 3) == 0) {
      mbuf[warp * 16 + g] = ok ? m0 : -INFINITY;
      mbuf[warp * 16 + g + 8] = ok ? m1 : -INFINITY;
      lbuf[warp * 16 + g] = l0;
      lbuf[warp * 16 + g + 8] = l1;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int col = n * 8 + 2 * (lane & 3);
      obuf[(warp * 16 + g) * D + col] = o[n][0];
      obuf[(warp * 16 + g) * D + col + 1] = o[n][1];
      obuf[(warp * 16 + g + 8) * D + col] = o[n][2];
      obuf[(warp * 16 + g + 8) * D + col + 1] = o[n][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int r = idx / D, col = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mbuf[w * 16 + r]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = exp2f(mbuf[w * 16 + r] - M);
        L += lbuf[w * 16 + r] * f;
        O += obuf[(w * 16 + r) * D + col] * f;
      }
    }
    const int h = kvh * G + r;
    if (nch == 1) {
      p.out[static_cast<size_t>(t0) * p.nq * D + h * D + col] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
    } else {
      const size_t pi = (static_cast<size_t>(b) * p.max_chunks + chunk) * p.nq + h;
      p.part_o[pi * D + col] = O;
      if (col == 0) p.part_ml[pi] = make_float2(M, L);
    }
  }
}

// Merges the split-KV partials of every multi-chunk decode sequence: one CTA
// per (sequence, kCombineThreads * 4 / D q heads), a thread per 4 output
// columns of one head, chunks in order.  (One CTA per head and a thread per
// column gave thousands of short CTAs whose launch and load latency, not the
// bytes, set the time.)
constexpr int kCombineThreads = 256;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) k_attn_combine(AttnParams p) {
  pdl_wait();
  pdl_trigger();
  constexpr int kThreadsPerHead = D / 4;
  const int b = blockIdx.y;
  const int h = blockIdx.x * (kCombineThreads / kThreadsPerHead) + threadIdx.x / kThreadsPerHead;
  const int col = (threadIdx.x % kThreadsPerHead) * 4;
  if (h >= p.nq) return;
  const int t0 = p.qsl[b];
  if (p.qsl[b + 1] - t0 != 1) return;
  const int pos = p.positions[t0];
  const int n_keys = pos + 1;
  if (pos < 0 || n_keys > p.seq_lens[b] || (n_keys + kBS - 1) / kBS > p.max_blocks) return;
  const int nch = num_chunks((n_keys + kBS - 1) / kBS);
  if (nch <= 1 || nch > p.max_chunks) return;
  const size_t base = static_cast<size_t>(b) * p.max_chunks * p.nq + h;
  float M = -INFINITY;
  for (int c = 0; c < nch; ++c) M = fmaxf(M, p.part_ml[base + static_cast<size_t>(c) * p.nq].x);
  float L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int c = 0; c < nch; ++c) {
      const size_t pi = base + static_cast<size_t>(c) * p.nq;
      const float2 ml = p.part_ml[pi];
      const float4 o = *reinterpret_cast<const float4*>(p.part_o + pi * D + col);
      const float f = exp2f(ml.x - M);
      L += ml.y * f;
      O.x += o.x * f;
      O.y += o.y * f;
      O.z += o.z * f;
      O.w += o.w * f;
    }
  }
  uint2 u;
  u.x = pack_bf16x2(L > 0.f ? O.x / L : 0.f, L > 0.f ? O.y / L : 0.f);
  u.y = pack_bf16x2(L > 0.f ? O.z / L : 0.f, L > 0.f ? O.w / L : 0.f);
  *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(t0) * p.nq * D + h * D + col) = u;
}

// ---------------------------------------------------------------------------
// prefill
// ---------------------------------------------------------------------------
// Lists the prefill work: the 16-token query tiles of every sequence with at
// least two new tokens, longest causal range first within a sequence, so the
// prefill grid holds no CTAs for decode sequences.  One CTA, a block-wide
// exclusive scan over the sequences in rounds of 1024.
__global__ void __launch_bounds__(1024) k_attn_plan(const int32_t* __restrict__ qsl, int B, int tile_tokens,
                                                    uint32_t* items, int max_items) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int n = 0;
    if (b < B) {
      const int ql = qsl[b + 1] - qsl[b];
      n = ql >= 2 ? (ql + tile_tokens - 1) / tile_tokens : 0;
    }
    int inc = n;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = lane < static_cast<int>(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += t;
      }
      warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + inc - n;
    for (int j = 0; j < n; ++j)
      if (excl + j < max_items) items[excl + j] = (static_cast<uint32_t>(b) << 16) | static_cast<uint32_t>(n - 1 - j);
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_tot[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
  for (int i = carry + threadIdx.x; i < max_items; i += blockDim.x) items[i] = kNoItem;
}

constexpr int kPreMaxHeads = 8;  // q heads (consumer warps) per prefill CTA

template <int D>
__global__ void __launch_bounds__((kPreMaxHeads + 1) * 32)
    k_attn_prefill(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnParams p) {
  constexpr int TB = tile_bytes(D);      // one 16-key block of K (or V)
  constexpr int STB = 4 * TB;            // 64 keys
  constexpr int QS = (D + 8) * 2;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t ring = raw + pad;                               // [stage][K 64 keys | V 64 keys]
  uint8_t* qtiles = smem + kPreStages * 2 * STB;                 // [warp][16][D + 8]
  uint64_t* bars = reinterpret_cast<uint64_t*>(qtiles + kPreMaxHeads * 16 * QS);  // full[S], empty[S]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kPreStages);

  pdl_wait();
  pdl_trigger();
  const int n_hc = (p.group + kPreMaxHeads - 1) / kPreMaxHeads;  // head chunks per KV head
  const uint32_t item = p.pre_items[blockIdx.y];
  if (item == kNoItem) return;
  const int b = static_cast<int>(item >> 16), qt = static_cast<int>(item & 0xFFFFu);
  const int kvh = blockIdx.x / n_hc, hc = blockIdx.x % n_hc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = min(kPreMaxHeads, p.group - hc * kPreMaxHeads);  // q heads of this CTA
  const int h_first = kvh * p.group + hc * kPreMaxHeads;
  if (warp > G) return;
  const int t0 = p.qsl[b];
  const int qlen = p.qsl[b + 1] - t0;
  if (qlen < 2 || qt * 16 >= qlen) return;
  const int tq = t0 + qt * 16;              // first token of this q tile
  const int nrows = min(16, qlen - qt * 16);

  // largest position of the tile (keys needed: 0 .. p_hi)
  int p_hi = -1;
  for (int r = 0; r < nrows; ++r) p_hi = max(p_hi, p.positions[tq + r]);
  const int n_keys = p_hi + 1;
  if (n_keys > p.seq_lens[b] || (n_keys + kBS - 1) / kBS > p.max_blocks) {
    if (kvh == 0 && threadIdx.x == 0) report_error(p.err, kErrGuard, kWhereQueryLen);
    return;
  }
  const int ntiles = (n_keys + kPreKeys - 1) / kPreKeys;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kPreStages;

  if (warp < G) {
    uint8_t* qs = qtiles + warp * 16 * QS;
    const int h = h_first + warp;
    for (int i = lane; i < 16 * (D / 8); i += 32) {
      const int r = i / (D / 8), c = i % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < nrows) v = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(tq + r) * p.nq + h) * D)[c];
      *reinterpret_cast<uint4*>(qs + r * QS + c * 16) = v;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPreStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, G);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == G) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks;
      const int nblk = (n_keys + kBS - 1) / kBS;
      uint32_t uses[kPreStages] = {};
      bool ok = true;
      for (int kt = 0; kt < ntiles && ok; ++kt) {
        const int st = kt % kPreStages;
        if (!mbar_wait(empty0 + 8 * st, ((kt / kPreStages) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        int nload = min(4, nblk - kt * 4);
        mbar_arrive_expect_tx(full0 + 8 * st, nload * 2 * TB);
        for (int i = 0; i < nload; ++i) {
          int blk = bt[kt * 4 + i];
          if (blk < 0 || blk >= p.num_blocks) {
            report_error(p.err, kErrGuard, kWhereBlockTable);
            blk = 0;
          }
          const int row = (blk * p.nkv + kvh) * kBS;
          const uint32_t dst = ring + st * 2 * STB + i * TB;
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx) {
            tma_load_2d(dst + bx * 2048, &tmK, full0 + 8 * st, bx * 64, row, pol);
            tma_load_2d(dst + STB + bx * 2048, &tmV, full0 + 8 * st, bx * 64, row, pol);
          }
        }
        uses[st]++;
      }
      if (!ok) {
        report_error(p.err, kErrTimeout, kWhereAttnPrefill);
        *abort_flag = 1;
      }
      for (int s = 0; s < kPreStages; ++s)
        if (uses[s] > 0) mbar_wait(full0 + 8 * s, (uses[s] - 1) & 1u, nullptr);
    }
    return;
  }
  if (warp >= G) return;

  // ---------------- consumer warps: q head kvh*G + warp ----------------
  uint32_t qa[D / 16][4];
  {
    const int m = lane >> 3;
    const int row = (m & 1) * 8 + (lane & 7);
    const uint32_t base = smem_u32(qtiles + warp * 16 * QS) + row * QS + (m >> 1) * 16;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) ldsm_x4(base + kk * 32, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }
  const int g = lane >> 2;
  const int pos0 = g < nrows ? p.positions[tq + g] : -1;      // row g
  const int pos1 = g + 8 < nrows ? p.positions[tq + g + 8] : -1;  // row g + 8
  int p_lo = p_hi;
  for (int r = 0; r < nrows; ++r) p_lo = min(p_lo, p.positions[tq + r]);

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool ok = true;

  for (int kt = 0; kt < ntiles; ++kt) {
    const int st = kt % kPreStages;
    if (!mbar_wait(full0 + 8 * st, (kt / kPreStages) & 1, abort_flag)) {
      ok = false;
      break;
    }
    const uint32_t ks = ring + st * 2 * STB;
    const uint32_t vs = ks + STB;
    const int kbase = kt * kPreKeys;
    const bool need_mask = kbase + kPreKeys - 1 > p_lo;
    const int nblk_t = min(4, (n_keys - kbase + kBS - 1) / kBS);  // 16-key blocks holding keys (warp-uniform)
    // S = q K^T over the whole 64-key tile (8 n-tiles of 8 keys)
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    {
      const int krow = (lane >> 4) * 8 + (lane & 7);
      const int csel = (lane >> 3) & 1;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        if (blk < nblk_t) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int ch = 2 * kk + csel;
            uint32_t r0, r1, r2, r3;
            ldsm_x4(ks + blk * TB + (ch >> 3) * 2048 + sw128_offset(krow, ch & 7), r0, r1, r2, r3);
            mma_bf16_16816(s[2 * blk], qa[kk], r0, r1);
            mma_bf16_16816(s[2 * blk + 1], qa[kk], r2, r3);
          }
        }
      }
    }
    // scale to the log2 domain; causal mask (keys past n_keys are past every
    // row's position, so the same test removes them)
    const int kq = kbase + 2 * (lane & 3);
    if (need_mask) {
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = kq + n * 8 + (c & 1);
          const int lim = c < 2 ? pos0 : pos1;
          s[n][c] = key <= lim ? s[n][c] * p.scale_log2 : -INFINITY;
        }
    } else {
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[n][c] *= p.scale_log2;
    }
    // online softmax once per tile: new row maxima, rescale of O and l
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
      mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
    }
    mx0 = quad_max(mx0);
    mx1 = quad_max(mx1);
    const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
    const float b0 = nm0 == -INFINITY ? 0.f : nm0;
    const float b1 = nm1 == -INFINITY ? 0.f : nm1;
    const float a0 = exp2f(m0 - b0), a1 = exp2f(m1 - b1);
    m0 = nm0;
    m1 = nm1;
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      s[n][0] = exp2f(s[n][0] - b0);
      s[n][1] = exp2f(s[n][1] - b0);
      s[n][2] = exp2f(s[n][2] - b1);
      s[n][3] = exp2f(s[n][3] - b1);
      ls0 += s[n][0] + s[n][1];
      ls1 += s[n][2] + s[n][3];
    }
    l0 = l0 * a0 + ls0;
    l1 = l1 * a1 + ls1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= a0;
      o[n][1] *= a0;
      o[n][2] *= a1;
      o[n][3] *= a1;
    }
    // O += P V, one 16-key block per k-step
    {
      const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
      const int csel = lane >> 4;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        if (blk < nblk_t) {
          uint32_t pa[4];
          pa[0] = pack_bf16x2(s[2 * blk][0], s[2 * blk][1]);
          pa[1] = pack_bf16x2(s[2 * blk][2], s[2 * blk][3]);
          pa[2] = pack_bf16x2(s[2 * blk + 1][0], s[2 * blk + 1][1]);
          pa[3] = pack_bf16x2(s[2 * blk + 1][2], s[2 * blk + 1][3]);
          const int key0 = kbase + blk * kBS;
          const int kqb = key0 + 2 * (lane & 3);
          const bool tail = key0 + kBS > n_keys;
#pragma unroll
          for (int nd = 0; nd < D / 16; ++nd) {
            const int ch = 2 * nd + csel;
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(vs + blk * TB + (ch >> 3) * 2048 + sw128_offset(vrow, ch & 7), r0, r1, r2, r3);
            if (tail) {
              r0 = mask_pair(r0, kqb, n_keys);
              r1 = mask_pair(r1, kqb + 8, n_keys);
              r2 = mask_pair(r2, kqb, n_keys);
              r3 = mask_pair(r3, kqb + 8, n_keys);
            }
            mma_bf16_16816(o[2 * nd], pa, r0, r1);
            mma_bf16_16816(o[2 * nd + 1], pa, r2, r3);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }
  if (!ok) {
    if (lane == 0) report_error(p.err, kErrTimeout, kWhereAttnPrefill);
    *abort_flag = 1;
    return;
  }
  l0 = quad_sum(l0);
  l1 = quad_sum(l1);
  const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int h = h_first + warp;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int col = n * 8 + 2 * (lane & 3);
    if (g < nrows)
      *reinterpret_cast<uint32_t*>(p.out + (static_cast<size_t>(tq + g) * p.nq + h) * D + col) =
          pack_bf16x2(o[n][0] * i0, o[n][1] * i0);
    if (g + 8 < nrows)
      *reinterpret_cast<uint32_t*>(p.out + (static_cast<size_t>(tq + g + 8) * p.nq + h) * D + col) =
          pack_bf16x2(o[n][2] * i1, o[n][3] * i1);
  }
}

// ---------------------------------------------------------------------------
// prefill on the 5th-generation tensor cores (head_dim 128, 128 % group == 0)
//
// One CTA per (sequence, KV head, 128/G query tokens): the 128 MMA rows are
// those tokens x the G q heads of the group (row r = token r/G, head r%G), so
// every K/V tile is read once per group.  Warp 0 streams Q (one 3-D TMA box per
// 64 columns) and the 64-key K tiles, warp 6 the 64-key V tiles (a 2-stage
// ring each, so the next K tile never waits behind a V stage that P V still
// holds); each reads a tile's block numbers before it waits for a free stage.
// One thread of warp 1 issues S = Q K^T into a double-buffered TMEM
// accumulator, one thread of warp 7 O += P V into a TMEM accumulator (V is the
// MN-major B operand): split over two threads, the next S is issued while the
// other thread waits for P, and neither waits behind the other's MMAs.  Warps
// 2-5 (one row each) read each S tile from TMEM once, write P as bf16 pairs
// back over the first half of that S buffer (tcgen05.st), and rescale O in
// TMEM only when a row's running max grows by more than 2^8.  P V takes its A
// operand from tensor memory, so the softmax of tile j+1 runs while P V of
// tile j is in the tensor pipe.  S buffer j%2 is next written by S of tile
// j+2, which waits for the buffer's P V-done barrier (committed after P V of
// tile j by the other thread).  Each S buffer has its own P-ready barrier, and
// O is read after the once-only drain barrier: the softmax warps may drift a
// tile apart, and a single P-ready barrier or a parity wait on the per-tile
// P V barrier would then mix up tiles.
// ---------------------------------------------------------------------------
constexpr int kTcThreads = 256;  // warp 0 Q + K loads, 1 S MMAs, 2-5 softmax, 6 V loads, 7 P V MMAs
constexpr int kTcKeys = 64;                        // keys per K/V tile (64 or 128; 128-key tiles with one S
                                                   // buffer and one-stage rings measured 2.23 vs 1.88 ms)
constexpr int kTcSBufs = 2;                        // S buffers in tensor memory (2, or 1 with 128-key tiles)
constexpr int kTcTileBytes = kTcKeys * 128 * 2;    // K or V tile: two 64-column halves
constexpr int kTcHalf = kTcKeys * 128;             // bytes of one 64-column half of K or V
constexpr int kTcQHalf = 128 * 128;                // bytes of one 64-column half of Q (16 KB)
constexpr int kTcSlack = 256;                      // alignment slack kept small so two CTAs share an SM
constexpr int kTcKStages = 2;                     // K ring (three stages measured slower: 1.796 vs 1.727 ms)
constexpr int kTcVStages = 2;                     // V ring
static_assert(kTcSBufs * kTcKeys + 128 <= 256, "S buffers and O must fit 256 tensor-memory columns");
static_assert(kTcKeys == 64 || kTcKeys == 128, "the softmax handles 64- or 128-key tiles");
constexpr int kTcSmem = 2 * kTcQHalf + (kTcKStages + kTcVStages) * kTcTileBytes + 256 + kTcSlack;
constexpr float kRescaleLog2 = 8.0f;               // lazy rescale threshold (factor 256)

__global__ void __launch_bounds__(kTcThreads, 2)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_wait();
  pdl_trigger();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad > kTcSlack) {  // the dynamic shared memory base is 1024-aligned in practice
    if (threadIdx.x == 0) report_error(p.err, kErrGuard, kWhereAttnPrefill);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t q_s = sb;                                   // Q: two 64-column halves
  auto k_s = [&](int st) { return sb + 2u * kTcQHalf + st * kTcTileBytes; };
  auto v_s = [&](int st) { return sb + 2u * kTcQHalf + (kTcKStages + st) * kTcTileBytes; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kTcQHalf + (kTcKStages + kTcVStages) * kTcTileBytes);
  const uint32_t bar0 = smem_u32(bars);
  // K and V have their own rings: a K stage is free as soon as its S = Q K^T
  // is done, so the next K tiles are fetched while P V still runs
  // P ready: one barrier per S buffer.  With one barrier for every tile a
  // softmax warp that finished tile j could run through tile j+1 (its S is
  // already there) and arrive again before a slower warp arrived for tile j,
  // completing tile j's phase while part of P(j) was still being written.  A
  // warp cannot reach tile j+2 before P V of tile j is issued, so the arrivals
  // at p_full0 + 8 * (j % 2) all belong to tile j.  (With one S buffer a warp
  // cannot reach tile j+1 before P V of tile j is issued either.)
  const uint32_t q_full = bar0, k_full0 = bar0 + 8, k_empty0 = k_full0 + 8 * kTcKStages,
                 v_full0 = k_empty0 + 8 * kTcKStages, v_empty0 = v_full0 + 8 * kTcVStages,
                 s_full0 = v_empty0 + 8 * kTcVStages, p_full0 = s_full0 + 8 * kTcSBufs,
                 o_done = p_full0 + 8 * kTcSBufs, drain = o_done + 8, pv_done0 = drain + 8,
                 s_drain = pv_done0 + 8 * kTcSBufs;
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(bars + 1 + 2 * kTcKStages + 2 * kTcVStages + 3 * kTcSBufs + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* p_hi_s = reinterpret_cast<int*>(tmem_slot + 2);
  int* p_lo_s = reinterpret_cast<int*>(tmem_slot + 3);

  const uint32_t item = p.pre_items[blockIdx.y];
  if (item == kNoItem) return;
  const int G = p.group, QT = 128 / G;
  const int b = static_cast<int>(item >> 16), qt = static_cast<int>(item & 0xFFFFu);
  const int kvh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = p.qsl[b];
  const int qlen = p.qsl[b + 1] - t0;
  if (qlen < 2 || qt * QT >= qlen) return;
  const int tq = t0 + qt * QT;
  const int nrows_tok = min(QT, qlen - qt * QT);

  if (threadIdx.x == 0) {
    *p_hi_s = -1;
    *p_lo_s = 0x7fffffff;
  }
  __syncthreads();
  if (threadIdx.x < nrows_tok) {
    const int ps = p.positions[tq + threadIdx.x];
    atomicMax(p_hi_s, ps);
    atomicMin(p_lo_s, ps);
  }
  __syncthreads();
  const int n_keys = *p_hi_s + 1;
  const int pos_lo = *p_lo_s;  // tiles ending at or below it need no causal mask
  if (n_keys > p.seq_lens[b] || (n_keys + kBS - 1) / kBS > p.max_blocks || n_keys < 1) {
    if (kvh == 0 && threadIdx.x == 0) report_error(p.err, kErrGuard, kWhereQueryLen);
    return;
  }
  const int nblk = (n_keys + kBS - 1) / kBS;
  const int ntiles = (n_keys + kTcKeys - 1) / kTcKeys;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kTcKStages; ++i) {
      mbar_init(k_full0 + 8 * i, 1);
      mbar_init(k_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < kTcVStages; ++i) {
      mbar_init(v_full0 + 8 * i, 1);
      mbar_init(v_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < kTcSBufs; ++i) {
      mbar_init(s_full0 + 8 * i, 1);
      mbar_init(p_full0 + 8 * i, 4);
    }
    for (int i = 0; i < kTcSBufs; ++i) mbar_init(pv_done0 + 8 * i, 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(s_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S buffers at columns 0 (and kTcKeys), O at kTcSBufs * kTcKeys
  constexpr int kOCol = kTcSBufs * kTcKeys;

  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers: Q and K (warp 0), V (warp 6) ----------------
    const bool is_k = warp == 0;
    if (lane == 0) {
      bool ok = true;
      uint32_t uses[kTcKStages > kTcVStages ? kTcKStages : kTcVStages] = {};
      const int nst = is_k ? kTcKStages : kTcVStages;
      const uint64_t pol = policy_evict_normal();
      if (is_k) {
        mbar_arrive_expect_tx(q_full, 32768);
        tma_load_3d(q_s, &tmQ, q_full, 0, kvh * G, tq, pol);
        tma_load_3d(q_s + kTcQHalf, &tmQ, q_full, 64, kvh * G, tq, pol);
      }
      const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks;
      const CUtensorMap* tm = is_k ? &tmK : &tmV;
      const uint32_t full0 = is_k ? k_full0 : v_full0, empty0 = is_k ? k_empty0 : v_empty0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % nst;
        // the tile's block numbers are read before the wait for a free stage
        // (blocks past the context load the first block again: finite data the
        // mask removes)
        int blks[kTcKeys / kBS];
#pragma unroll
        for (int i = 0; i < kTcKeys / kBS; ++i) {
          const int jb = j * (kTcKeys / kBS) + i;
          blks[i] = bt[jb < nblk ? jb : 0];
        }
        if (!mbar_wait(empty0 + 8 * st, ((j / nst) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t dst = is_k ? k_s(st) : v_s(st);
        const uint32_t bar = full0 + 8 * st;
        mbar_arrive_expect_tx(bar, kTcTileBytes);
#pragma unroll
        for (int i = 0; i < kTcKeys / kBS; ++i) {
          int blk = blks[i];
          if (blk < 0 || blk >= p.num_blocks) {
            report_error(p.err, kErrGuard, kWhereBlockTable);
            blk = 0;
          }
          const int row = (blk * p.nkv + kvh) * kBS;
          tma_load_2d(dst + i * 2048, tm, bar, 0, row, pol);
          tma_load_2d(dst + kTcHalf + i * 2048, tm, bar, 64, row, pol);
        }
        uses[st]++;
      }
      if (!ok) {
        report_error(p.err, kErrTimeout, kWhereAttnPrefill);
        *abort_flag = 1;
      }
      // every load this thread issued lands before the CTA can exit
      if (is_k) mbar_wait(q_full, 0, nullptr);
      for (int st = 0; st < nst; ++st)
        if (uses[st] > 0) mbar_wait(full0 + 8 * st, (uses[st] - 1) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 7) {
    // ---------------- MMA issuers: S = Q K^T (warp 1), O += P V (warp 7) ----------------
    constexpr uint32_t idS = idesc_bf16_f32(128, kTcKeys);
    constexpr uint32_t idPV = idesc_bf16_f32_bmn(128, 128);
    // Operand descriptors, built once: only the start-address field (address
    // / 16, bits 0-13; every shared address here is below 2^18) moves from one
    // MMA to the next, so each MMA adds a constant to a precomputed low word.
    const uint64_t sw0 = smem_desc_sw128(0), vd0 = smem_desc_sw128_lbo_sbo(0, kTcHalf, 1024);
    const uint32_t sw_hi = static_cast<uint32_t>(sw0 >> 32), v_hi = static_cast<uint32_t>(vd0 >> 32);
    const uint32_t sw_lo = static_cast<uint32_t>(sw0), v_lo = static_cast<uint32_t>(vd0);
    auto desc = [](uint32_t lo, uint32_t hi) { return (static_cast<uint64_t>(hi) << 32) | lo; };
    bool ok = true, issued = false;
    if (warp == 1) {
      // S(j) overwrites the buffer P(j - 2) was written to: it waits until
      // P V(j - 2), issued by the other warp, has completed.  (Each issuer
      // first waits for its operand tile, which has usually landed long
      // before, so the wait that ends last is the one nearest the MMAs.)
      const uint32_t q_lo = sw_lo + (q_s >> 4);
      const uint32_t k_lo0 = sw_lo + (k_s(0) >> 4);  // stage st lies st * kTcTileBytes further on
      ok = mbar_wait(q_full, 0, abort_flag);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int st = j % kTcSBufs, kst = j % kTcKStages;
        if (!mbar_wait(k_full0 + 8 * kst, (j / kTcKStages) & 1, abort_flag) ||
            (j >= kTcSBufs && !mbar_wait(pv_done0 + 8 * st, ((j - kTcSBufs) / kTcSBufs) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t d = tmem + st * kTcKeys;
          const uint32_t kb = k_lo0 + kst * (kTcTileBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t cq = (kk >> 2) * kTcQHalf + (kk & 3) * 32;
            const uint32_t ck = (kk >> 2) * kTcHalf + (kk & 3) * 32;
            tc_mma_f16(d, desc(q_lo + (cq >> 4), sw_hi), desc(kb + (ck >> 4), sw_hi), idS, kk > 0 ? 1u : 0u);
          }
          tc_commit(s_full0 + 8 * st);
          tc_commit(k_empty0 + 8 * kst);
          issued = true;
        }
        __syncwarp();
      }
    } else {
      const uint32_t v_lo0 = v_lo + (v_s(0) >> 4);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int sbuf = j % kTcSBufs, vst = j % kTcVStages;
        if (!mbar_wait(v_full0 + 8 * vst, (j / kTcVStages) & 1, abort_flag) ||
            !mbar_wait(p_full0 + 8 * sbuf, (j / kTcSBufs) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vb = v_lo0 + vst * (kTcTileBytes >> 4);
          const uint32_t pa = tmem + sbuf * kTcKeys;
#pragma unroll
          for (int ks = 0; ks < kTcKeys / 16; ++ks) {  // P: 16 keys = 8 packed columns per step
            tc_mma_f16_ts(tmem + kOCol, pa + ks * 8, desc(vb + ks * (2048 >> 4), v_hi), idPV,
                          (j > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(v_empty0 + 8 * vst);
          tc_commit(o_done);
          tc_commit(pv_done0 + 8 * sbuf);
          issued = true;
        }
        __syncwarp();
      }
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereAttnPrefill);
      *abort_flag = 1;
    }
    // each issuer waits for its own MMAs before the CTA frees tensor memory;
    // the P V issuer's drain also tells the softmax warps that O is final
    const uint32_t fin = warp == 1 ? s_drain : drain;
    if (lane == 0 && issued) tc_commit(fin);
    __syncwarp();
    if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) mbar_wait(fin, 0, nullptr);
  } else {
    // ---------------- softmax warps (2-5): one row each ----------------
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int tok = r / G, hq = r % G;
    const bool row_ok = tok < nrows_tok;
    const int pos = row_ok ? p.positions[tq + tok] : -1;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kTcSBufs;
      if (!mbar_wait(s_full0 + 8 * st, (j / kTcSBufs) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S of this tile: masked, scaled row maximum (four independent max
      // chains; eight and sixteen measured no faster), 64 columns per load;
      // t keeps the last 64 columns read
      const int kbase = j * kTcKeys;
      const bool full_tile = kbase + kTcKeys - 1 <= pos_lo;  // CTA-uniform
      const int lim = pos - kbase;                           // column e is visible when e <= lim
      const uint32_t s_addr = lane_addr + st * kTcKeys;
      float t[64];
      float mx8[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx8[i] = -INFINITY;
#pragma unroll
      for (int h = 0; h < kTcKeys / 64; ++h) {
        tmem_ld64(s_addr + h * 64, t);
        if (full_tile) {  // the softmax warps are issue-bound: two scores per max instruction
#pragma unroll
          for (int c2 = 0; c2 < 32; ++c2) mx8[c2 & 3] = fmax3(mx8[c2 & 3], t[2 * c2], t[2 * c2 + 1]);
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (h * 64 + e <= lim) mx8[e & 3] = fmaxf(mx8[e & 3], t[e]);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = fmaxf(mx, mx8[i]);
      mx = mx == -INFINITY ? -INFINITY : mx * p.scale_log2;
      const float m_new = fmaxf(m_run, mx);
      // Rescale (rare): only when some row of the warp gains more than 2^8.
      const bool need = j > 0 && m_new > m_run + kRescaleLog2;
      const bool warp_rescale = __any_sync(0xffffffffu, need);
      if (j == 0) m_run = m_new;
      if (warp_rescale) {
        // P V of the previous tile must be done before O is rescaled (P V of
        // the tile before it is: S of this tile was issued after it)
        if (!mbar_wait(o_done, (j - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(lane_addr + kOCol + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(lane_addr + kOCol + c * 32, o);
        }
        l *= alpha;
        m_run = m_new;
      }
      const float base = m_run == -INFINITY ? 0.f : m_run;
      // P = exp2(S - max) as bf16 pairs, 32 scores at a time: packed column c
      // holds keys 2c and 2c + 1, written over S column c.  Scale-and-shift and
      // the row sum run as paired fp32 operations.
      uint64_t ls2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) ls2[i] = f2_pack(0.f, 0.f);
      const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
      const uint64_t nbase2 = f2_pack(-base, -base);
      auto emit32 = [&](const float* v, int c0, float* pw, auto masked) {
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          const int e = 2 * c2;
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(v[e], v[e + 1]), scale2, nbase2), a0, a1);
          float x0 = fast_exp2(a0);
          float x1 = fast_exp2(a1);
          if (decltype(masked)::value) {
            x0 = c0 + e <= lim ? x0 : 0.f;
            x1 = c0 + e + 1 <= lim ? x1 : 0.f;
          }
          ls2[c2 & 3] = f2_add(ls2[c2 & 3], f2_pack(x0, x1));
          pw[c2] = __uint_as_float(pack_bf16x2(x0, x1));
        }
      };
      auto emit_tile = [&](auto masked) {
        if constexpr (kTcKeys == 64) {
          float pw[32];
          emit32(t, 0, pw, masked);
          emit32(t + 32, 32, pw + 16, masked);
          tmem_st32(s_addr, pw);
        } else {
          // columns 0-63 are read again (t holds 64-127); chunk q's weights
          // go to columns 16q..16q+15, all of them read by then
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {
            float u[32], pw[16];
            tmem_ld32(s_addr + q * 32, u);
            emit32(u, q * 32, pw, masked);
            tmem_st16(s_addr + q * 16, pw);
          }
#pragma unroll
          for (int q = 2; q < 4; ++q) {
            float pw[16];
            emit32(t + (q - 2) * 32, q * 32, pw, masked);
            tmem_st16(s_addr + q * 16, pw);
          }
        }
      };
      if (full_tile)
        emit_tile(std::false_type{});
      else
        emit_tile(std::true_type{});
      {
        float s[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(ls2[i], s[2 * i], s[2 * i + 1]);
        l += ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
      }
      // keys past the context inside the last loaded block: zero their V rows
      // (P is zero there, but stale cache contents must not reach the MMA),
      // once the tile's V load has landed
      if (j == ntiles - 1) {
        const int vst = j % kTcVStages;
        if (!mbar_wait(v_full0 + 8 * vst, (j / kTcVStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int valid = n_keys - kbase;
        uint8_t* vg = smem + (v_s(vst) - sb);
        for (int i = threadIdx.x - 64; i < (kTcKeys - valid) * 2 * 8; i += 128) {
          const int rowv = valid + i / 16, hf = (i / 8) & 1, c16 = i & 7;
          *reinterpret_cast<uint4*>(vg + hf * kTcHalf + rowv * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full0 + 8 * st);
    }
    // every MMA of the CTA has completed before O is read: the drain barrier,
    // committed once after the last P V, completes exactly once.  (o_done,
    // committed after every P V and waited on by parity, cannot say so: a warp
    // that finished the last tile may find P V of the tile before it still
    // pending, a phase whose parity differs from the last one's.)
    if (ok && !mbar_wait(drain, 0, abort_flag)) ok = false;
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereAttnPrefill);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = p.out + (static_cast<size_t>(tq + tok) * p.nq + kvh * G + hq) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(lane_addr + kOCol + c * 32, o);
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv;
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_bf16x2(o[8 * q + 0], o[8 * q + 1]);
            u.y = pack_bf16x2(o[8 * q + 2], o[8 * q + 3]);
            u.z = pack_bf16x2(o[8 * q + 4], o[8 * q + 5]);
            u.w = pack_bf16x2(o[8 * q + 6], o[8 * q + 7]);
            d4[q] = u;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// cache [num_blocks * nkv * 16 rows, D] with a 16 x 64 box, 128-byte swizzle
bool make_cache_tmap(CUtensorMap* m, const void* base, long long rows, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBS)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [T, nq, 128] as a 3-D tensor (d, head, token) with a box of 64 columns x
// `group` heads x `tokens` tokens: one box is 128 rows of the prefill tile
bool make_q_tmap(CUtensorMap* m, const void* base, int T, int nq, int group, int tokens) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(nq), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(nq) * 128 * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tokens)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
size_t decode_smem() {
  return 1024 + kDecWarps * kDecStages * 2 * tile_bytes(D) + 16 * (D + 8) * 2 + 8 * kDecWarps * kDecStages;
}

template <int D>
size_t prefill_smem() {
  return 1024 + kPreStages * 2 * 4 * tile_bytes(D) + kPreMaxHeads * 16 * (D + 8) * 2 + 8 * 2 * kPreStages + 16;
}

template <int D>
int launch_prefill_d(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, bool tc,
                     int tile_tokens, int items, bool pdl, cudaStream_t s);

// One non-blocking stream per device, created on first use and kept for the
// life of the process.
cudaStream_t side_stream() {
  constexpr int kDevs = 64;
  static cudaStream_t st[kDevs] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (st[dev] == nullptr && cudaStreamCreateWithFlags(&st[dev], cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    st[dev] = nullptr;
  }
  return st[dev];
}

// The fork and join events of the current host thread on the current device,
// created on first use and reused by every later call of that thread (a
// stream wait takes the event's state when it is enqueued, so re-recording
// afterwards does not disturb it).  Creating them outside any stream capture
// (the first call of a thread is eager) keeps the call capture-safe.
bool fork_join_events(cudaEvent_t* fork, cudaEvent_t* join) {
  constexpr int kDevs = 64;
  thread_local cudaEvent_t ev[kDevs][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return false;
  for (int i = 0; i < 2; ++i) {
    if (ev[dev][i] == nullptr && cudaEventCreateWithFlags(&ev[dev][i], cudaEventDisableTiming) != cudaSuccess) {
      ev[dev][i] = nullptr;
      cudaGetLastError();
      return false;
    }
  }
  *fork = ev[dev][0];
  *join = ev[dev][1];
  return true;
}

template <int D>
int launch_d(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, AttnParams& p, cudaStream_t s,
             bool* joined) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(k_attn_decode<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(decode_smem<D>()));
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(k_attn_prefill<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(prefill_smem<D>()));
  });
  if (attr != cudaSuccess) return attr;
  const int max_blk = (a.max_seq_len + kBS - 1) / kBS;
  p.max_chunks = num_chunks(max_blk);
  if (p.max_chunks < 1) p.max_chunks = 1;
  const bool tc = a.max_query_len >= 2 && D == 128 && 128 % p.group == 0;
  const int tile_tokens = tc ? 128 / p.group : 16;  // tensor-core prefill: 128 rows = tokens x group heads
  const int items = (a.T + tile_tokens - 1) / tile_tokens + a.B;
  // With prefill sequences in the batch, the decode kernels (HBM-bound) run on
  // the library's side stream beside the prefill kernel (tensor-bound): the
  // caller's stream forks to it after the previous kernel and joins it before
  // the next.  Otherwise everything runs in order on the caller's stream.
  cudaStream_t sd = s;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  if (a.max_query_len >= 2 && a.overlap) {
    cudaStream_t side = side_stream();
    if (side != nullptr && fork_join_events(&ev_fork, &ev_join) && cudaEventRecord(ev_fork, s) == cudaSuccess &&
        cudaStreamWaitEvent(side, ev_fork, 0) == cudaSuccess) {
      sd = side;
    } else {
      cudaGetLastError();
    }
  }
  const bool forked = sd != s;
  if (joined) *joined = forked;
  // the first kernel on each stream takes the caller's dependency mode (none
  // after a fork), the ones after it overlap their predecessor
  bool pdl_s = a.pdl != 0, pdl_d = forked ? false : a.pdl != 0;
  cudaError_t e = cudaSuccess;
  if (a.max_query_len >= 2) {
    e = launch_kernel(k_attn_plan, dim3(1), dim3(1024), 0, s, pdl_s, a.qsl, a.B, tile_tokens, p.pre_items, items);
    pdl_s = true;
    if (!forked) pdl_d = true;
  }
  if (e == cudaSuccess) {
    dim3 gd(a.B * a.nkv, p.max_chunks, 1);  // chunk-major: every sequence's first chunk first
    e = launch_kernel(k_attn_decode<D>, gd, dim3(kDecWarps * 32), decode_smem<D>(), sd, pdl_d, tk, tv, p);
    if (e == cudaSuccess && p.max_chunks > 1) {
      constexpr int heads_per_cta = kCombineThreads / (D / 4);
      e = launch_kernel(k_attn_combine<D>, dim3((a.nq + heads_per_cta - 1) / heads_per_cta, a.B),
                        dim3(kCombineThreads), 0, sd, true, p);
    }
    if (!forked) pdl_s = true;
  }
  if (e == cudaSuccess && a.max_query_len >= 2)
    e = static_cast<cudaError_t>(launch_prefill_d<D>(a, tk, tv, p, tc, tile_tokens, items, pdl_s, s));
  if (forked) {  // join even after a failed launch, so the caller's stream never runs ahead of the side stream
    const cudaError_t j1 = cudaEventRecord(ev_join, sd);
    const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(s, ev_join, 0) : j1;
    if (e == cudaSuccess) e = j2;
  }
  return e;
}

template <int D>
int launch_prefill_d(const AttnArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, bool tc,
                     int tile_tokens, int items, bool pdl, cudaStream_t s) {
  if (tc) {
    static std::once_flag tc_once;
    static cudaError_t tc_attr = cudaSuccess;
    std::call_once(tc_once, [] {
      tc_attr = cudaFuncSetAttribute(k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    });
    if (tc_attr != cudaSuccess) return tc_attr;
    CUtensorMap tq;
    if (!make_q_tmap(&tq, a.q, a.T, a.nq, p.group, tile_tokens)) return cudaErrorInvalidValue;
    return launch_kernel(k_attn_prefill_tc, dim3(a.nkv, items), dim3(kTcThreads), kTcSmem, s, pdl, tq, tk,
                         tv, p);
  }
  const int n_hc = (p.group + kPreMaxHeads - 1) / kPreMaxHeads;
  const int warps = (p.group < kPreMaxHeads ? p.group : kPreMaxHeads) + 1;
  return launch_kernel(k_attn_prefill<D>, dim3(a.nkv * n_hc, items), dim3(warps * 32), prefill_smem<D>(), s,
                       pdl, tk, tv, p);
}

}  // namespace

size_t attn_partials_bytes(int B, int T, int max_seq_len, int nq, int head_dim) {
  const int nch = num_chunks((max_seq_len + kBS - 1) / kBS);
  const size_t n = static_cast<size_t>(B) * (nch < 1 ? 1 : nch) * nq;
  return n * head_dim * sizeof(float) + n * sizeof(float2) +
         static_cast<size_t>(max_prefill_items(T, B)) * sizeof(uint32_t) + 256;
}

int attention_launch(const AttnArgs& a, cudaStream_t s, bool* joined) {
  if (joined) *joined = false;
  if (a.T <= 0 || a.B <= 0) return 0;
  const long long rows = static_cast<long long>(a.num_blocks) * a.nkv * kBS;
  CUtensorMap tk, tv;
  if (!make_cache_tmap(&tk, a.k_cache, rows, a.head_dim)) return cudaErrorInvalidValue;
  if (!make_cache_tmap(&tv, a.v_cache, rows, a.head_dim)) return cudaErrorInvalidValue;
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.qsl = a.qsl;
  p.seq_lens = a.seq_lens;
  p.positions = a.positions;
  p.block_table = a.block_table;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.nq = a.nq;
  p.nkv = a.nkv;
  p.group = a.nq / a.nkv;
  p.scale_log2 = kLog2e / sqrtf(static_cast<float>(a.head_dim));
  p.err = a.err;
  const int max_blk = (a.max_seq_len + kBS - 1) / kBS;
  const size_t n = static_cast<size_t>(a.B) * (num_chunks(max_blk) < 1 ? 1 : num_chunks(max_blk)) * a.nq;
  if (attn_partials_bytes(a.B, a.T, a.max_seq_len, a.nq, a.head_dim) > a.partials_bytes) return cudaErrorInvalidValue;
  if (a.B > 65535 || max_prefill_items(a.T, a.B) > 65535) return cudaErrorInvalidValue;  // item packing, grid y
  p.part_o = a.partials;
  p.part_ml = reinterpret_cast<float2*>(a.partials + n * a.head_dim);
  p.pre_items = reinterpret_cast<uint32_t*>(p.part_ml + n);
  if (a.head_dim == 128) return launch_d<128>(a, tk, tv, p, s, joined);
  if (a.head_dim == 64) return launch_d<64>(a, tk, tv, p, s, joined);
  return cudaErrorInvalidValue;
}

}  // namespace llama
