// Tensor-core GEMM y = x * W^T for the four projections (and lm_head), on the
// 5th-generation tensor cores: TMA loads 128-byte-swizzled K-major tiles into
// a shared-memory ring, one thread issues tcgen05.mma (M=128, N=256 or 192, K=16)
// into an fp32 accumulator in tensor memory, and four epilogue warps drain it
// with tcgen05.ld and apply the fused epilogue:
//   * plain bf16 store                         (o_proj, down_proj)
//   * RoPE on q/k + q store + paged K/V scatter (qkv_proj; the cache update
//     precedes attention, as LlamaAttention.forward does)
//   * SiluAndMul: silu(x[:d]) * x[d:]          (gate_up_proj; a tile loads 128
//     gate rows and the matching 128 up rows, so both halves meet in one
//     thread)
//   * fp32 store                               (lm_head logits)
// Every tensor a module of the layer returns is bf16 (the model's dtype), so
// the fused epilogues round the projection output to bf16 before RoPE and
// before SiluAndMul, exactly where the unfused modules would store it.
//
// Three schedules, by the number of output tiles against the SM count:
//   * at least one wave of tiles (prefill): k_gemm_tc, persistent (one CTA
//     per SM), whole tiles in a grouped raster for L2 reuse, the accumulator
//     double-buffered so the epilogue of one tile overlaps the MMAs of the
//     next;
//   * at most half as many tiles as SMs (decode qkv, o_proj, down_proj):
//     k_gemm_cluster, split-K over a thread-block cluster whose CTAs hand
//     their fp32 slices to each other through distributed shared memory;
//   * in between, below one wave of tiles: k_gemm_tc stream-K, every CTA an
//     equal share of (tile, k-block) units, partial tiles in a workspace, and
//     k_gemm_fixup summing them in CTA order (deterministic) spread over many
//     CTAs.
// SwiGLU over one row block (the decode gate_up) uses 192-column tiles when
// they fill the waves better than 256-column ones (k_gemm_tc<SwiGLU, 192>).
// The operand ring holds as many stages as fit: a 64-row A box when M <= 64
// and narrow tiles make each stage smaller and the ring deeper.
// Grouped mode (the experts of an MoE block): k_gemm_tc walks a tile list
// built on the device, each entry naming its A rows, its expert's B rows and
// how many of its rows are valid.  A row scale (an RMSNorm's rsqrt, its
// weights folded into B) may multiply the product before any epilogue.
// The kernels wait for the previous kernel of the call (pdl_wait) only where
// they first need its results; the weight tiles of their first stages are
// requested before that.
//
// Sources: [WALKTHROUGH] "模型库与算子层 — 代码走读", Linear layers (F.linear with
// Parameter(out, in)); [LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B", §4
// LlamaAttention and LlamaMLP (merged qkv / gate_up projections, SiluAndMul);
// [CODE-READING] "vLLM Llama 代码解析", §4 (RoPE on q and k only).
#include <cuda.h>
#include <math.h>

#include <cmath>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace llama {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;  // accumulator columns per tile
constexpr int kNarrowBN = 192;  // SwiGLU tiles of decode-sized M (96 gate + 96 up columns)
constexpr int BK = 64;   // one 128-byte swizzle row of bf16
constexpr int kMaxStages = 8;  // operand stages: as many as fit (4 of 48 KB for 256-column tiles and 128-row A boxes)
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int NUM_THREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
// k_gemm_cluster: warp 0 TMA, warp 1 MMA, warps 2-7 wait for the accumulator;
// then all eight move it, two warps per tensor-memory lane quarter
constexpr int kClusterThreads = 256;
constexpr int TMEM_COLS = 2 * BN;
constexpr int kMaxSmemBytes = 232448;              // the opt-in limit per CTA (227 KB)
constexpr int kRingBudget = kMaxSmemBytes - 2048;  // the ring; the rest: barriers, rope table, alignment slack

struct GemmParams {
  int M, N, K;
  int tiles_m, tiles_n, kb, tiles;
  int sk, grid, group_m;
  long long units;
  int b_row_step;    // row offset of the second 128-row B box (128, or I for SwiGLU)
  int b_tile_rows;   // B rows advanced per output tile (256, or 128 for SwiGLU)
  int b_evict_first;
  // operand ring: stages of stage_bytes, the A box (a_rows rows: 128, or 64
  // when M <= 64, the MMA then reading B bytes as rows 64-127 of A, whose
  // accumulator rows are never stored) first in each stage
  int stages, stage_bytes, a_rows;
  void* out;
  int ldo, n_out;
  float* partials;
  int* err;
  QkvEpilogueArgs qkv;
  float2 rope_tab[64];  // qkv epilogue: per rotated pair, revolutions per position as (hi, lo)
  // grouped mode (the experts of an MoE block): tiles come from a list built on
  // the device, {A row, B base row of the tile's expert, N tile, valid rows}
  const int4* group_tiles;
  const int* group_count;
  // per-row scale of the product before the epilogue (an RMSNorm's rsqrt
  // with its weights folded into B), or null
  const float* row_scale;
};

struct Work {
  int tile, kb0, kb1;
  int4 desc;  // grouped mode: the tile's list entry
};

// Grouped mode: the tile count is read once and every list entry one tile
// ahead of its use, so no role waits on a global load at a tile boundary.
struct Feed {
  long long count;
  int4 next;
};

__device__ __forceinline__ Feed feed_init(const GemmParams& p, long long cursor) {
  Feed f{0, make_int4(0, 0, 0, 0)};
  if (p.group_tiles != nullptr) {
    f.count = *p.group_count;
    if (cursor < f.count) f.next = p.group_tiles[cursor];
  }
  return f;
}

// A row, B rows, output tile coordinates and the row bound of a work item
struct TileCoords {
  int tm, tn, arow, brow0, m_limit;
};

__device__ __forceinline__ bool next_work(const GemmParams& p, long long& cursor, long long end, Work& w,
                                          Feed& feed) {
  if (p.sk) {
    if (cursor >= end) return false;
    w.tile = static_cast<int>(cursor / p.kb);
    w.kb0 = static_cast<int>(cursor % p.kb);
    long long tile_end = static_cast<long long>(w.tile + 1) * p.kb;
    long long e = end < tile_end ? end : tile_end;
    w.kb1 = w.kb0 + static_cast<int>(e - cursor);
    cursor = e;
    return true;
  }
  const bool grouped = p.group_tiles != nullptr;
  if (cursor >= (grouped ? feed.count : p.tiles)) return false;
  w.tile = static_cast<int>(cursor);
  w.kb0 = 0;
  w.kb1 = p.kb;
  cursor += p.grid;
  if (grouped) {
    w.desc = feed.next;
    if (cursor < feed.count) feed.next = p.group_tiles[cursor];
  }
  return true;
}

__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& tm, int& tn) {
  const int group = p.group_m * p.tiles_n;
  const int g = tile / group;
  const int first_m = g * p.group_m;
  int gm = p.tiles_m - first_m;
  if (gm > p.group_m) gm = p.group_m;
  const int r = tile - g * group;
  tm = first_m + r % gm;
  tn = r / gm;
}

__device__ __forceinline__ TileCoords resolve_tile(const GemmParams& p, const Work& w) {
  TileCoords c;
  if (p.group_tiles != nullptr) {
    const int4 t = w.desc;
    c.tm = t.x / BM;
    c.tn = t.z;
    c.arow = t.x;
    c.brow0 = t.y + t.z * p.b_tile_rows;
    c.m_limit = t.x + t.w;
  } else {
    tile_coords(p, w.tile, c.tm, c.tn);
    c.arow = c.tm * BM;
    c.brow0 = c.tn * p.b_tile_rows;
    c.m_limit = p.M;
  }
  return c;
}

__host__ __device__ __forceinline__ long long sk_start(long long units, int grid, int c) {
  return units * c / grid;
}

// the CTA whose stream-K range holds unit u
__device__ __forceinline__ int sk_owner(const GemmParams& p, long long u) {
  int c = static_cast<int>((u * p.grid) / p.units);
  while (c + 1 < p.grid && sk_start(p.units, p.grid, c + 1) <= u) ++c;
  while (c > 0 && sk_start(p.units, p.grid, c) > u) --c;
  return c;
}

// ---------------------------------------------------------------------------
// RoPE frequency table: per pair i, the rotation rate in revolutions per
// position, r_i = inv_freq'_i / (2 pi), split into a float pair (hi, lo) so
// that the angle of a large position can be reduced exactly.
// inv_freq_i = theta^(-2i/d); llama3: wavelengths shorter than
// orig/high_freq_factor keep their frequency, longer than orig/low_freq_factor
// are divided by factor, in between they blend linearly in orig/wavelength.
// ---------------------------------------------------------------------------
// Computed once per launch on the host, in double precision (the device's
// FP64 rate is low and the fixup kernel would pay for it on its critical path).
void rope_table_host(const RopeParams& rp, int head_dim, float2* tab) {
  const int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    double inv = std::pow(static_cast<double>(rp.theta), -2.0 * i / head_dim);
    if (rp.llama3) {
      const double two_pi = 6.283185307179586476925287;
      const double lam = two_pi / inv;
      const double orig = static_cast<double>(rp.original_max_pos);
      const double lo = rp.low_freq_factor, hi = rp.high_freq_factor, f = rp.factor;
      if (lam < orig / hi) {
      } else if (lam > orig / lo) {
        inv = inv / f;
      } else {
        const double s = (orig / lam - lo) / (hi - lo);
        inv = (1.0 - s) * inv / f + s * inv;
      }
    }
    const double r = inv * 0.15915494309189533576888;  // 1 / (2 pi)
    const float rh = static_cast<float>(r);
    const float rl = static_cast<float>(r - static_cast<double>(rh));
    tab[i] = make_float2(rh, rl);
  }
}

__device__ __forceinline__ void copy_rope_table(const GemmParams& p, float2* tab, int tid, int nthreads) {
  for (int i = tid; i < p.qkv.head_dim / 2; i += nthreads) tab[i] = p.rope_tab[i];
}

// sin/cos of 2*pi*pos*r with r = (hi + lo): the product pos*hi is split into
// its rounded value and exact error, the integer revolutions are dropped and
// the remaining fraction goes to sincospif.
__device__ __forceinline__ void rope_sincos(int pos, float2 r, float& s, float& c) {
  const float fp = static_cast<float>(pos);
  const float ph = fp * r.x;
  const float pe = fmaf(fp, r.x, -ph);
  const float fr = ph - floorf(ph);
  const float t = fr + (pe + fp * r.y);
  sincospif(2.0f * t, &s, &c);
}

__device__ __forceinline__ void store_bf16x32(void* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d[q] = u;
  }
}

// ---------------------------------------------------------------------------
// Epilogue.  A tile's accumulator row is split into column units that can be
// finished independently: 8 chunks of 32 columns (bf16/f32 stores), 4 chunks
// of 32 SwiGLU outputs (each reads gate columns c.. and up columns 128+c..), or
// 4 (head, 32-pair chunk) units of the qkv tile.  `ld(col, v)` returns
// accumulator columns [col, col+32) of the thread's row; the TMEM loader is
// warp-collective, so every call is made under tile-uniform control.
// ---------------------------------------------------------------------------
template <int EPI>
struct EpiUnits {
  static constexpr int kUnits = (EPI == kEpiBf16 || EPI == kEpiF32) ? 8 : 4;
};

__device__ __forceinline__ void store_chunk(const GemmParams& p, int row, int n, const float (&v)[32], bool f32out) {
  if (f32out) {
    float* o = reinterpret_cast<float*>(p.out) + static_cast<size_t>(row) * p.ldo + n;
    if (n + 32 <= p.n_out) {
      float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int q = 0; q < 8; ++q) o4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
      for (int e = 0; e < 32 && n + e < p.n_out; ++e) o[e] = v[e];
    }
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * p.ldo + n;
    if (n + 32 <= p.n_out) {
      store_bf16x32(o, v);
    } else {
      for (int e = 0; e < 32 && n + e < p.n_out; ++e) o[e] = __float2bfloat16_rn(v[e]);
    }
  }
}

// Where this row's k/v go in the paged cache (slot < 0: nowhere).
struct QkvRow {
  int pos, slot, blk, off;
};

__device__ __forceinline__ QkvRow qkv_row(const GemmParams& p, int row, bool valid) {
  const QkvEpilogueArgs& q = p.qkv;
  QkvRow r;
  r.pos = valid ? q.positions[row] : 0;
  r.slot = valid ? q.slots[row] : -1;
  if (r.slot >= q.num_blocks * q.block_size) {
    report_error(p.err, kErrGuard, kWhereSlot);
    r.slot = -1;
  }
  r.blk = r.slot >= 0 ? r.slot / q.block_size : 0;
  r.off = r.slot >= 0 ? r.slot % q.block_size : 0;
  return r;
}

// RoPE on pairs (j+e, half+j+e) of the head starting at global column col,
// then the store: q to the q buffer, k to the cache.  qkv_proj's output is a
// bf16 tensor that rotary_emb then reads, hence the rounding first.
__device__ __forceinline__ void qkv_rotate_store(const GemmParams& p, int row, const QkvRow& r, int col, int j,
                                                 float (&lo)[32], float (&hi)[32], const float (&sn)[32],
                                                 const float (&cs)[32]) {
  const QkvEpilogueArgs& q = p.qkv;
  const int d = q.head_dim, half = d >> 1;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float x1 = round_bf16(lo[e]), x2 = round_bf16(hi[e]);
    lo[e] = x1 * cs[e] - x2 * sn[e];
    hi[e] = x2 * cs[e] + x1 * sn[e];
  }
  if (col < q.q_size) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * p.ldo + col + j;
    store_bf16x32(o, lo);
    store_bf16x32(o + half, hi);
  } else if (r.slot >= 0) {
    const int kh = (col - q.q_size) / d;
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(q.k_cache) +
                       ((static_cast<size_t>(r.blk) * q.n_kv_heads + kh) * q.block_size + r.off) * d + j;
    store_bf16x32(o, lo);
    store_bf16x32(o + half, hi);
  }
}

__device__ __forceinline__ void qkv_v_store(const GemmParams& p, const QkvRow& r, int col, int j,
                                            const float (&v)[32]) {
  const QkvEpilogueArgs& q = p.qkv;
  if (r.slot < 0) return;
  const int vh = (col - q.q_size - q.kv_size) / q.head_dim;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(q.v_cache) +
                     ((static_cast<size_t>(r.blk) * q.n_kv_heads + vh) * q.block_size + r.off) * q.head_dim + j;
  store_bf16x32(o, v);
}

// SiluAndMul on 32 outputs: gate_up_proj's output is a bf16 tensor that
// SiluAndMul then reads, hence the rounding of both halves first.
__device__ __forceinline__ void swiglu32(float (&g)[32], const float (&u)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float gv = round_bf16(g[e]);
    const float sg = gv / (1.0f + __expf(-gv));
    g[e] = sg * round_bf16(u[e]);
  }
}

// One column unit of one row (used by the stream-K fixup, where every thread
// owns a (row, unit) pair).
template <int EPI, class Loader>
__device__ __forceinline__ void epilogue_unit(const GemmParams& p, int tm, int tn, int row_in_tile, int unit,
                                              Loader& ld, const float2* rope_tab) {
  const int row = tm * BM + row_in_tile;
  if (row >= p.M) return;
  if constexpr (EPI == kEpiBf16 || EPI == kEpiF32) {
    const int c = unit * 32;
    const int n = tn * BN + c;
    if (n >= p.n_out) return;
    float v[32];
    ld(c, v);
    store_chunk(p, row, n, v, EPI == kEpiF32);
  } else if constexpr (EPI == kEpiSwiGlu) {
    const int c = unit * 32;
    const int n = tn * (BN / 2) + c;
    if (n >= p.n_out) return;
    float g[32], u[32];
    ld(c, g);
    ld(BN / 2 + c, u);
    swiglu32(g, u);
    store_chunk(p, row, n, g, false);
  } else {
    const QkvEpilogueArgs& q = p.qkv;
    const int d = q.head_dim, half = d >> 1;
    const int per_head = half / 32;  // 32-pair chunks per head
    const int hc = (unit / per_head) * d;
    const int j = (unit % per_head) * 32;
    const int col = tn * BN + hc;
    if (col >= p.N) return;
    const QkvRow r = qkv_row(p, row, true);
    float lo[32], hi[32];
    ld(hc + j, lo);
    ld(hc + half + j, hi);
    if (col < q.q_size + q.kv_size) {
      float sn[32], cs[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) rope_sincos(r.pos, rope_tab[j + e], sn[e], cs[e]);
      qkv_rotate_store(p, row, r, col, j, lo, hi, sn, cs);
    } else {
      qkv_v_store(p, r, col, j, lo);
      qkv_v_store(p, r, col, half + j, hi);
    }
  }
}

// The whole tile for one row (one thread per row, the GEMM kernel's epilogue
// warps).  For qkv the j-chunks are the outer loop so sin/cos are shared by
// the heads of the tile.
template <int EPI, int NB = BN, class Loader>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, int tm, int tn, int row_in_tile, Loader& ld,
                                              const float2* rope_tab, int m_limit) {
  static_assert(NB == BN || EPI == kEpiSwiGlu, "narrow tiles are SwiGLU tiles");
  const int row = tm * BM + row_in_tile;
  const bool valid = row < m_limit;
  if constexpr (EPI == kEpiBf16 || EPI == kEpiF32) {
    const int n_base = tn * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n_base + c >= p.n_out) break;  // tile-uniform
      float v[32];
      ld(c, v);
      if (valid) store_chunk(p, row, n_base + c, v, EPI == kEpiF32);
    }
  } else if constexpr (EPI == kEpiSwiGlu) {
    const int n_base = tn * (NB / 2);
#pragma unroll 1
    for (int c = 0; c < NB / 2; c += 32) {
      if (n_base + c >= p.n_out) break;
      float g[32], u[32];
      ld(c, g);
      ld(NB / 2 + c, u);
      if (!valid) continue;
      swiglu32(g, u);
      store_chunk(p, row, n_base + c, g, false);
    }
  } else {  // kEpiQkv
    const QkvEpilogueArgs& q = p.qkv;
    const int d = q.head_dim;
    const int half = d >> 1;
    const int n0 = tn * BN;
    const QkvRow r = qkv_row(p, row, valid);
#pragma unroll 1
    for (int j = 0; j < half; j += 32) {
      if (n0 >= q.q_size + q.kv_size) break;  // tile holds only v heads
      float sn[32], cs[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) rope_sincos(r.pos, rope_tab[j + e], sn[e], cs[e]);
#pragma unroll 1
      for (int hc = 0; hc < BN; hc += d) {
        const int col = n0 + hc;
        if (col >= q.q_size + q.kv_size) break;
        float lo[32], hi[32];
        ld(hc + j, lo);
        ld(hc + half + j, hi);
        if (valid) qkv_rotate_store(p, row, r, col, j, lo, hi, sn, cs);
      }
    }
    // v heads: plain copy into the cache
#pragma unroll 1
    for (int hc = 0; hc < BN; hc += d) {
      const int col = n0 + hc;
      if (col >= p.N) break;
      if (col < q.q_size + q.kv_size) continue;
#pragma unroll 1
      for (int j = 0; j < d; j += 32) {
        float v[32];
        ld(hc + j, v);
        if (valid) qkv_v_store(p, r, col, j, v);
      }
    }
  }
}

struct TmemLoader {
  uint32_t taddr;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const { tmem_ld32(taddr + col, v); }
};

// A loader whose values are multiplied by the row's scale (1 without one).
template <class Loader>
struct ScaledLoader {
  const Loader& ld;
  float s;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const {
    ld(col, v);
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] *= s;
  }
};

__device__ __forceinline__ float row_scale_of(const GemmParams& p, int row, int m_limit) {
  return p.row_scale != nullptr && row < m_limit ? p.row_scale[row] : 1.f;
}

// Partial tiles in the workspace: two slots per CTA (its first work item, and
// the split tile that ends its range), each [BN / 4][BM] float4, so 32
// consecutive rows of one 4-column group are 512 contiguous bytes.
__device__ __forceinline__ float4* partial_slot(float* partials, int cta, int slot) {
  return reinterpret_cast<float4*>(partials) + (static_cast<size_t>(cta) * 2 + slot) * (BM * BN / 4);
}

// Sum of the partial tiles that CTAs c_first..c_last left for one tile, in
// CTA order.  A CTA whose range starts inside the tile holds it in slot 0
// (its first work item), the others in slot 1.
struct PartialLoader {
  float* partials;
  long long units, t0;
  int grid, c_first, c_last, row;
  bool valid;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 0.f;
    if (!valid) return;
    for (int c = c_first; c <= c_last; ++c) {
      const int slot = sk_start(units, grid, c) >= t0 ? 0 : 1;
      const float4* src = partial_slot(partials, c, slot) + (col / 4) * BM + row;
      float4 t[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) t[q] = __ldcg(src + q * BM);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[4 * q] += t[q].x;
        v[4 * q + 1] += t[q].y;
        v[4 * q + 2] += t[q].z;
        v[4 * q + 3] += t[q].w;
      }
    }
  }
};

// NB: the tile width (BN, or 192 for the narrow SwiGLU tiles of decode-sized
// M: 96 gate and 96 up rows of B, in the first 24 KB of each stage's B slot).
template <int EPI, int NB = BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;

  static_assert(NB == BN || (EPI == kEpiSwiGlu && NB % 64 == 0 && NB < BN), "tile width");
  const int nst = p.stages, stage_bytes = p.stage_bytes, a_bytes = p.a_rows * BK * 2;
  const int stage_tx = a_bytes + NB * BK * 2;  // bytes a stage's loads deliver
  uint8_t* meta = smem + nst * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta);  // full[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * (2 * nst + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float2* rope_tab = reinterpret_cast<float2*>(meta + 512);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (nst + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * nst + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * nst + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * nst + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if constexpr (EPI == kEpiQkv) {
    if (warp >= 2) copy_rope_table(p, rope_tab, threadIdx.x - 64, NUM_THREADS - 64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  long long cursor, end;
  if (p.sk) {
    cursor = sk_start(p.units, p.grid, blockIdx.x);
    end = sk_start(p.units, p.grid, blockIdx.x + 1);
  } else {
    cursor = blockIdx.x;
    end = 0;
  }

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // The weight tiles of the first nst k-blocks are requested before
    // waiting for the previous kernel (no kernel of the chain writes weights);
    // their activation tiles follow once it has completed.
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = p.b_evict_first ? policy_evict_first() : policy_evict_normal();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t uses[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) uses[s] = 0;
    bool waited = false;
    int n_pre = 0;
    int pre_kb[kMaxStages], pre_row[kMaxStages];
    auto finish_wait = [&]() {
      pdl_wait();
      if (lane == 0)
        for (int i = 0; i < n_pre; ++i)
          tma_load_2d(sbase + i * stage_bytes, &tmA, full_bar(i), pre_kb[i] * BK, pre_row[i], pol_a);
      __syncwarp();
      waited = true;
    };
    Work w;
    bool ok = true;
    if (p.group_tiles != nullptr) finish_wait();  // the tile list itself comes from the previous kernel
    Feed feed = feed_init(p, cursor);
    while (ok && next_work(p, cursor, end, w, feed)) {
      const TileCoords tc = resolve_tile(p, w);
      const int arow = tc.arow;
      const int brow0 = tc.brow0;
      const int brow1 = brow0 + p.b_row_step;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sa = sbase + stage * stage_bytes;
          const uint32_t sb = sa + a_bytes;
          mbar_arrive_expect_tx(full_bar(stage), stage_tx);
          if (waited) tma_load_2d(sa, &tmA, full_bar(stage), kb * BK, arow, pol_a);
          tma_load_2d(sb, &tmB, full_bar(stage), kb * BK, brow0, pol_b);
          tma_load_2d(sb + NB * BK, &tmB, full_bar(stage), kb * BK, brow1, pol_b);  // second NB / 2 rows
        }
        __syncwarp();
        if (!waited) {  // stage == n_pre here
          pre_kb[n_pre] = kb;
          pre_row[n_pre] = arow;
          ++n_pre;
        }
        uses[stage]++;
        if (++stage == nst) {
          stage = 0;
          phase ^= 1u;
        }
        if (!waited && n_pre == nst) finish_wait();
      }
    }
    if (!waited) finish_wait();
    // Every load is queued: the next kernel may be scheduled now.  (A trigger
    // at the start would park its CTAs beside this persistent kernel for its
    // whole run.)
    if (lane == 0) pdl_trigger();
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmProducer);
      *abort_flag = 1;
    }
    // wait for every load this warp issued to land before the CTA can exit
    for (int s = 0; s < nst; ++s)
      if (uses[s] > 0) mbar_wait(full_bar(s), (uses[s] - 1) & 1u, nullptr);
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // its bounded waits start only once the previous kernel has completed
    pdl_wait();
    constexpr uint32_t idesc = idesc_bf16_f32(BM, NB);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, issued = false;
    Work w;
    Feed feed = feed_init(p, cursor);
    while (ok && next_work(p, cursor, end, w, feed)) {
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = sbase + stage * stage_bytes;
          const uint32_t sb = sa + a_bytes;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            tc_mma_f16(d_tmem, smem_desc_sw128(sa + 32 * k), smem_desc_sw128(sb + 32 * k), idesc,
                       (kb > w.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          issued = true;
        }
        __syncwarp();
        if (++stage == nst) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(tfull_bar(acc));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmMma);
      *abort_flag = 1;
    }
    // all MMAs this thread issued must finish before tensor memory is freed
    if (lane == 0 && issued) tc_commit(drain_bar);
    __syncwarp();
    if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) mbar_wait(drain_bar, 0, nullptr);
  } else {
    // ---------------- epilogue warps ----------------
    const int quad = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row_in_tile = quad * 32 + lane;
    pdl_wait();
    int acc = 0;
    uint32_t acc_phase = 0;
    int nseg = 0;
    Work w;
    bool ok = true;
    Feed feed = feed_init(p, cursor);
    while (next_work(p, cursor, end, w, feed)) {
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const TileCoords tc = resolve_tile(p, w);
      const int tm = tc.tm, tn = tc.tn;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      const bool valid = tm * BM + row_in_tile < tc.m_limit;
      if (w.kb0 == 0 && w.kb1 == p.kb) {
        TmemLoader tl{taddr};
        ScaledLoader<TmemLoader> ld{tl, row_scale_of(p, tm * BM + row_in_tile, tc.m_limit)};
        epilogue_tile<EPI, NB>(p, tm, tn, row_in_tile, ld, rope_tab, tc.m_limit);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
      } else {
        // a split tile: this CTA's partial goes to the workspace
        float4* dst = partial_slot(p.partials, blockIdx.x, nseg == 0 ? 0 : 1) + row_in_tile;
#pragma unroll 1
        for (int c = 0; c < NB && tm * BM + quad * 32 < tc.m_limit; c += 32) {  // rows past M are never read
          float v[32];
          tmem_ld32(taddr + c, v);
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[(c / 4 + q) * BM] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
      }
      ++nseg;
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmEpilogue);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// The persistent GEMM on SM pairs: a 2-CTA cluster computes 256 x 256 output
// tiles with M = 256 pair MMAs (tcgen05.mma.cta_group::2).  CTA r loads rows
// 128r..128r+127 of the tile's A rows and its half of the tile's B rows
// (plain: B rows 128r.. of the tile; SwiGLU: the 128 gate rows on rank 0 and
// the matching up rows on rank 1) and receives D rows 128r.. in its own
// tensor memory, all 256 columns, so the epilogue of each CTA is the 1-CTA
// kernel's over its 128 rows.  Per k-block each SM loads 32 KB instead of
// 48 KB for the same MMA work: the B operand is shared by the pair.
//   * both producers (warp 0) wait for their own stage's empty barrier and
//     load into their own shared memory, signalling rank 0's full barrier
//     (rank 0 expects the pair's 64 KB);
//   * one thread of rank 0 issues the MMAs and commits to the empty, tfull
//     and drain barriers of both CTAs at once (multicast commit);
//   * the epilogue warps of both CTAs drain their own accumulator and arrive
//     on rank 0's tempty barrier (8 arrivals).
// ---------------------------------------------------------------------------
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_A_BYTES = BM * BK * 2;              // 16 KB: this CTA's 128 rows of A
constexpr int PAIR_B_BYTES = (BN / 2) * BK * 2;        // 16 KB: this CTA's 128 rows of B
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_SMEM_BYTES = PAIR_STAGES * PAIR_STAGE_BYTES + 2048;

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;

  uint8_t* meta = smem + PAIR_STAGES * PAIR_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta);  // full[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * (2 * PAIR_STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float2* rope_tab = reinterpret_cast<float2*>(meta + 512);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (PAIR_STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * PAIR_STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * PAIR_STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * PAIR_STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 or 1
  const bool lead = rank == 0;
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);
  // this CTA and its peer stop waiting once either of them gives up
  auto give_up = [&]() {
    *abort_flag = 1;
    st_cluster_u32(peer_abort, 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);  // the four epilogue warps of each CTA
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  if constexpr (EPI == kEpiQkv) {
    if (warp >= 2) copy_rope_table(p, rope_tab, threadIdx.x - 64, NUM_THREADS - 64);
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int npairs = static_cast<int>(gridDim.x) >> 1;
  const long long first = static_cast<long long>(blockIdx.x >> 1);

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = p.b_evict_first ? policy_evict_first() : policy_evict_normal();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t uses[PAIR_STAGES];
#pragma unroll
    for (int s = 0; s < PAIR_STAGES; ++s) uses[s] = 0;
    bool waited = false, ok = true;
    int n_pre = 0;
    int pre_kb[PAIR_STAGES], pre_row[PAIR_STAGES];
    auto finish_wait = [&]() {
      pdl_wait();
      if (lane == 0)
        for (int i = 0; i < n_pre; ++i)
          tma_load_2d_pair(sbase + i * PAIR_STAGE_BYTES, &tmA, mapa_shared(full_bar(i), 0), pre_kb[i] * BK,
                           pre_row[i], pol_a);
      __syncwarp();
      waited = true;
    };
    for (long long t = first; ok && t < p.tiles; t += npairs) {
      int tm, tn;
      tile_coords(p, static_cast<int>(t), tm, tn);
      const int arow = tm * 2 * BM + static_cast<int>(rank) * BM;
      const int brow = tn * p.b_tile_rows + static_cast<int>(rank) * p.b_row_step;
      for (int kb = 0; kb < p.kb; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sa = sbase + stage * PAIR_STAGE_BYTES;
          const uint32_t sb = sa + PAIR_A_BYTES;
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (lead) mbar_arrive_expect_tx(full_bar(stage), 2 * PAIR_STAGE_BYTES);
          if (waited) tma_load_2d_pair(sa, &tmA, fb, kb * BK, arow, pol_a);
          tma_load_2d_pair(sb, &tmB, fb, kb * BK, brow, pol_b);
        }
        __syncwarp();
        if (!waited) {
          pre_kb[n_pre] = kb;
          pre_row[n_pre] = arow;
          ++n_pre;
        }
        uses[stage]++;
        if (++stage == PAIR_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (!waited && n_pre == PAIR_STAGES) finish_wait();
      }
    }
    if (!waited) finish_wait();
    if (lane == 0) pdl_trigger();
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmProducer);
      give_up();
    }
    // rank 0's full barriers count the bytes of both CTAs: once every last
    // phase has completed, every load of the pair has landed
    if (lead)
      for (int s = 0; s < PAIR_STAGES; ++s)
        if (uses[s] > 0) mbar_wait(full_bar(s), (uses[s] - 1) & 1u, nullptr);
  } else if (warp == 1) {
    // ---------------- MMA issuer (rank 0) ----------------
    pdl_wait();
    if (lead) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long t = first; ok && t < p.tiles; t += npairs) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = sbase + stage * PAIR_STAGE_BYTES;
            const uint32_t sb = sa + PAIR_A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma_f16_pair(d_tmem, smem_desc_sw128(sa + 32 * k), smem_desc_sw128(sb + 32 * k), idesc,
                              (kb > 0 || k > 0) ? 1u : 0u);
            tc_commit_pair(empty_bar(stage), 3);
          }
          __syncwarp();
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) tc_commit_pair(tfull_bar(acc), 3);
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmMma);
        give_up();
      }
      // completes in both CTAs once every MMA issued above has (at once if none was)
      if (lane == 0) tc_commit_pair(drain_bar, 3);
      __syncwarp();
    }
    // no CTA frees tensor memory the pair's MMAs may still write
    mbar_wait(drain_bar, 0, nullptr);
  } else {
    // ---------------- epilogue warps (both CTAs) ----------------
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    const uint32_t tempty_lead0 = mapa_shared(tempty_bar(0), 0);
    pdl_wait();
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (long long t = first; t < p.tiles; t += npairs) {
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      int tm, tn;
      tile_coords(p, static_cast<int>(t), tm, tn);
      const int vtm = 2 * tm + static_cast<int>(rank);  // this CTA's 128-row block
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      TmemLoader tl{taddr};
      ScaledLoader<TmemLoader> ld{tl, row_scale_of(p, vtm * BM + row_in_tile, p.M)};
      epilogue_tile<EPI>(p, vtm, tn, row_in_tile, ld, rope_tab, p.M);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_lead0 + 8u * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmEpilogue);
      give_up();
    }
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Split-K over a thread-block cluster, for problems with at most half as many
// tiles as SMs (decode-sized M).  The S CTAs of a cluster compute one tile,
// CTA rank r over k-blocks [r*kb/S, (r+1)*kb/S).  CTA r finishes the column
// units u with u % S == r of every row.  Once every CTA's MMAs are done (a
// cluster barrier), each CTA writes the 32-column chunks of its accumulator
// straight into the shared memory of the CTA that finishes them (remote
// stores into the operand ring, idle by then), a second barrier makes them
// visible, and each CTA sums the S slices of its own chunks in rank order from
// its own shared memory.  Stores to another CTA need no round trip, unlike
// loads from it, so the reduction is not bound by distributed-shared-memory
// latency.  No partial tile leaves the chip and no second kernel runs.
// ---------------------------------------------------------------------------

// The unit that reads accumulator chunk c (columns 32c..32c+31) in
// epilogue_unit and which of the unit's chunks it is; every unit reads
// kChunksPerUnit chunks.
template <int EPI>
struct ChunkMap {
  static constexpr int kChunksPerUnit = (EPI == kEpiBf16 || EPI == kEpiF32) ? 1 : 2;
  __device__ __forceinline__ static void of(const GemmParams& p, int c, int& unit, int& which) {
    if constexpr (EPI == kEpiBf16 || EPI == kEpiF32) {
      unit = c;
      which = 0;
    } else if constexpr (EPI == kEpiSwiGlu) {  // gate columns 32u.., up columns BN/2 + 32u..
      unit = c % (BN / 64);
      which = c / (BN / 64);
    } else {  // qkv: per head, lo chunks j then hi chunks half + j
      const int per_head = p.qkv.head_dim / 64;
      const int head = c / (2 * per_head), within = c % (2 * per_head);
      unit = head * per_head + within % per_head;
      which = within / per_head;
    }
  }
};

// Chunks CTA r receives: those of units r, r + S, ...; slot of chunk (unit, which).
template <int EPI>
__host__ __device__ constexpr int cluster_local_chunks(int S) {
  return (EpiUnits<EPI>::kUnits + S - 1) / S * ChunkMap<EPI>::kChunksPerUnit;
}

// Receive buffer of CTA r: [source rank s][local chunk][8 float4 columns][BM rows],
// so a warp's 32 rows write and read 512 contiguous bytes.
__device__ __forceinline__ uint32_t recv_offset(int s, int nloc, int li, int q, int row) {
  return static_cast<uint32_t>((((s * nloc + li) * 8 + q) * BM + row) * 16);
}

template <int EPI>
struct PushLoader {
  const GemmParams& p;
  const uint8_t* recv;  // this CTA's receive buffer
  int S, nloc, row;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const {
    int unit, which;
    ChunkMap<EPI>::of(p, col / 32, unit, which);
    const int li = unit / S * ChunkMap<EPI>::kChunksPerUnit + which;
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 0.f;
    for (int s = 0; s < S; ++s) {
      float4 t[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) t[q] = *reinterpret_cast<const float4*>(recv + recv_offset(s, nloc, li, q, row));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[4 * q] += t[q].x;
        v[4 * q + 1] += t[q].y;
        v[4 * q + 2] += t[q].z;
        v[4 * q + 3] += t[q].w;
      }
    }
  }
};

template <int EPI>
__global__ void __launch_bounds__(kClusterThreads, 1)
    k_gemm_cluster(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;

  const int nst = p.stages, stage_bytes = p.stage_bytes, a_bytes = p.a_rows * BK * 2;
  uint8_t* meta = smem + nst * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta);  // full[S], empty[S], tfull, drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(meta + 8 * (2 * nst + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float2* rope_tab = reinterpret_cast<float2*>(meta + 512);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (nst + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * nst);
  const uint32_t drain_bar = bar0 + 8u * (2 * nst + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int tile = static_cast<int>(blockIdx.x) / S;
  const int kb0 = static_cast<int>(static_cast<long long>(rank) * p.kb / S);
  const int kb1 = static_cast<int>(static_cast<long long>(rank + 1) * p.kb / S);
  int tm, tn;
  tile_coords(p, tile, tm, tn);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), BN);
    tmem_relinquish();
  }
  if constexpr (EPI == kEpiQkv) {
    if (warp >= 2) copy_rope_table(p, rope_tab, threadIdx.x - 64, kClusterThreads - 64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (weights of the first stages before the
    // previous kernel completes, as in k_gemm_tc) ----------------
    const uint64_t pol_a = policy_evict_last();
    const uint64_t pol_b = policy_evict_first();
    const int arow = tm * BM;
    const int brow0 = tn * p.b_tile_rows;
    const int brow1 = brow0 + p.b_row_step;
    uint32_t uses[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) uses[s] = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool waited = false, ok = true;
    int n_pre = 0;
    int pre_kb[kMaxStages];
    auto finish_wait = [&]() {
      pdl_wait();
      if (lane == 0)
        for (int i = 0; i < n_pre; ++i)
          tma_load_2d(sbase + i * stage_bytes, &tmA, full_bar(i), pre_kb[i] * BK, arow, pol_a);
      __syncwarp();
      waited = true;
    };
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t sa = sbase + stage * stage_bytes;
        const uint32_t sb = sa + a_bytes;
        mbar_arrive_expect_tx(full_bar(stage), a_bytes + B_BYTES);
        if (waited) tma_load_2d(sa, &tmA, full_bar(stage), kb * BK, arow, pol_a);
        tma_load_2d(sb, &tmB, full_bar(stage), kb * BK, brow0, pol_b);
        tma_load_2d(sb + B_BYTES / 2, &tmB, full_bar(stage), kb * BK, brow1, pol_b);
      }
      __syncwarp();
      if (!waited) pre_kb[n_pre++] = kb;
      uses[stage]++;
      if (++stage == nst) {
        stage = 0;
        phase ^= 1u;
      }
      if (!waited && n_pre == nst) finish_wait();
    }
    if (!waited) finish_wait();
    if (lane == 0) pdl_trigger();
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmProducer);
      *abort_flag = 1;
    }
    for (int s = 0; s < nst; ++s)
      if (uses[s] > 0) mbar_wait(full_bar(s), (uses[s] - 1) & 1u, nullptr);
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true, issued = false;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sa = sbase + stage * stage_bytes;
        const uint32_t sb = sa + a_bytes;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc_mma_f16(tmem_base, smem_desc_sw128(sa + 32 * k), smem_desc_sw128(sb + 32 * k), idesc,
                     (kb > kb0 || k > 0) ? 1u : 0u);
        tc_commit(empty_bar(stage));
        issued = true;
      }
      __syncwarp();
      if (++stage == nst) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmMma);
      *abort_flag = 1;
    } else if (lane == 0) {
      tc_commit(tfull_bar);
    }
    if (lane == 0 && issued) tc_commit(drain_bar);
    __syncwarp();
    if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) mbar_wait(drain_bar, 0, nullptr);
  } else {
    // ---------------- epilogue warps: wait for the accumulator ----------------
    pdl_wait();
    if (!mbar_wait(tfull_bar, 0, abort_flag)) {
      if (lane == 0) report_error(p.err, kErrTimeout, kWhereGemmEpilogue);
      *abort_flag = 1;
    }
  }

  constexpr int kUnits = EpiUnits<EPI>::kUnits;
  const int nloc = cluster_local_chunks<EPI>(S);
  if (S * nloc * BM * 128 > nst * stage_bytes) {  // the host never picks such an S
    if (threadIdx.x == 0) report_error(p.err, kErrGuard, kWhereGemmEpilogue);
    *abort_flag = 1;
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // every MMA of the cluster is done: the operand rings may be written
  tc_fence_after();
  const int quad = warp & 3;
  if (!*abort_flag && tm * BM + quad * 32 < p.M) {  // rows past M are never read
    // this warp's 32 accumulator rows, half of the chunks (warps q and q + 4
    // share lane quarter q), into the ring of the CTA that finishes each
    // chunk; the next chunk is loaded while this one is stored
    constexpr int kPerWarp = BN / 32 / 2;
    const int row_in_tile = quad * 32 + lane;
    const int c0 = (warp >> 2) * kPerWarp;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    auto push = [&](int c, const uint32_t (&r)[32]) {
      int unit, which;
      ChunkMap<EPI>::of(p, c, unit, which);
      const int li = unit / S * ChunkMap<EPI>::kChunksPerUnit + which;
      const uint32_t dst = mapa_shared(sbase + recv_offset(rank, nloc, li, 0, row_in_tile),
                                       static_cast<uint32_t>(unit % S));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_cluster_f4(dst + q * BM * 16, make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                     __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
    };
    uint32_t r0[32], r1[32];
    tmem_ld32_async(taddr + c0 * 32, r0);
    tmem_ld_wait(r0);
#pragma unroll
    for (int i = 0; i < kPerWarp; i += 2) {
      tmem_ld32_async(taddr + (c0 + i + 1) * 32, r1);
      push(c0 + i, r0);
      tmem_ld_wait(r1);
      if (i + 2 < kPerWarp) tmem_ld32_async(taddr + (c0 + i + 2) * 32, r0);
      push(c0 + i + 1, r1);
      if (i + 2 < kPerWarp) tmem_ld_wait(r0);
    }
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // every chunk has arrived; no CTA touches another's shared memory after this
  tc_fence_after();
  if (!*abort_flag) {
    // the units of this CTA, row group by row group, spread over the eight warps
    int item = 0;
    for (int u = rank; u < kUnits; u += S) {
      for (int g = 0; g < BM / 32; ++g) {
        if (tm * BM + g * 32 >= p.M) break;
        if ((item++ & 7) != warp) continue;
        const int row_in_tile = g * 32 + lane;
        PushLoader<EPI> pl{p, smem, S, nloc, row_in_tile};
        ScaledLoader<PushLoader<EPI>> ld{pl, row_scale_of(p, tm * BM + row_in_tile, p.M)};
        epilogue_unit<EPI>(p, tm, tn, row_in_tile, u, ld, rope_tab);
      }
    }
  }
  if (warp == 1) tmem_dealloc(tmem_base, BN);
}

// Sums the stream-K partial tiles of every tile that was split across CTAs
// and applies the epilogue.  One thread per (row, column unit): warp w of a
// CTA finishes unit w for 32 consecutive rows (its lanes), so every partial
// load of a warp is 512 contiguous bytes, and a tile is spread over BM / 32
// CTAs so the reads of a decode-sized problem run on many SMs at once.
constexpr int kFixRows = 32;

template <int EPI>
__global__ void __launch_bounds__(EpiUnits<EPI>::kUnits * 32) k_gemm_fixup(const __grid_constant__ GemmParams p) {
  constexpr int kUnits = EpiUnits<EPI>::kUnits;
  __shared__ float2 rope_tab[64];
  pdl_wait();
  pdl_trigger();
  const int tile = blockIdx.x;
  const long long t0 = static_cast<long long>(tile) * p.kb;
  const int c_first = sk_owner(p, t0), c_last = sk_owner(p, t0 + p.kb - 1);
  if (c_first == c_last) return;  // the whole tile was in one CTA
  int tm, tn;
  tile_coords(p, tile, tm, tn);
  if (tm * BM + static_cast<int>(blockIdx.y) * kFixRows >= p.M) return;  // no valid row in this CTA
  if constexpr (EPI == kEpiQkv) {
    copy_rope_table(p, rope_tab, threadIdx.x, kUnits * 32);
    __syncthreads();
  }
  const int unit = threadIdx.x >> 5;
  const int row_in_tile = blockIdx.y * kFixRows + (threadIdx.x & 31);
  PartialLoader pl{p.partials, p.units, t0, p.grid, c_first, c_last, row_in_tile, tm * BM + row_in_tile < p.M};
  ScaledLoader<PartialLoader> ld{pl, row_scale_of(p, tm * BM + row_in_tile, p.M)};
  epilogue_unit<EPI>(p, tm, tn, row_in_tile, unit, ld, rope_tab);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

// 2-D bf16 tensor [rows, cols] (cols contiguous) with a box of box_rows x 64
// columns and 128-byte swizzle; out-of-range elements read as zero.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int EPI>
cudaError_t set_smem_attrs() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(k_gemm_tc<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemBytes);
    if constexpr (EPI == kEpiSwiGlu)
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(k_gemm_tc<EPI, kNarrowBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxSmemBytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_gemm_cluster<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemBytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(k_gemm_pair<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, PAIR_SMEM_BYTES);
  });
  return err;
}

// 2-CTA clusters of k_gemm_pair<EPI> resident at once (one per TPC with both
// SMs free); cached per device.
template <int EPI>
int max_active_pairs() {
  constexpr int kDevs = 64;
  static int cache[kDevs] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = -1;
    if (set_smem_attrs<EPI>() == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(2 * 128);
      cfg.blockDim = dim3(NUM_THREADS);
      cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int v = 0;
      if (cudaOccupancyMaxActiveClusters(&v, k_gemm_pair<EPI>, &cfg) == cudaSuccess && v > 0) n = v;
      else cudaGetLastError();
    }
    cache[dev] = n;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

int max_active_pairs_of(int epi) {
  switch (epi) {
    case kEpiBf16:
      return max_active_pairs<kEpiBf16>();
    case kEpiQkv:
      return max_active_pairs<kEpiQkv>();
    case kEpiSwiGlu:
      return max_active_pairs<kEpiSwiGlu>();
    case kEpiF32:
      return max_active_pairs<kEpiF32>();
    default:
      return 0;
  }
}

// Clusters of S CTAs of k_gemm_cluster<EPI> that fit on the device at once
// (they need S SMs of one GPC each); cached per device.
template <int EPI>
int max_active_clusters(int S) {
  constexpr int kDevs = 64;
  static int cache[kDevs][9] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs || S < 2 || S > 8) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][S] == 0) {
    int n = -1;
    if (set_smem_attrs<EPI>() == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(S * 64);
      cfg.blockDim = dim3(kClusterThreads);
      cfg.dynamicSmemBytes = kMaxSmemBytes;  // one CTA per SM whatever the ring
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = static_cast<unsigned>(S);
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int v = 0;
      if (cudaOccupancyMaxActiveClusters(&v, k_gemm_cluster<EPI>, &cfg) == cudaSuccess && v > 0) n = v;
      else cudaGetLastError();
    }
    cache[dev][S] = n;
  }
  return cache[dev][S] > 0 ? cache[dev][S] : 0;
}

int max_active_clusters_of(int epi, int S) {
  switch (epi) {
    case kEpiBf16:
      return max_active_clusters<kEpiBf16>(S);
    case kEpiQkv:
      return max_active_clusters<kEpiQkv>(S);
    case kEpiSwiGlu:
      return max_active_clusters<kEpiSwiGlu>(S);
    case kEpiF32:
      return max_active_clusters<kEpiF32>(S);
    default:
      return 0;
  }
}

// Stages of stage_bytes that fit the ring budget.
int ring_stages(int stage_bytes) {
  const int n = kRingBudget / stage_bytes;
  return n < kMaxStages ? n : kMaxStages;
}

// The chunks a CTA of an S-CTA cluster receives fit its operand ring.
bool cluster_chunks_fit(int epi, int S, int ring_bytes) {
  int n = 0;
  switch (epi) {
    case kEpiBf16:
      n = cluster_local_chunks<kEpiBf16>(S);
      break;
    case kEpiQkv:
      n = cluster_local_chunks<kEpiQkv>(S);
      break;
    case kEpiSwiGlu:
      n = cluster_local_chunks<kEpiSwiGlu>(S);
      break;
    case kEpiF32:
      n = cluster_local_chunks<kEpiF32>(S);
      break;
    default:
      return false;
  }
  return S * n * BM * 128 <= ring_bytes;
}

template <int EPI>
int launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int cluster, bool pair,
                 bool narrow, bool pdl, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(p.stages) * p.stage_bytes + 2048;
  const cudaError_t attr_err = set_smem_attrs<EPI>();
  if (attr_err != cudaSuccess) return attr_err;
  if (pair)
    return launch_kernel_cluster(k_gemm_pair<EPI>, dim3(p.grid), dim3(NUM_THREADS), PAIR_SMEM_BYTES, s, pdl, 2, ta,
                                 tb, p);
  if (cluster > 1)
    return launch_kernel_cluster(k_gemm_cluster<EPI>, dim3(p.tiles * cluster), dim3(kClusterThreads), smem, s, pdl,
                                 cluster, ta, tb, p);
  if constexpr (EPI == kEpiSwiGlu) {
    if (narrow)
      return launch_kernel(k_gemm_tc<EPI, kNarrowBN>, dim3(p.grid), dim3(NUM_THREADS), smem, s, pdl, ta, tb, p);
  }
  cudaError_t e = launch_kernel(k_gemm_tc<EPI>, dim3(p.grid), dim3(NUM_THREADS), smem, s, pdl, ta, tb, p);
  if (e != cudaSuccess || !p.sk) return e;
  return launch_kernel(k_gemm_fixup<EPI>, dim3(p.tiles, BM / kFixRows), dim3(EpiUnits<EPI>::kUnits * 32), 0, s,
                       true, p);
}

}  // namespace

size_t gemm_partials_bytes(int sms) { return static_cast<size_t>(sms) * 2 * BM * BN * sizeof(float); }

// process-wide schedule override (llama_set_gemm_schedule); -1 = automatic
std::atomic<int> g_gemm_schedule{-1};

int gemm_launch(const GemmArgs& a, cudaStream_t s) {
  if (a.M <= 0) return 0;
  GemmParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.out = a.out;
  p.ldo = a.ldo;
  p.err = a.err;
  p.qkv = a.qkv;
  if (a.epi == kEpiQkv) {
    if (a.qkv.head_dim > 128 || a.qkv.head_dim % 64) return cudaErrorInvalidValue;
    rope_table_host(a.qkv.rope, a.qkv.head_dim, p.rope_tab);
  }
  p.partials = a.partials;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.kb = (a.K + BK - 1) / BK;
  if (a.epi == kEpiSwiGlu) {
    const int I = a.N / 2;
    p.tiles_n = (I + BN / 2 - 1) / (BN / 2);
    p.b_tile_rows = BN / 2;
    p.b_row_step = I;
    p.n_out = I;
  } else {
    p.tiles_n = (a.N + BN - 1) / BN;
    p.b_tile_rows = BN;
    p.b_row_step = BN / 2;
    p.n_out = a.N;
  }
  p.tiles = p.tiles_m * p.tiles_n;
  p.group_tiles = static_cast<const int4*>(a.group_tiles);
  p.group_count = a.group_count;
  p.row_scale = a.row_scale;
  const bool grouped = a.group_tiles != nullptr;
  const int mode = a.force_mode != -1 ? a.force_mode : g_gemm_schedule.load(std::memory_order_relaxed);
  // Raster: 24 M-tiles per group, so the 152 concurrent tiles cover 24
  // activation panels x ~6 weight panels, and weight loads are marked
  // evict-first so the activation panels of the group stay in L2 while the
  // weights stream past (measured on the 70B gate_up GEMM: 1.48 -> 1.73
  // PFLOP/s at 4128 rows, 1.48 -> 1.68 at 32768 rows, against 16-tile groups
  // with normal eviction).
  // Grouped mode: an expert's weight tiles are shared by the tiles of its
  // other row blocks, running at about the same time, so they keep the normal
  // policy (MoE block at 4096 tokens: 0.448 -> 0.423 ms).
  p.b_evict_first = grouped ? 0 : 1;
  p.group_m = p.tiles_m < 24 ? p.tiles_m : 24;
  const int sms = num_sms();
  // A box of 64 rows when M <= 64 (not for SM pairs or expert tiles): every
  // stage is 8 KB smaller, so the ring holds more stages of weights in flight.
  p.a_rows = (a.M <= 64 && !grouped && mode != 3) ? 64 : BM;
  const int wide_stage = p.a_rows * BK * 2 + B_BYTES;
  // At most sms / 2 tiles: split K over clusters of S CTAs (S as large as the
  // SMs allow, at least two k-blocks per CTA, all clusters resident at once).
  if (grouped && a.group_count == nullptr) return cudaErrorInvalidValue;
  int cluster = 0;
  if (!grouped && (mode == -1 || mode == 2) && p.tiles * 2 <= sms) {
    for (int S = sms / p.tiles < 8 ? sms / p.tiles : 8; S >= 2; --S) {
      if (p.kb < 2 * S || !cluster_chunks_fit(a.epi, S, ring_stages(wide_stage) * wide_stage) ||
          max_active_clusters_of(a.epi, S) < p.tiles)
        continue;
      cluster = S;
      break;
    }
  }
  // stream-K below one wave of whole tiles (the 8B decode gate_up, 112 tiles:
  // 48.8 us against 49.5 for whole tiles); from one wave up whole tiles win
  // (the 70B decode gate_up, 224 tiles: 162.9 us against 168.3 for stream-K
  // and its fixup)
  bool sk = cluster == 0 && p.tiles < sms;
  // Narrow SwiGLU tiles for one row block (decode): 192 columns instead of 256
  // when they fill the SMs' waves better, as whole tiles without a fixup (the
  // 8B decode gate_up: 150 tiles in one wave instead of 112 tiles of stream-K;
  // the 70B one: 299 tiles in two waves instead of 224).
  bool narrow = false;
  if (a.epi == kEpiSwiGlu && !grouped && mode == -1 && cluster == 0 && p.tiles_m == 1) {
    const int I = a.N / 2;
    const long long t_narrow = (I + kNarrowBN / 2 - 1) / (kNarrowBN / 2);
    const long long waves_narrow = (t_narrow + sms - 1) / sms, waves_wide = (p.tiles + sms - 1) / sms;
    if (waves_narrow * kNarrowBN < waves_wide * BN) {
      narrow = true;
      sk = false;
      p.tiles_n = static_cast<int>(t_narrow);
      p.b_tile_rows = kNarrowBN / 2;
      p.tiles = p.tiles_m * p.tiles_n;
    }
  }
  if (mode == 0 || mode == 3) sk = false;
  if (mode == 1) sk = true;
  if (grouped) sk = false;
  // SM pairs (k_gemm_pair) only when asked for (schedule 3).  On the 70B
  // gate_up GEMM (4128 and 32768 rows) the pair kernel keeps the tensor pipe
  // 89-90% busy against 78% for single-SM tiles, but the part is then held by
  // its power limit: the SM clock drops from 1.85 to 1.62-1.65 GHz, its
  // raster re-reads more weights from DRAM (4.9-9.8 GB against 2.4 GB per
  // launch), and in a seconds-long loop single-SM tiles are faster (2.42 vs
  // 2.46-2.63 ms at 4128 rows, 18.9 vs 19.5-21.2 ms at 32768).
  const bool pair = mode == 3 && !grouped;
  int npairs = 0;
  if (pair) {
    npairs = max_active_pairs_of(a.epi);
    if (npairs <= 0) return cudaErrorInvalidConfiguration;
    p.tiles_m = (a.M + 2 * BM - 1) / (2 * BM);
    p.tiles = p.tiles_m * p.tiles_n;
    p.group_m = p.tiles_m < 12 ? p.tiles_m : 12;  // 3072 activation rows per raster group, as above
  }
  p.stage_bytes = p.a_rows * BK * 2 + (narrow ? kNarrowBN : BN) * BK * 2;
  p.stages = ring_stages(p.stage_bytes);
  p.units = static_cast<long long>(p.tiles) * p.kb;
  if (sk) {
    long long g = p.units < sms ? p.units : sms;
    if (g < 1) g = 1;
    p.grid = static_cast<int>(g);
    if (gemm_partials_bytes(p.grid) > a.partials_bytes || a.partials == nullptr) return cudaErrorInvalidValue;
  } else if (pair) {
    p.grid = 2 * (p.tiles < npairs ? p.tiles : npairs);  // every pair has at least one tile
  } else {
    p.grid = grouped ? sms : (p.tiles < sms ? p.tiles : sms);  // grouped: the tile count is on the device
  }
  p.sk = sk ? 1 : 0;

  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a.A, a.M, a.K, p.a_rows)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.B, a.b_rows > 0 ? a.b_rows : a.N, a.K, (narrow ? kNarrowBN : BN) / 2))
    return cudaErrorInvalidValue;
  switch (a.epi) {
    case kEpiBf16:
      return launch_typed<kEpiBf16>(ta, tb, p, cluster, pair, narrow, a.pdl != 0, s);
    case kEpiQkv:
      return launch_typed<kEpiQkv>(ta, tb, p, cluster, pair, narrow, a.pdl != 0, s);
    case kEpiSwiGlu:
      return launch_typed<kEpiSwiGlu>(ta, tb, p, cluster, pair, narrow, a.pdl != 0, s);
    case kEpiF32:
      return launch_typed<kEpiF32>(ta, tb, p, cluster, pair, narrow, a.pdl != 0, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace llama
