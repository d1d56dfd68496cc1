// Host-side launch interface of the kernels (internal to the library; the
// public C ABI is include/llama_layer.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "llama_layer.h"

namespace llama {

enum GemmEpilogue : int {
  kEpiBf16 = 0,    // out[m, n] = bf16(acc)
  kEpiQkv = 1,     // RoPE on q/k columns, q -> q buffer, k/v -> paged caches
  kEpiSwiGlu = 2,  // out[m, j] = bf16(silu(gate_j) * up_j)
  kEpiF32 = 3,     // out[m, n] = acc (fp32)
};

struct RopeParams {
  float theta;
  int llama3;  // 0: plain frequencies, 1: llama3 frequency rule
  float factor, low_freq_factor, high_freq_factor;
  int original_max_pos;
};

struct QkvEpilogueArgs {
  int q_size, kv_size, head_dim, n_kv_heads, block_size, num_blocks;
  const int32_t* positions;  // [M]
  const int32_t* slots;      // [M], < 0 = skip
  void* k_cache;             // [num_blocks, n_kv, block, head_dim] bf16
  void* v_cache;
  RopeParams rope;
};

struct GemmArgs {
  int epi;
  const void* A;  // [M, K] bf16 row-major (activations)
  const void* B;  // [N, K] bf16 row-major (weights, [out, in]); SwiGLU: rows [gate(I); up(I)]
  int M, N, K;    // for SwiGLU, N = 2 * I
  void* out;      // bf16 or f32 [M, ldo]
  int ldo;
  QkvEpilogueArgs qkv;
  float* partials;  // stream-K partial tiles (see gemm_partials_bytes)
  size_t partials_bytes;
  int* err;
  int force_mode;  // -1 auto (or the llama_set_gemm_schedule override), 0 data-parallel, 1 stream-K,
                  // 2 cluster split-K where it fits, 3 SM pairs
  int pdl;         // 1: may start before the previous kernel on the stream (one of this library's) completes
  // Grouped mode (MoE experts): when group_tiles is set, the tiles are
  // {A row, B base row, N tile, valid rows} entries of a device list with
  // *group_count entries (written by a kernel earlier in the call); B holds
  // b_rows rows (all experts stacked) and A holds M rows.  Data-parallel only.
  const void* group_tiles;
  const int* group_count;
  int b_rows;
  // [M] fp32: row r of the product is multiplied by row_scale[r] before the
  // epilogue (an RMSNorm's rsqrt, its weights folded into B); null = 1
  const float* row_scale;
};

size_t gemm_partials_bytes(int num_sms);
int gemm_launch(const GemmArgs& a, cudaStream_t s);  // returns 0 or a CUDA error code

// fused residual add + RMSNorm over rows of length H
//   r = x (+ res_in); h = r * rsqrt(mean(r^2) + eps) * gamma
// With gamma null the norm is folded into the next GEMM: h is not written and
// Cache-slot mapping of a batch: slot[t] = block_table[b][pos/bs]*bs + pos%bs
// for token t of sequence b at position pos (-1 when out of range).
struct SlotMapArgs {
  const int32_t* positions;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int B, max_blocks, bs, num_blocks;
  int32_t* slots;  // [T] output; null: no slot mapping
  int* err;
};

// inv_out[row] receives rsqrt(mean(r^2) + eps).
// row_index_qsl != nullptr: output row b reads input row qsl[b+1]-1 (last
// token of sequence b), otherwise row b reads row b.
// slot_map != nullptr: the kernel also writes the batch's cache slots (one per
// row; rows must be the batch's tokens).
int add_rmsnorm_launch(const void* x, const void* res_in, void* res_out, void* h_out, const void* gamma,
                       int rows, int H, float eps, const int32_t* row_index_qsl, bool pdl, cudaStream_t s,
                       float* inv_out = nullptr, const SlotMapArgs* slot_map = nullptr);

// one CTA whose bounded wait on a barrier nothing arrives at runs out
int selftest_wait_launch(int* err, cudaStream_t s);

// w_folded[o, i] = bf16(w[o, i] * gamma[i]) for a [rows, cols] weight
int fold_norm_launch(const void* gamma, const void* w, int rows, int cols, void* w_folded, cudaStream_t s);

int kv_write_launch(const void* k, const void* v, const int32_t* slots, int T, int n_kv, int head_dim,
                    int block_size, int num_blocks, void* k_cache, void* v_cache, int* err, cudaStream_t s);

int embed_launch(const void* table, const int32_t* ids, int T, int H, int vocab, void* out, int* err, bool pdl,
                 cudaStream_t s);

int argmax_launch(const float* logits, int rows, int vocab, int32_t* out, bool pdl, cudaStream_t s);

// temperature / top-k / top-p sampling of fp32 logits rows (one uniform per
// row supplied by the caller); out_logprobs may be null
int sample_launch(const float* logits, int rows, int vocab, const float* temperature, const int32_t* top_k,
                  const float* top_p, const float* uniform, int32_t* out_tokens, float* out_logprobs, bool pdl,
                  cudaStream_t s);

struct AttnArgs {
  const void* q;        // [T, nq, d] bf16 (rotated)
  const void* k_cache;  // [num_blocks, nkv, bs, d]
  const void* v_cache;
  void* out;            // [T, nq * d] bf16
  const int32_t* qsl;   // [B+1]
  const int32_t* seq_lens;
  const int32_t* positions;
  const int32_t* block_table;  // [B, max_blocks]
  int T, B, max_blocks, num_blocks;
  int nq, nkv, head_dim, block_size;
  int max_query_len, max_seq_len;
  float* partials;  // decode split-KV partials
  size_t partials_bytes;
  int* err;
  int pdl;          // as GemmArgs::pdl
  int overlap;      // 1: with prefill sequences present, run the decode kernels on a side stream
};

// split-KV partials + the prefill work list of a batch of B sequences and T tokens
size_t attn_partials_bytes(int B, int T, int max_seq_len, int nq, int head_dim);
// *joined (if given) is set when the caller's stream waited on the side
// stream: the next kernel then has a full dependency, not a programmatic one.
int attention_launch(const AttnArgs& a, cudaStream_t s, bool* joined = nullptr);

// Sparse MoE block: workspace layout (byte offsets from a 256-aligned base)
// and the launch sequence.
struct MoeLayout {
  size_t rows;  // rows of the permuted activation matrices (segments padded to 128)
  size_t logits, ids, wts, slot_row, offset, fill, counts, tiles1, tiles2, x_perm, act, y_perm, gpart, total;
  size_t gpart_bytes;
};
MoeLayout moe_layout(int T, int H, int E, int K, int I, int sms);

struct MoeArgs {
  const void* h;         // [T, H] bf16
  const void* w_router;  // [E, H]
  const void* w13;       // [E, 2I, H]: gate rows then up rows per expert
  const void* w2;        // [E, H, I]
  void* out;             // [T, H] bf16
  int32_t* out_ids;      // [T, K] or null
  float* out_wts;        // [T, K] or null
  int T, H, E, K, I;
  uint8_t* ws;           // 256-aligned, moe_layout(...).total - 256 bytes
  int* err;
  bool chain;            // the first kernel may overlap the kernel before it (one of this library's)
};
int moe_launch(const MoeArgs& a, cudaStream_t s);

int num_sms();

// process-wide GEMM schedule override (-1 automatic); see llama_set_gemm_schedule
extern std::atomic<int> g_gemm_schedule;

// The configuration and batch checks every attention entry point makes
// (LLAMA_OK or the status it would return), with nothing launched.
int attention_args_status(const LlamaLayerConfig* cfg, const LlamaBatch* batch);

}  // namespace llama
