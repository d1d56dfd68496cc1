// C ABI of the library (declared in include/llama_layer.h): argument checks,
// workspace layout and the launch sequence of a layer and of a stack.
//
// Layer sequence ([CODE-READING] "vLLM Llama 代码解析" §3-§5, [LLAMA-70B]
// "LLama — DeepSeek-R1-Distill-Llama-70B" §3-§4 and LlamaMLP):
//   slot map -> input fused add+RMSNorm -> qkv GEMM (+RoPE, +cache scatter)
//   -> paged attention -> o_proj GEMM -> post-attention fused add+RMSNorm
//   -> gate_up GEMM (+SiluAndMul) -> down GEMM
// Stack ([CODE-READING] §2.1, [WALKTHROUGH] "模型库与算子层 — 代码走读" LlamaModel):
//   embedding gather -> layers with the residual threaded (None at layer 0)
//   -> final fused add+RMSNorm of each sequence's last token -> lm_head GEMM
//   -> argmax.
// Qwen3-MoE layer ([LLAMA-70B] Qwen3MoeSparseMoeBlock): the layer sequence up
// to the post-attention norm, then the sparse MoE block in place of gate_up
// and down.  With folded norms (null norm weights) the norm kernels write each
// row's rsqrt and the qkv and gate_up GEMMs scale their rows by it.
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "llama_layer.h"

namespace llama {

__device__ int g_device_error[2];

namespace {

constexpr int kMaxDevices = 64;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 0;
  return d;
}

// Optional timing of the gate_up GEMM launches inside the layer calls
// (llama_gate_up_timer_start / _stop): a pair of CUDA events around each
// launch, on the launching stream.
struct GateUpTimer {
  std::mutex mu;
  std::atomic<bool> on{false};
  int used = 0;
  std::vector<cudaEvent_t> ev;  // start, stop of launch i at 2i, 2i + 1
};

GateUpTimer& gate_up_timer() {
  static GateUpTimer t;
  return t;
}

// the event pair of the next timed launch (its start recorded), or -1
int gate_up_timer_begin(cudaStream_t s) {
  GateUpTimer& t = gate_up_timer();
  if (!t.on.load(std::memory_order_relaxed)) return -1;
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.on.load(std::memory_order_relaxed) || 2 * (t.used + 1) > static_cast<int>(t.ev.size())) return -1;
  const int i = t.used++;
  cudaEventRecord(t.ev[2 * i], s);
  return i;
}

void gate_up_timer_end(int i, cudaStream_t s) {
  if (i < 0) return;
  GateUpTimer& t = gate_up_timer();
  std::lock_guard<std::mutex> lock(t.mu);
  if (2 * i + 1 < static_cast<int>(t.ev.size())) cudaEventRecord(t.ev[2 * i + 1], s);
}

int* device_error_word() {
  static int* ptr[kMaxDevices] = {};
  static std::mutex mu;
  const int d = current_device();
  std::lock_guard<std::mutex> lock(mu);
  if (ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) ptr[d] = static_cast<int*>(p);
  }
  return ptr[d];
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int check_cfg(const LlamaLayerConfig* c) {
  if (c == nullptr) return LLAMA_ERR_ARG;
  if (c->hidden_act != 0) return LLAMA_ERR_ARG;  // only silu
  if (c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->intermediate <= 0)
    return LLAMA_ERR_ARG;
  if (c->n_heads % c->n_kv_heads != 0) return LLAMA_ERR_ARG;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return LLAMA_ERR_ARG;
  if (c->rope_scaling != 0 && c->rope_scaling != 1) return LLAMA_ERR_ARG;
  if (c->rope_scaling == 1 &&
      (!(c->rs_factor > 0.f) || !(c->rs_high_freq_factor > c->rs_low_freq_factor) || c->rs_original_max_pos <= 0 ||
       !(c->rs_low_freq_factor > 0.f)))
    return LLAMA_ERR_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return LLAMA_ERR_UNSUPPORTED;
  if (c->n_heads / c->n_kv_heads > 16) return LLAMA_ERR_UNSUPPORTED;
  if (c->block_size != 16) return LLAMA_ERR_UNSUPPORTED;
  if (c->hidden % 8 || c->intermediate % 8 || c->hidden > 16384) return LLAMA_ERR_UNSUPPORTED;
  return LLAMA_OK;
}

int check_batch(const LlamaBatch* b, const LlamaLayerConfig* c) {
  if (b == nullptr) return LLAMA_ERR_ARG;
  if (b->num_tokens < 0 || b->num_seqs < 0) return LLAMA_ERR_ARG;
  if (b->num_tokens == 0) return LLAMA_OK;
  if (b->num_seqs < 1 || b->num_seqs > b->num_tokens) return LLAMA_ERR_ARG;
  if (!b->positions || !b->query_start_loc || !b->seq_lens || !b->block_table) return LLAMA_ERR_ARG;
  if (b->max_blocks_per_seq < 1 || b->num_blocks < 1 || b->max_query_len < 1 || b->max_seq_len < 1)
    return LLAMA_ERR_ARG;
  if (b->max_query_len > b->num_tokens || b->max_query_len > b->max_seq_len) return LLAMA_ERR_ARG;
  // cache rows and slots are 32-bit on the device
  if (static_cast<long long>(b->num_blocks) * c->n_kv_heads * c->block_size > 0x7fffffffLL) return LLAMA_ERR_ARG;
  if (static_cast<long long>(b->num_seqs) * b->max_blocks_per_seq > 0x7fffffffLL) return LLAMA_ERR_ARG;
  if (b->num_seqs > 65535) return LLAMA_ERR_UNSUPPORTED;                   // grid z dimension
  if ((b->num_tokens + 7) / 8 + b->num_seqs > 65535) return LLAMA_ERR_UNSUPPORTED;  // prefill work items
  return LLAMA_OK;
}

struct Layout {
  size_t slots, rscale, h, q, o, a, gpart, apart, hf, logits, total;
  size_t gpart_bytes, apart_bytes;
};

Layout make_layout(const LlamaLayerConfig& c, int T, int B, int max_seq_len, int vocab) {
  Layout L{};
  const size_t t = T > 0 ? T : 0;
  const size_t qsz = static_cast<size_t>(c.n_heads) * c.head_dim;
  size_t off = 0;
  L.slots = off;
  off += align256(t * 4);
  L.rscale = off;  // per-row rsqrt of a norm folded into the next GEMM
  off += align256(t * 4);
  L.h = off;
  off += align256(t * c.hidden * 2);
  L.q = off;
  off += align256(t * qsz * 2);
  L.o = off;
  off += align256(t * qsz * 2);
  L.a = off;
  off += align256(t * c.intermediate * 2);
  L.gpart = off;
  L.gpart_bytes = gemm_partials_bytes(num_sms());
  off += align256(L.gpart_bytes);
  L.apart = off;
  L.apart_bytes =
      attn_partials_bytes(B > 0 ? B : 1, T > 0 ? T : 1, max_seq_len > 0 ? max_seq_len : 1, c.n_heads, c.head_dim);
  off += align256(L.apart_bytes);
  if (vocab > 0) {
    L.hf = off;
    off += align256(static_cast<size_t>(B) * c.hidden * 2);
    L.logits = off;
    off += align256(static_cast<size_t>(B) * vocab * 4);
  }
  L.total = off + 256;  // slack for aligning the caller's base pointer
  return L;
}

uint8_t* ws_base(void* ws) {
  const uintptr_t p = reinterpret_cast<uintptr_t>(ws);
  return reinterpret_cast<uint8_t*>((p + 255) & ~static_cast<uintptr_t>(255));
}

RopeParams rope_of(const LlamaLayerConfig& c) {
  RopeParams r{};
  r.theta = c.rope_theta;
  r.llama3 = c.rope_scaling;
  r.factor = c.rs_factor;
  r.low_freq_factor = c.rs_low_freq_factor;
  r.high_freq_factor = c.rs_high_freq_factor;
  r.original_max_pos = c.rs_original_max_pos;
  return r;
}

int cuda_status(int e) { return e == 0 ? LLAMA_OK : LLAMA_ERR_CUDA; }

// Both norm weights present, or both NULL (folded into w_qkv and w_gate_up).
int check_weights(const LlamaLayerWeights* w) {
  if (w == nullptr) return LLAMA_ERR_ARG;
  if ((w->ln1_w == nullptr) != (w->ln2_w == nullptr)) return LLAMA_ERR_ARG;
  const bool folded = w->ln1_w == nullptr;
  const void* ps[6] = {w->ln1_w, w->w_qkv, w->w_o, w->ln2_w, w->w_gate_up, w->w_down};
  for (int i = 0; i < 6; ++i) {
    const void* p = ps[i];
    if (folded && (i == 0 || i == 3)) continue;
    if (p == nullptr) return LLAMA_ERR_ARG;
    if (!a16(p)) return LLAMA_ERR_UNSUPPORTED;
  }
  return LLAMA_OK;
}

AttnArgs attn_args(const LlamaLayerConfig& c, const LlamaBatch& b, const void* q, const void* kc, const void* vc,
                   void* out, float* part, size_t part_bytes, int* err, bool pdl) {
  AttnArgs a{};
  a.q = q;
  a.k_cache = kc;
  a.v_cache = vc;
  a.out = out;
  a.qsl = b.query_start_loc;
  a.seq_lens = b.seq_lens;
  a.positions = b.positions;
  a.block_table = b.block_table;
  a.T = b.num_tokens;
  a.B = b.num_seqs;
  a.max_blocks = b.max_blocks_per_seq;
  a.num_blocks = b.num_blocks;
  a.nq = c.n_heads;
  a.nkv = c.n_kv_heads;
  a.head_dim = c.head_dim;
  a.block_size = c.block_size;
  a.max_query_len = b.max_query_len;
  a.max_seq_len = b.max_seq_len;
  a.partials = part;
  a.partials_bytes = part_bytes;
  a.err = err;
  a.pdl = pdl ? 1 : 0;
  a.overlap = 1;
  return a;
}

// The kernels of one layer, in order.  chain: the first kernel (the input
// norm, which reads nothing before it waits) may overlap the kernel before it
// on the stream; every later kernel overlaps its predecessor in the layer.
// The MLP of a Qwen3-MoE layer: the sparse block's config, weights and
// workspace, and where the chosen experts go (or null).
struct MoeMlp {
  const LlamaMoeConfig* cfg;
  const void *w_router, *w13, *w2;
  uint8_t* ws;
  int32_t* out_ids;
};

int layer_impl(const LlamaLayerConfig& c, const LlamaLayerWeights& w, const LlamaBatch& b, void* hidden,
               const void* res_in, void* res_out, void* kc, void* vc, uint8_t* ws, const Layout& L, bool chain,
               cudaStream_t s, const MoeMlp* moe = nullptr) {
  const int T = b.num_tokens;
  if (T == 0) return LLAMA_OK;
  int* err = device_error_word();
  const int H = c.hidden, I = c.intermediate;
  const int qsz = c.n_heads * c.head_dim, kvsz = c.n_kv_heads * c.head_dim;
  int32_t* slots = reinterpret_cast<int32_t*>(ws + L.slots);
  auto h = ws + L.h;
  auto q = ws + L.q;
  auto o = ws + L.o;
  auto a = ws + L.a;
  float* gpart = reinterpret_cast<float*>(ws + L.gpart);
  float* apart = reinterpret_cast<float*>(ws + L.apart);
  // folded norms: the norm kernels write only r and the row's rsqrt, and the
  // qkv / gate_up GEMMs read r and scale their rows by it (their weights carry
  // the norm weights)
  const bool folded = w.ln1_w == nullptr;
  float* rscale = folded ? reinterpret_cast<float*>(ws + L.rscale) : nullptr;
  int e;

  // cache slots: the caller's, or derived on the device by the input norm
  // kernel (its CTA of row t writes token t's slot)
  const int32_t* slot_map = b.slot_mapping;
  SlotMapArgs sm{};
  if (slot_map == nullptr) {
    sm = SlotMapArgs{b.positions, b.query_start_loc, b.seq_lens, b.block_table, b.num_seqs,
                     b.max_blocks_per_seq, c.block_size, b.num_blocks, slots, err};
    slot_map = slots;
  }
  // input_layernorm
  e = add_rmsnorm_launch(hidden, res_in, res_out, h, w.ln1_w, T, H, c.rms_eps, nullptr, chain, s, rscale,
                         sm.slots != nullptr ? &sm : nullptr);
  if (e) return cuda_status(e);
  const void* normed = folded ? res_out : h;  // the A operand of qkv (and, after the second norm, gate_up)
  auto gemm = [&](int epi, const void* A, const void* B, int N, int K, void* out, int ldo) {
    GemmArgs g{};
    g.epi = epi;
    g.A = A;
    g.B = B;
    g.M = T;
    g.N = N;
    g.K = K;
    g.out = out;
    g.ldo = ldo;
    g.partials = gpart;
    g.partials_bytes = L.gpart_bytes;
    g.err = err;
    g.force_mode = -1;
    g.pdl = 1;
    return g;
  };
  // qkv_proj + RoPE + cache update
  GemmArgs g = gemm(kEpiQkv, normed, w.w_qkv, qsz + 2 * kvsz, H, q, qsz);
  g.row_scale = rscale;
  g.qkv.q_size = qsz;
  g.qkv.kv_size = kvsz;
  g.qkv.head_dim = c.head_dim;
  g.qkv.n_kv_heads = c.n_kv_heads;
  g.qkv.block_size = c.block_size;
  g.qkv.num_blocks = b.num_blocks;
  g.qkv.positions = b.positions;
  g.qkv.slots = slot_map;
  g.qkv.k_cache = kc;
  g.qkv.v_cache = vc;
  g.qkv.rope = rope_of(c);
  e = gemm_launch(g, s);
  if (e) return cuda_status(e);
  // attention
  bool joined = false;
  e = attention_launch(attn_args(c, b, q, kc, vc, o, apart, L.apart_bytes, err, true), s, &joined);
  if (e) return cuda_status(e);
  // o_proj -> y (in the h buffer)
  GemmArgs go = gemm(kEpiBf16, o, w.w_o, H, qsz, h, H);
  go.pdl = joined ? 0 : 1;
  e = gemm_launch(go, s);
  if (e) return cuda_status(e);
  // post_attention_layernorm: r2 = y + r (in res_out), h2 (in the h buffer)
  e = add_rmsnorm_launch(h, res_out, res_out, h, w.ln2_w, T, H, c.rms_eps, nullptr, true, s, rscale);
  if (e) return cuda_status(e);
  if (moe != nullptr) {  // the sparse MoE block in place of the dense MLP
    MoeArgs m{};
    m.h = h;
    m.w_router = moe->w_router;
    m.w13 = moe->w13;
    m.w2 = moe->w2;
    m.out = hidden;
    m.out_ids = moe->out_ids;
    m.T = T;
    m.H = H;
    m.E = moe->cfg->num_experts;
    m.K = moe->cfg->top_k;
    m.I = moe->cfg->moe_intermediate;
    m.ws = moe->ws;
    m.err = err;
    m.chain = true;
    return cuda_status(moe_launch(m, s));
  }
  // gate_up_proj + SiluAndMul
  GemmArgs gu = gemm(kEpiSwiGlu, normed, w.w_gate_up, 2 * I, H, a, I);
  gu.row_scale = rscale;
  const int timed = gate_up_timer_begin(s);
  e = gemm_launch(gu, s);
  gate_up_timer_end(timed, s);
  if (e) return cuda_status(e);
  // down_proj -> hidden_states
  e = gemm_launch(gemm(kEpiBf16, a, w.w_down, H, I, hidden, H), s);
  return cuda_status(e);
}

}  // namespace

int attention_args_status(const LlamaLayerConfig* cfg, const LlamaBatch* batch) {
  const int st = check_cfg(cfg);
  return st ? st : check_batch(batch, cfg);
}

std::atomic<unsigned long long> g_launch_count{0};

int num_sms() {
  static std::atomic<int> sms[kMaxDevices];  // zero-initialised (static storage); filled once per device
  const int d = current_device();
  int v = sms[d].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0) v = 1;
    sms[d].store(v, std::memory_order_relaxed);
  }
  return v;
}

}  // namespace llama

using namespace llama;

extern "C" {

size_t llama_workspace_size(const LlamaLayerConfig* cfg, int max_tokens, int max_seqs, int max_seq_len, int vocab) {
  if (check_cfg(cfg) != LLAMA_OK || max_tokens < 0 || max_seqs < 0 || vocab < 0) return 0;
  return make_layout(*cfg, max_tokens, max_seqs, max_seq_len, vocab).total;
}

int llama_layer_forward(const LlamaLayerConfig* cfg, const LlamaLayerWeights* weights, const LlamaBatch* batch,
                        void* hidden_states, const void* residual_in, void* residual_out, void* k_cache,
                        void* v_cache, void* workspace, size_t workspace_bytes, llama_stream_t stream) {
  int st = check_cfg(cfg);
  if (st) return st;
  if ((st = check_weights(weights))) return st;
  if ((st = check_batch(batch, cfg))) return st;
  if (batch->num_tokens == 0) return LLAMA_OK;
  if (!hidden_states || !residual_out || !k_cache || !v_cache) return LLAMA_ERR_ARG;
  if (residual_out == hidden_states) return LLAMA_ERR_ARG;
  if (!a16(hidden_states) || !a16(residual_out) || !a16(k_cache) || !a16(v_cache) ||
      (residual_in && !a16(residual_in)))
    return LLAMA_ERR_UNSUPPORTED;
  const Layout L = make_layout(*cfg, batch->num_tokens, batch->num_seqs, batch->max_seq_len, 0);
  if (workspace == nullptr || workspace_bytes < L.total) return LLAMA_ERR_WORKSPACE;
  return layer_impl(*cfg, *weights, *batch, hidden_states, residual_in, residual_out, k_cache, v_cache,
                    ws_base(workspace), L, true, reinterpret_cast<cudaStream_t>(stream));
}

int llama_stack_forward(const LlamaLayerConfig* cfg, int num_layers, const LlamaLayerWeights* layers,
                        const void* final_norm_w, const void* lm_head_w, int vocab, const void* embed_w,
                        const int32_t* input_ids, const LlamaBatch* batch, void* hidden_states, void* residual,
                        void* const* k_caches, void* const* v_caches, int32_t* out_tokens, float* out_logits,
                        void* workspace, size_t workspace_bytes, llama_stream_t stream) {
  int st = check_cfg(cfg);
  if (st) return st;
  if (num_layers < 1 || layers == nullptr || k_caches == nullptr || v_caches == nullptr) return LLAMA_ERR_ARG;
  for (int l = 0; l < num_layers; ++l) {
    if ((st = check_weights(&layers[l]))) return st;
    if (!k_caches[l] || !v_caches[l]) return LLAMA_ERR_ARG;
    if (!a16(k_caches[l]) || !a16(v_caches[l])) return LLAMA_ERR_UNSUPPORTED;
  }
  if ((st = check_batch(batch, cfg))) return st;
  if (!final_norm_w || !lm_head_w || vocab < 1 || !hidden_states || !residual || !out_tokens) return LLAMA_ERR_ARG;
  if ((embed_w == nullptr) != (input_ids == nullptr)) return LLAMA_ERR_ARG;
  if (vocab % 8) return LLAMA_ERR_UNSUPPORTED;
  if (!a16(final_norm_w) || !a16(lm_head_w) || !a16(hidden_states) || !a16(residual) ||
      (embed_w && !a16(embed_w)) || (out_logits && !a16(out_logits)))
    return LLAMA_ERR_UNSUPPORTED;
  if (batch->num_tokens == 0) return LLAMA_OK;
  const Layout L = make_layout(*cfg, batch->num_tokens, batch->num_seqs, batch->max_seq_len, vocab);
  if (workspace == nullptr || workspace_bytes < L.total) return LLAMA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = ws_base(workspace);
  int* err = device_error_word();
  const int T = batch->num_tokens, B = batch->num_seqs, H = cfg->hidden;
  int e;
  if (embed_w) {
    e = embed_launch(embed_w, input_ids, T, H, vocab, hidden_states, err, true, s);
    if (e) return LLAMA_ERR_CUDA;
  }
  for (int l = 0; l < num_layers; ++l) {
    st = layer_impl(*cfg, layers[l], *batch, hidden_states, l == 0 ? nullptr : residual, residual, k_caches[l],
                    v_caches[l], ws, L, true, s);
    if (st) return st;
  }
  // final norm over the last token of every sequence
  void* hf = ws + L.hf;
  e = add_rmsnorm_launch(hidden_states, residual, nullptr, hf, final_norm_w, B, H, cfg->rms_eps,
                         batch->query_start_loc, true, s);
  if (e) return LLAMA_ERR_CUDA;
  float* logits = out_logits ? out_logits : reinterpret_cast<float*>(ws + L.logits);
  GemmArgs g{};
  g.epi = kEpiF32;
  g.A = hf;
  g.B = lm_head_w;
  g.M = B;
  g.N = vocab;
  g.K = H;
  g.out = logits;
  g.ldo = vocab;
  g.partials = reinterpret_cast<float*>(ws + L.gpart);
  g.partials_bytes = L.gpart_bytes;
  g.err = err;
  g.force_mode = -1;
  g.pdl = 1;
  e = gemm_launch(g, s);
  if (e) return LLAMA_ERR_CUDA;
  e = argmax_launch(logits, B, vocab, out_tokens, true, s);
  return e ? LLAMA_ERR_CUDA : LLAMA_OK;
}

int kv_cache_write(const void* k, const void* v, const int32_t* slot_mapping, int num_tokens, int n_kv_heads,
                   int head_dim, int block_size, int num_blocks, void* k_cache, void* v_cache, llama_stream_t stream) {
  if (num_tokens < 0 || n_kv_heads < 1 || head_dim < 8 || head_dim % 8 || block_size < 1 || num_blocks < 1)
    return LLAMA_ERR_ARG;
  if (num_tokens == 0) return LLAMA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return LLAMA_ERR_ARG;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return LLAMA_ERR_ARG;
  if (!a16(k) || !a16(v) || !a16(k_cache) || !a16(v_cache)) return LLAMA_ERR_UNSUPPORTED;
  const int e = kv_write_launch(k, v, slot_mapping, num_tokens, n_kv_heads, head_dim, block_size, num_blocks, k_cache,
                                v_cache, device_error_word(), reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

}  // extern "C"

namespace {

// A GEMM on its own, with its partial tiles in the caller's workspace.
int standalone_gemm(GemmArgs& g, void* workspace, cudaStream_t s) {
  g.partials = reinterpret_cast<float*>(ws_base(workspace));
  g.partials_bytes = gemm_partials_bytes(num_sms());
  g.err = device_error_word();
  g.force_mode = -1;
  g.pdl = 0;
  return gemm_launch(g, s);
}

}  // namespace

extern "C" {

size_t llama_linear_workspace_size(void) {
  return gemm_partials_bytes(num_sms()) + 256;
}

int llama_linear(const void* x, const void* w, int M, int N, int K, void* y, int out_fp32, void* workspace,
                 size_t workspace_bytes, llama_stream_t stream) {
  if (M < 0 || N < 1 || K < 1) return LLAMA_ERR_ARG;
  if (M == 0) return LLAMA_OK;
  if (!x || !w || !y) return LLAMA_ERR_ARG;
  if (N % 8 || K % 8) return LLAMA_ERR_UNSUPPORTED;
  if (!a16(x) || !a16(w) || !a16(y)) return LLAMA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < llama_linear_workspace_size()) return LLAMA_ERR_WORKSPACE;
  GemmArgs g{};
  g.epi = out_fp32 ? kEpiF32 : kEpiBf16;
  g.A = x;
  g.B = w;
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = y;
  g.ldo = N;
  return cuda_status(standalone_gemm(g, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

int llama_gate_up_silu(const void* x, const void* w_gate_up, int M, int I, int K, void* a, void* workspace,
                       size_t workspace_bytes, llama_stream_t stream) {
  if (M < 0 || I < 1 || K < 1) return LLAMA_ERR_ARG;
  if (M == 0) return LLAMA_OK;
  if (!x || !w_gate_up || !a) return LLAMA_ERR_ARG;
  if (I % 8 || K % 8) return LLAMA_ERR_UNSUPPORTED;
  if (!a16(x) || !a16(w_gate_up) || !a16(a)) return LLAMA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < llama_linear_workspace_size()) return LLAMA_ERR_WORKSPACE;
  GemmArgs g{};
  g.epi = kEpiSwiGlu;
  g.A = x;
  g.B = w_gate_up;
  g.M = M;
  g.N = 2 * I;
  g.K = K;
  g.out = a;
  g.ldo = I;
  return cuda_status(standalone_gemm(g, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

int llama_fused_add_rmsnorm(const void* x, const void* residual_in, void* residual_out, void* h, const void* gamma,
                            int rows, int H, float eps, llama_stream_t stream) {
  if (rows < 0 || H < 8 || H % 8 || H > 16384 || !(eps >= 0.f)) return LLAMA_ERR_ARG;
  if (rows == 0) return LLAMA_OK;
  if (!x || !h || !gamma) return LLAMA_ERR_ARG;
  if (!a16(x) || !a16(h) || !a16(gamma) || (residual_in && !a16(residual_in)) ||
      (residual_out && !a16(residual_out)))
    return LLAMA_ERR_UNSUPPORTED;
  return cuda_status(add_rmsnorm_launch(x, residual_in, residual_out, h, gamma, rows, H, eps, nullptr, false,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int llama_paged_attention(const LlamaLayerConfig* cfg, const LlamaBatch* batch, const void* q, const void* k_cache,
                          const void* v_cache, void* out, void* workspace, size_t workspace_bytes,
                          llama_stream_t stream) {
  int st = check_cfg(cfg);
  if (st) return st;
  if ((st = check_batch(batch, cfg))) return st;
  if (batch->num_tokens == 0) return LLAMA_OK;
  if (!q || !k_cache || !v_cache || !out) return LLAMA_ERR_ARG;
  if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(out)) return LLAMA_ERR_UNSUPPORTED;
  const size_t part =
      attn_partials_bytes(batch->num_seqs, batch->num_tokens, batch->max_seq_len, cfg->n_heads, cfg->head_dim);
  if (workspace == nullptr || workspace_bytes < part + 256) return LLAMA_ERR_WORKSPACE;
  AttnArgs a = attn_args(*cfg, *batch, q, k_cache, v_cache, out, reinterpret_cast<float*>(ws_base(workspace)), part,
                         device_error_word(), false);
  return cuda_status(attention_launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

int llama_sample(const float* logits, int rows, int vocab, const float* temperature, const int32_t* top_k,
                 const float* top_p, const float* uniform, int32_t* out_tokens, float* out_logprobs,
                 llama_stream_t stream) {
  if (rows < 0 || vocab < 1) return LLAMA_ERR_ARG;
  if (rows == 0) return LLAMA_OK;
  if (!logits || !temperature || !top_k || !top_p || !uniform || !out_tokens) return LLAMA_ERR_ARG;
  if (static_cast<long long>(rows) * vocab > 0x7fffffffffffLL) return LLAMA_ERR_ARG;
  return cuda_status(sample_launch(logits, rows, vocab, temperature, top_k, top_p, uniform, out_tokens, out_logprobs,
                                   false, reinterpret_cast<cudaStream_t>(stream)));
}

static int check_moe_cfg(const LlamaMoeConfig* c) {
  if (c == nullptr) return LLAMA_ERR_ARG;
  if (c->hidden < 8 || c->num_experts < 1 || c->top_k < 1 || c->moe_intermediate < 8) return LLAMA_ERR_ARG;
  if (c->top_k > c->num_experts) return LLAMA_ERR_ARG;
  if (c->hidden % 8 || c->moe_intermediate % 8) return LLAMA_ERR_UNSUPPORTED;
  if (c->num_experts > 512 || c->top_k > 32) return LLAMA_ERR_UNSUPPORTED;
  return LLAMA_OK;
}

size_t llama_moe_workspace_size(const LlamaMoeConfig* cfg, int max_tokens) {
  if (check_moe_cfg(cfg) != LLAMA_OK || max_tokens < 0) return 0;
  return moe_layout(max_tokens, cfg->hidden, cfg->num_experts, cfg->top_k, cfg->moe_intermediate, num_sms()).total;
}

int llama_moe_forward(const LlamaMoeConfig* cfg, const void* h, int num_tokens, const void* w_router, const void* w13,
                      const void* w2, void* out, int32_t* out_expert_ids, float* out_expert_weights, void* workspace,
                      size_t workspace_bytes, llama_stream_t stream) {
  int st = check_moe_cfg(cfg);
  if (st) return st;
  if (num_tokens < 0) return LLAMA_ERR_ARG;
  if (num_tokens == 0) return LLAMA_OK;
  if (!h || !w_router || !w13 || !w2 || !out) return LLAMA_ERR_ARG;
  if (!a16(h) || !a16(w_router) || !a16(w13) || !a16(w2) || !a16(out)) return LLAMA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_tokens) * cfg->top_k > 0x7fffffffLL) return LLAMA_ERR_UNSUPPORTED;
  const MoeLayout L =
      moe_layout(num_tokens, cfg->hidden, cfg->num_experts, cfg->top_k, cfg->moe_intermediate, num_sms());
  if (L.rows > 0x7fffffffULL) return LLAMA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < L.total) return LLAMA_ERR_WORKSPACE;
  MoeArgs a{};
  a.h = h;
  a.w_router = w_router;
  a.w13 = w13;
  a.w2 = w2;
  a.out = out;
  a.out_ids = out_expert_ids;
  a.out_wts = out_expert_weights;
  a.T = num_tokens;
  a.H = cfg->hidden;
  a.E = cfg->num_experts;
  a.K = cfg->top_k;
  a.I = cfg->moe_intermediate;
  a.ws = ws_base(workspace);
  a.err = device_error_word();
  return cuda_status(moe_launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t llama_moe_layer_workspace_size(const LlamaLayerConfig* cfg, const LlamaMoeConfig* moe, int max_tokens,
                                      int max_seqs, int max_seq_len) {
  if (check_cfg(cfg) != LLAMA_OK || check_moe_cfg(moe) != LLAMA_OK || moe->hidden != cfg->hidden) return 0;
  if (max_tokens < 0 || max_seqs < 0) return 0;
  const size_t layer = align256(make_layout(*cfg, max_tokens, max_seqs, max_seq_len, 0).total);
  return layer + moe_layout(max_tokens, moe->hidden, moe->num_experts, moe->top_k, moe->moe_intermediate, num_sms())
                     .total;
}

int llama_moe_layer_forward(const LlamaLayerConfig* cfg, const LlamaMoeConfig* moe,
                            const LlamaMoeLayerWeights* weights, const LlamaBatch* batch, void* hidden_states,
                            const void* residual_in, void* residual_out, void* k_cache, void* v_cache,
                            int32_t* out_expert_ids, void* workspace, size_t workspace_bytes,
                            llama_stream_t stream) {
  int st = check_cfg(cfg);
  if (st) return st;
  if ((st = check_moe_cfg(moe))) return st;
  if (moe->hidden != cfg->hidden || weights == nullptr) return LLAMA_ERR_ARG;
  const void* ps[7] = {weights->ln1_w, weights->w_qkv, weights->w_o, weights->ln2_w,
                       weights->w_router, weights->w13, weights->w2};
  for (const void* p : ps) {
    if (p == nullptr) return LLAMA_ERR_ARG;
    if (!a16(p)) return LLAMA_ERR_UNSUPPORTED;
  }
  if ((st = check_batch(batch, cfg))) return st;
  if (batch->num_tokens == 0) return LLAMA_OK;
  if (!hidden_states || !residual_out || !k_cache || !v_cache) return LLAMA_ERR_ARG;
  if (residual_out == hidden_states) return LLAMA_ERR_ARG;
  if (!a16(hidden_states) || !a16(residual_out) || !a16(k_cache) || !a16(v_cache) ||
      (residual_in && !a16(residual_in)))
    return LLAMA_ERR_UNSUPPORTED;
  const int T = batch->num_tokens;
  if (static_cast<long long>(T) * moe->top_k > 0x7fffffffLL) return LLAMA_ERR_UNSUPPORTED;
  const Layout L = make_layout(*cfg, T, batch->num_seqs, batch->max_seq_len, 0);
  const MoeLayout ML = moe_layout(T, moe->hidden, moe->num_experts, moe->top_k, moe->moe_intermediate, num_sms());
  if (ML.rows > 0x7fffffffULL) return LLAMA_ERR_UNSUPPORTED;
  const size_t layer_bytes = align256(L.total);
  if (workspace == nullptr || workspace_bytes < layer_bytes + ML.total) return LLAMA_ERR_WORKSPACE;
  uint8_t* base = ws_base(workspace);
  LlamaLayerWeights w{};
  w.ln1_w = weights->ln1_w;
  w.w_qkv = weights->w_qkv;
  w.w_o = weights->w_o;
  w.ln2_w = weights->ln2_w;
  MoeMlp mm{moe, weights->w_router, weights->w13, weights->w2, base + layer_bytes, out_expert_ids};
  return layer_impl(*cfg, w, *batch, hidden_states, residual_in, residual_out, k_cache, v_cache, base, L, true,
                    reinterpret_cast<cudaStream_t>(stream), &mm);
}

int llama_fold_norm_weights(const void* norm_weight, const void* w, int rows, int cols, void* w_folded,
                            llama_stream_t stream) {
  if (norm_weight == nullptr || w == nullptr || w_folded == nullptr || rows < 0 || cols <= 0) return LLAMA_ERR_ARG;
  if (cols % 8 || !a16(norm_weight) || !a16(w) || !a16(w_folded)) return LLAMA_ERR_UNSUPPORTED;
  return cuda_status(fold_norm_launch(norm_weight, w, rows, cols, w_folded, reinterpret_cast<cudaStream_t>(stream)));
}

int llama_selftest_wait_timeout(llama_stream_t stream) {
  return cuda_status(selftest_wait_launch(device_error_word(), reinterpret_cast<cudaStream_t>(stream)));
}

int llama_get_device_error(llama_stream_t stream, int* detail) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LLAMA_ERR_CUDA;
  int* w = device_error_word();
  if (w == nullptr) return LLAMA_ERR_CUDA;
  int host[2] = {0, 0};
  if (cudaMemcpy(host, w, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (cudaMemset(w, 0, sizeof(host)) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return LLAMA_ERR_CUDA;
  if (detail) *detail = host[1];
  if (host[0] & kErrTimeout) return LLAMA_ERR_TIMEOUT;
  if (host[0] & kErrGuard) return LLAMA_ERR_DEVICE_GUARD;
  return LLAMA_OK;
}

const char* llama_status_string(int status) {
  switch (status) {
    case LLAMA_OK:
      return "ok";
    case LLAMA_ERR_ARG:
      return "invalid argument";
    case LLAMA_ERR_UNSUPPORTED:
      return "unsupported shape or alignment";
    case LLAMA_ERR_CUDA:
      return "CUDA error";
    case LLAMA_ERR_WORKSPACE:
      return "workspace missing or too small";
    case LLAMA_ERR_DEVICE_GUARD:
      return "device guard: an index was out of range";
    case LLAMA_ERR_TIMEOUT:
      return "device wait timed out";
    case LLAMA_ERR_SCRATCH_LIMIT:
      return "batch needs more split-KV scratch than llama_paged_attention_noalloc's fixed array";
    default:
      return "unknown status";
  }
}

int llama_num_sms(void) { return num_sms(); }

uint64_t llama_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

int llama_gate_up_timer_start(int max_launches) {
  if (max_launches < 1 || max_launches > (1 << 20)) return LLAMA_ERR_ARG;
  GateUpTimer& t = gate_up_timer();
  std::lock_guard<std::mutex> lock(t.mu);
  if (t.on.load()) return LLAMA_ERR_ARG;
  for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
  t.ev.assign(2 * static_cast<size_t>(max_launches), nullptr);
  for (auto& e : t.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      cudaGetLastError();
      for (cudaEvent_t x : t.ev)
        if (x) cudaEventDestroy(x);
      t.ev.clear();
      return LLAMA_ERR_CUDA;
    }
  }
  t.used = 0;
  t.on.store(true);
  return LLAMA_OK;
}

int llama_gate_up_timer_stop(float* total_ms, int* launches) {
  GateUpTimer& t = gate_up_timer();
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.on.load()) return LLAMA_ERR_ARG;
  t.on.store(false);
  float total = 0.f;
  int st = LLAMA_OK;
  for (int i = 0; i < t.used; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess) {
      cudaGetLastError();
      st = LLAMA_ERR_CUDA;
      break;
    }
    total += ms;
  }
  if (total_ms) *total_ms = total;
  if (launches) *launches = t.used;
  for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
  t.ev.clear();
  t.used = 0;
  return st;
}

int llama_set_gemm_schedule(int schedule) {
  if (schedule < -1 || schedule > 3) return LLAMA_ERR_ARG;
  g_gemm_schedule.store(schedule, std::memory_order_relaxed);
  return LLAMA_OK;
}

}  // extern "C"
