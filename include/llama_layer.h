/*
 * llama_layer.h - C ABI of the GB300 (sm_103a) Llama decoder-layer forward.
 *
 * The library computes, over one flat batch of tokens drawn from many
 * sequences,
 *
 *     hidden_states, residual = layer(positions, hidden_states, residual)
 *
 * for one Llama decoder layer (llama_layer_forward), for a stack of layers
 * followed by the final norm, lm_head and greedy sampling
 * (llama_stack_forward), and the paged KV-cache write on its own
 * (kv_cache_write).  Past that path: the building blocks on their own
 * (llama_linear, llama_gate_up_silu, llama_fused_add_rmsnorm,
 * llama_paged_attention), sampling with temperature, top-k and top-p
 * (llama_sample), the Qwen3-MoE sparse block and decoder layer
 * (llama_moe_forward, llama_moe_layer_forward), norm weights folded into the
 * projections (llama_fold_norm_weights) and a self-test of the device-side
 * failure path (llama_selftest_wait_timeout).
 *
 * Sources (three web pages on vLLM's llama.py), cited by tag:
 *   [LLAMA-70B]    "LLama - DeepSeek-R1-Distill-Llama-70B" (hotelren.com
 *                  walk-through): config.json; section 3 input_layernorm
 *                  (RMSNorm with the residual add fused in); section 4
 *                  LlamaAttention; LlamaMLP and SiluAndMul; the final RMSNorm;
 *                  the Sampler.
 *   [WALKTHROUGH]  "模型库与算子层 — 代码走读" (vllm-learning code
 *                  walkthrough): LlamaModel, LlamaDecoderLayer, Attention
 *                  (_update_kv_cache, attn_backend.forward with block_table),
 *                  Linear layers (F.linear, weights stored [out, in]).
 *   [CODE-READING] "vLLM Llama 代码解析" (yeyulingfeng.com): section 1
 *                  LlamaForCausalLM (packed_modules_mapping, compute_logits),
 *                  section 2.1 LlamaModel.forward (layer loop carrying the
 *                  residual, final norm), section 4 LlamaAttention, section 5
 *                  LlamaMLP.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; all
 *     struct pointers (cfg, weights, batch, the per-layer arrays) are HOST
 *     pointers read during the call only.
 *   - Tensors are dense row-major; bf16 unless stated; 16-byte aligned.
 *   - The caller owns all memory.  The library never allocates or frees
 *     device memory: scratch comes from the caller's workspace, whose size
 *     llama_workspace_size() returns.
 *   - Work is enqueued on `stream` and runs asynchronously; nothing
 *     synchronises the host.  Results are valid once the stream reaches them.
 *     Each kernel of a call may start its prologue while the kernel before
 *     it on the stream finishes (programmatic dependent launch) and reads
 *     that kernel's results only after it has completed.  The first kernel
 *     of llama_layer_forward, llama_stack_forward and llama_moe_layer_forward
 *     (an embedding gather or a norm) reads nothing before then, so work
 *     queued before the call is complete before any of its data is read;
 *     the other entry points' first kernels start only after everything
 *     queued before them has completed.
 *   - A workspace belongs to one call at a time: calls that may overlap on the
 *     GPU need separate workspaces.  Its contents need not be initialised.
 *   - A call returns LLAMA_OK, or a status code without launching anything
 *     when its arguments are rejected.  No C++ exception crosses the ABI.
 *   - Kernels never trap.  An out-of-range index met on the device (a cache
 *     slot, a block-table entry, a token id, a position past seq_lens) is
 *     recorded in a device error word and the access is skipped; a wait that
 *     runs past its limit (2 s) is recorded and the kernel winds down.
 *     llama_get_device_error() reports and clears the word.
 *   - The library keeps no other state than that error word (one per device),
 *     cached kernel attributes and SM counts, one non-blocking side stream
 *     per device (decode attention beside prefill attention in mixed
 *     batches), a fork/join event pair per host thread and device, a launch
 *     counter, and the fixed scratch array of llama_paged_attention_noalloc.
 */
#ifndef LLAMA_LAYER_H_
#define LLAMA_LAYER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers (same underlying type). */
typedef struct CUstream_st* llama_stream_t;

/* Status codes. */
enum {
  LLAMA_OK = 0,
  LLAMA_ERR_ARG = 1,          /* null pointer, inconsistent or invalid size, unsupported activation */
  LLAMA_ERR_UNSUPPORTED = 2,  /* valid but unsupported shape or alignment */
  LLAMA_ERR_CUDA = 3,         /* a CUDA launch or runtime call failed */
  LLAMA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than llama_workspace_size() */
  LLAMA_ERR_DEVICE_GUARD = 5, /* reported by llama_get_device_error: an index was out of range */
  LLAMA_ERR_TIMEOUT = 6,      /* reported by llama_get_device_error: a device wait gave up */
  LLAMA_ERR_SCRATCH_LIMIT = 7 /* llama_paged_attention_noalloc: the batch needs more than its fixed scratch */
};

/* Layer shape and constants.  [LLAMA-70B] config.json: hidden_size,
 * num_attention_heads, num_key_value_heads, head_dim, intermediate_size,
 * rms_norm_eps, rope_theta, rope_scaling (llama3), hidden_act.
 * Supported: head_dim 64 or 128; n_heads a multiple of n_kv_heads with
 * n_heads / n_kv_heads <= 16; hidden, intermediate and n_heads*head_dim
 * multiples of 8 (16-byte rows), hidden <= 16384; block_size 16;
 * hidden_act 0 (silu).  Any other activation is rejected with LLAMA_ERR_ARG,
 * as LlamaMLP raises for it ([LLAMA-70B] LlamaMLP). */
typedef struct {
  int hidden;
  int n_heads;
  int n_kv_heads;
  int head_dim;
  int intermediate;
  int block_size;          /* tokens per KV-cache block (16) */
  float rms_eps;
  float rope_theta;
  int rope_scaling;        /* 0: plain RoPE frequencies; 1: llama3 frequency rule */
  float rs_factor;         /* llama3: factor (8) */
  float rs_low_freq_factor;  /* llama3: low_freq_factor (1) */
  float rs_high_freq_factor; /* llama3: high_freq_factor (4) */
  int rs_original_max_pos;   /* llama3: original_max_position_embeddings (8192) */
  int hidden_act;          /* 0 = silu; anything else is rejected */
} LlamaLayerConfig;

/* Weights of one layer, bf16, stored [out, in] as F.linear expects
 * ([WALKTHROUGH] Linear layers).  The merged projections are packed in the
 * order of [CODE-READING] section 1 packed_modules_mapping:
 *   w_qkv     [(n_heads + 2*n_kv_heads)*head_dim, hidden]  rows q; k; v
 *   w_o       [hidden, n_heads*head_dim]
 *   w_gate_up [2*intermediate, hidden]                     rows gate; up
 *   w_down    [hidden, intermediate]
 *   ln1_w, ln2_w [hidden]  RMSNorm weights (input / post-attention). */
typedef struct {
  const void* ln1_w;
  const void* w_qkv;
  const void* w_o;
  const void* ln2_w;
  const void* w_gate_up;
  const void* w_down;
} LlamaLayerWeights;

/* Folded norms.  ln1_w and ln2_w may both be NULL when w_qkv and w_gate_up
 * carry the norm weights in their columns (llama_fold_norm_weights):
 *   norm(r) W^T = rsqrt(mean(r^2) + eps) * (r (W diag(gamma))^T),
 * so the norm kernels write only the residual r and each row's rsqrt, and the
 * qkv and gate_up GEMMs read r and scale their rows by it before their
 * epilogues (RoPE, SiluAndMul).  The normed activations h are then never
 * stored; the rounding to bf16 moves from h to the folded weights.  One NULL
 * and one non-NULL norm weight is LLAMA_ERR_ARG.  (The final norm of
 * llama_stack_forward is not folded.) */

/* w_folded[o, i] = bf16(w[o, i] * norm_weight[i]) for a weight w [rows, cols]
 * bf16 (cols a multiple of 8) and a norm weight [cols] bf16; w_folded may
 * equal w.  Asynchronous on stream. */
int llama_fold_norm_weights(const void* norm_weight, const void* w, int rows, int cols, void* w_folded,
                            llama_stream_t stream);

/* One flat batch ([CODE-READING] section 2.1: tokens of many sequences, with
 * their positions).  Sequence b owns tokens [query_start_loc[b],
 * query_start_loc[b+1]).  Its context length seq_lens[b] counts the cached
 * tokens plus this step's; its cache blocks are block_table[b][0 ..
 * ceil(seq_lens[b]/16)-1] ([WALKTHROUGH] Attention: kv_cache.block_table).
 * A token at position p attends to cache positions 0..p of its sequence
 * (this step's tokens are written first, so it sees itself).  A sequence with
 * one new token takes the split-KV decode path, one with two or more the
 * prefill path; both may appear in one batch.  The cache slots this step
 * writes lie only in blocks of their own sequence that no other sequence of
 * the batch reads (blocks shared between sequences hold only earlier
 * tokens): the decode path requests a sequence's blocks before its last one
 * while the qkv projection of the same call is still writing.
 * Device arrays (int32): positions [num_tokens], query_start_loc
 * [num_seqs+1], seq_lens [num_seqs], block_table [num_seqs,
 * max_blocks_per_seq], slot_mapping [num_tokens] or NULL (then slot =
 * block_table[b][pos/16]*16 + pos%16 is derived on the device; a negative
 * slot skips the token's cache write).  Host ints: max_query_len and
 * max_seq_len bound the batch's query lengths and seq_lens (they size the
 * launch grids; a sequence beyond them is reported as a device guard). */
typedef struct {
  int num_tokens;
  int num_seqs;
  int max_blocks_per_seq;
  int num_blocks;          /* blocks in each cache array */
  int max_query_len;
  int max_seq_len;
  const int32_t* positions;
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const int32_t* slot_mapping;
} LlamaBatch;

/* Bytes of workspace a call needs for at most max_tokens tokens, max_seqs
 * sequences and seq_lens up to max_seq_len; vocab > 0 adds what
 * llama_stack_forward needs for the logits of max_seqs rows.  Returns 0 for
 * an invalid config. */
size_t llama_workspace_size(const LlamaLayerConfig* cfg, int max_tokens, int max_seqs, int max_seq_len, int vocab);

/* One decoder layer ([CODE-READING] sections 3-5, [LLAMA-70B] sections 3-4
 * and LlamaMLP):
 *   h, r   = fused_add_rmsnorm(hidden_states, residual_in, ln1_w)
 *            (residual_in NULL: r = hidden_states, [LLAMA-70B] section 3)
 *   q,k,v  = split(h W_qkv^T); q, k rotated by RoPE at positions (v is not)
 *   cache  : k, v stored (bf16) at each token's slot ([WALKTHROUGH] Attention)
 *   o      = causal GQA attention of q over the paged cache
 *   h2, r2 = fused_add_rmsnorm(o W_o^T, r, ln2_w)
 *   out    = (silu(h2 W_gate^T) * (h2 W_up^T)) W_down^T
 * hidden_states [num_tokens, hidden]: input x, overwritten with out.
 * residual_in [num_tokens, hidden] or NULL; residual_out [num_tokens, hidden]
 * receives r2 (may equal residual_in).  k_cache, v_cache [num_blocks,
 * n_kv_heads, 16, head_dim] bf16 are updated in place. */
int llama_layer_forward(const LlamaLayerConfig* cfg, const LlamaLayerWeights* weights, const LlamaBatch* batch,
                        void* hidden_states, const void* residual_in, void* residual_out, void* k_cache,
                        void* v_cache, void* workspace, size_t workspace_bytes, llama_stream_t stream);

/* The model body and head over one flat batch ([CODE-READING] section 2.1;
 * [WALKTHROUGH] LlamaModel; [LLAMA-70B] final RMSNorm and Sampler):
 *   x = embed_w[input_ids] (if embed_w and input_ids are given; otherwise the
 *       caller has put the input rows in hidden_states)
 *   for each layer l: x, r = layer_l(positions, x, r), r = None at layer 0
 *   hf = rmsnorm(x + r, final_norm_w) for the last token of every sequence
 *   logits = hf lm_head_w^T (fp32, [num_seqs, vocab]); out_tokens = argmax
 *   (lowest index on ties).
 * layers, k_caches, v_caches are HOST arrays of num_layers entries (device
 * pointers inside).  hidden_states and residual are [num_tokens, hidden]
 * device buffers the call overwrites.  out_tokens [num_seqs] int32;
 * out_logits [num_seqs, vocab] fp32 or NULL. */
int llama_stack_forward(const LlamaLayerConfig* cfg, int num_layers, const LlamaLayerWeights* layers,
                        const void* final_norm_w, const void* lm_head_w, int vocab, const void* embed_w,
                        const int32_t* input_ids, const LlamaBatch* batch, void* hidden_states, void* residual,
                        void* const* k_caches, void* const* v_caches, int32_t* out_tokens, float* out_logits,
                        void* workspace, size_t workspace_bytes, llama_stream_t stream);

/* The paged KV-cache update on its own ([WALKTHROUGH] Attention,
 * _update_kv_cache): k, v [num_tokens, n_kv_heads, head_dim] bf16 are copied
 * to cache[slot/16][h][slot%16][:] for every token with slot_mapping >= 0;
 * slots >= num_blocks*16 are reported as a device guard and skipped. */
int kv_cache_write(const void* k, const void* v, const int32_t* slot_mapping, int num_tokens, int n_kv_heads,
                   int head_dim, int block_size, int num_blocks, void* k_cache, void* v_cache, llama_stream_t stream);

/* Building blocks of the layer, exposed for tests and for callers composing
 * their own step. */

/* y[M, N] = x[M, K] W[N, K]^T ([WALKTHROUGH] Linear layers); y bf16
 * (out_fp32 = 0) or fp32 (out_fp32 = 1).  K and N multiples of 8.
 * The workspace holds split-K partial tiles (llama_linear_workspace_size). */
int llama_linear(const void* x, const void* w, int M, int N, int K, void* y, int out_fp32, void* workspace,
                 size_t workspace_bytes, llama_stream_t stream);
size_t llama_linear_workspace_size(void);

/* a[M, I] = silu(x W_gate^T) * (x W_up^T) with w_gate_up [2I, K] holding the
 * gate rows then the up rows: the merged gate_up projection with SiluAndMul
 * in its epilogue ([LLAMA-70B] LlamaMLP; [CODE-READING] section 5).  a bf16.
 * I and K multiples of 8; workspace as for llama_linear. */
int llama_gate_up_silu(const void* x, const void* w_gate_up, int M, int I, int K, void* a, void* workspace,
                       size_t workspace_bytes, llama_stream_t stream);

/* r = x (+ residual_in); h = r / sqrt(mean(r^2) + eps) * gamma, per row of
 * length H ([LLAMA-70B] section 3; eps inside the square root).  residual_out
 * may be NULL or alias x / residual_in; h may alias x. */
int llama_fused_add_rmsnorm(const void* x, const void* residual_in, void* residual_out, void* h, const void* gamma,
                            int rows, int H, float eps, llama_stream_t stream);

/* Causal GQA attention of q [num_tokens, n_heads, head_dim] (already rotated)
 * over the paged caches, for the batch described by `batch`; writes
 * out [num_tokens, n_heads*head_dim].  ([WALKTHROUGH] Attention.)
 * The workspace llama_workspace_size() gives for the batch is large enough. */
int llama_paged_attention(const LlamaLayerConfig* cfg, const LlamaBatch* batch, const void* q, const void* k_cache,
                          const void* v_cache, void* out, void* workspace, size_t workspace_bytes,
                          llama_stream_t stream);

/* The paged attention above, for callers that cannot allocate device memory
 * at the point where they run attention.  Examples are a plugin that its host
 * framework hands only input and output buffers, a process whose memory pool
 * another runtime owns, and a loop that forbids allocation after start-up.
 * None of these can provide the workspace llama_paged_attention needs.  The
 * pages have no counterpart to this entry point.
 * The split-KV scratch is a fixed array of llama_paged_attention_noalloc_limit()
 * bytes (32 MiB) inside the library.  Every GPU that loads the library holds it
 * until the process exits.  A batch whose scratch needs more than that
 * (num_seqs * ceil(ceil(max_seq_len/16)/96) * n_heads * (head_dim+2) * 4
 * + 4 * (ceil(num_tokens/8) + num_seqs) + 512 bytes) is rejected with
 * LLAMA_ERR_SCRATCH_LIMIT before anything is launched; an invalid configuration
 * or batch is rejected first, with the status llama_paged_attention gives it.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.  The
 * address is kept for the life of the device's context: after cudaDeviceReset,
 * do not call this entry point again on that device.
 * All calls share the one array, so calls that overlap on the GPU race on it:
 * the caller must serialise them.  Nothing in it has to start at zero.
 * Arguments and results are those of llama_paged_attention. */
int llama_paged_attention_noalloc(const LlamaLayerConfig* cfg, const LlamaBatch* batch, const void* q,
                                  const void* k_cache, const void* v_cache, void* out, llama_stream_t stream);
size_t llama_paged_attention_noalloc_limit(void);

/* Sampling beyond greedy ([LLAMA-70B] Sampler, sample(): temperature scaling,
 * the top-k / top-p sampler, greedy rows below a temperature threshold, the
 * sampled tokens' logprobs).  For every row b of logits [rows, vocab] (fp32):
 *   temperature[b] < 1e-5: the token is the argmax (lowest index on ties);
 *   otherwise, with w_i = exp((l_i - max l) / temperature[b]):
 *     top-k keeps every token whose logit is >= the top_k[b]-th largest
 *       (ties kept; top_k[b] <= 0 or >= vocab keeps all),
 *     top-p keeps, inside that set, every token with w_i >= tau, tau the
 *       largest value whose kept mass is >= top_p[b] times the top-k set's
 *       mass (ties kept; top_p[b] >= 1 keeps all, <= 0 only the maximum),
 *     the token is the first kept token in index order at which the running
 *       kept mass exceeds uniform[b] times the total kept mass.
 * uniform [rows] holds the caller's random draws in [0, 1) (values outside are
 * clamped); temperature, top_p [rows] fp32 and top_k [rows] int32 are device
 * arrays.  out_tokens [rows] int32; out_logprobs [rows] fp32 (or NULL) gets
 * the raw log-softmax of the unscaled logits at the sampled token.  Masses
 * are exact 64-bit fixed-point sums (weights below 2^-40 count as zero), so a
 * call is deterministic. */
int llama_sample(const float* logits, int rows, int vocab, const float* temperature, const int32_t* top_k,
                 const float* top_p, const float* uniform, int32_t* out_tokens, float* out_logprobs,
                 llama_stream_t stream);

/* Sparse MoE block (the Qwen3 MoE MLP: [LLAMA-70B] Qwen3MoeSparseMoeBlock;
 * [WALKTHROUGH] Fused MoE).  For every token row t of h [num_tokens, hidden]:
 *   logits = h[t] w_router^T (fp32 accumulation, kept in fp32),
 *   the top_k experts by logit (equal logits: the lower expert index) with
 *   weights = softmax of their k logits (norm_topk_prob),
 *   y_e = SiluAndMul(h[t] w13[e]^T) w2[e]^T for each of them, every module
 *   output stored in bf16 like the dense MLP,
 *   out[t] = sum over the k experts, in routing order, of weight * y_e (fp32
 *   sum, bf16 out).  No shared expert.
 * w_router [num_experts, hidden], w13 [num_experts, 2*moe_intermediate,
 * hidden] (gate rows then up rows per expert), w2 [num_experts, hidden,
 * moe_intermediate], all bf16; out [num_tokens, hidden] bf16.  The chosen
 * experts and weights go to out_expert_ids [num_tokens, top_k] int32 and
 * out_expert_weights [num_tokens, top_k] fp32 when those are not NULL.
 * num_experts <= 512, top_k <= 32, hidden and moe_intermediate multiples of 8.
 * The workspace (llama_moe_workspace_size) holds the router logits, the
 * routing, the tokens permuted into per-expert segments of whole 128-row tiles
 * and the experts' intermediate activations. */
typedef struct {
  int hidden;
  int num_experts;
  int top_k;
  int moe_intermediate;
} LlamaMoeConfig;

size_t llama_moe_workspace_size(const LlamaMoeConfig* cfg, int max_tokens);
int llama_moe_forward(const LlamaMoeConfig* cfg, const void* h, int num_tokens, const void* w_router, const void* w13,
                      const void* w2, void* out, int32_t* out_expert_ids, float* out_expert_weights, void* workspace,
                      size_t workspace_bytes, llama_stream_t stream);

/* Weights of one Qwen3-MoE decoder layer: the attention half of a Llama
 * layer (same layouts as LlamaLayerWeights) and the MoE block's weights
 * (same layouts as llama_moe_forward). */
typedef struct {
  const void* ln1_w;
  const void* w_qkv;
  const void* w_o;
  const void* ln2_w;
  const void* w_router;  /* [num_experts, hidden] */
  const void* w13;       /* [num_experts, 2*moe_intermediate, hidden] */
  const void* w2;        /* [num_experts, hidden, moe_intermediate] */
} LlamaMoeLayerWeights;

/* Workspace bytes of llama_moe_layer_forward (0 for an invalid config or a
 * moe->hidden different from cfg->hidden). */
size_t llama_moe_layer_workspace_size(const LlamaLayerConfig* cfg, const LlamaMoeConfig* moe, int max_tokens,
                                      int max_seqs, int max_seq_len);

/* One Qwen3-MoE decoder layer ([LLAMA-70B] Qwen3MoeForCausalLM config and
 * Qwen3MoeSparseMoeBlock; decoder_sparse_step 1, no mlp_only_layers): the
 * steps of llama_layer_forward up to and including the post-attention fused
 * add+RMSNorm, then out = the sparse MoE block of llama_moe_forward applied
 * to h2 in place of the dense MLP.  cfg->intermediate is not used.  Arguments
 * and in-place rules as llama_layer_forward; out_expert_ids [num_tokens,
 * top_k] int32 (or NULL) receives each token's chosen experts. */
int llama_moe_layer_forward(const LlamaLayerConfig* cfg, const LlamaMoeConfig* moe,
                            const LlamaMoeLayerWeights* weights, const LlamaBatch* batch, void* hidden_states,
                            const void* residual_in, void* residual_out, void* k_cache, void* v_cache,
                            int32_t* out_expert_ids, void* workspace, size_t workspace_bytes,
                            llama_stream_t stream);

/* Self-test of the device-side failure path: launches one thread that waits
 * on a shared-memory barrier nothing arrives at, with the same bounded wait
 * every kernel uses (a 2 s wall-clock limit).  The wait gives up, the timeout
 * is recorded in the device error word (detail 64), and the kernel returns, so
 * the context stays usable: llama_get_device_error then reports
 * LLAMA_ERR_TIMEOUT.  Returns the launch status. */
int llama_selftest_wait_timeout(llama_stream_t stream);

/* Synchronises `stream`, returns LLAMA_OK, LLAMA_ERR_DEVICE_GUARD or
 * LLAMA_ERR_TIMEOUT for the current device's error word, and clears it.
 * *detail (may be NULL) receives the code of the first place that reported. */
int llama_get_device_error(llama_stream_t stream, int* detail);

/* Human-readable name of a status code (static string). */
const char* llama_status_string(int status);

/* Number of streaming multiprocessors of the current device (cached). */
int llama_num_sms(void);

/* Kernels this process has launched through the library so far, on every
 * device (a host-side counter, incremented when a launch is accepted).  The
 * difference across a region counts that region's kernels. */
uint64_t llama_launch_count(void);

/* Timing of the dominant kernel inside the layer and stack calls: between
 * llama_gate_up_timer_start and llama_gate_up_timer_stop, every gate_up GEMM
 * launch that llama_layer_forward or llama_stack_forward makes (up to
 * max_launches) is bracketed by a pair of CUDA events on its stream.  _stop
 * synchronises those events and returns the summed elapsed time (ms) and the
 * number of launches timed.  A process-wide setting for benchmarks; the pages
 * have no counterpart.  The events cost a little: the launch after them no
 * longer overlaps its predecessor's prologue.  Not for use during stream
 * capture.  Returns LLAMA_ERR_ARG for a bad count or when already running
 * (start) / not running (stop), LLAMA_ERR_CUDA if an event call fails. */
int llama_gate_up_timer_start(int max_launches);
int llama_gate_up_timer_stop(float* total_ms, int* launches);

/* Overrides how every projection GEMM of this process is scheduled (a process-
 * wide setting, read at each launch; for tests and benchmarks that need one
 * schedule).  The pages have no counterpart: they call library GEMMs.
 *   -1  automatic (the default): cluster split-K for at most half as many
 *       128 x 256 output tiles as SMs, stream-K below as many tiles as SMs,
 *       and whole tiles on single SMs from there on;
 *    0  whole 128 x 256 tiles on single SMs;
 *    1  stream-K on single SMs (needs the linear workspace);
 *    2  cluster split-K where the tiles fit, else as -1;
 *    3  whole 256 x 256 tiles on SM pairs (2-CTA clusters issuing tcgen05
 *       pair MMAs; the B operand is loaded once for both SMs).  Slower than 0
 *       on GB300 at the 70B shapes, where the part is power-limited; kept as
 *       an option.
 * Every schedule gives the same results up to the order of fp32 summation
 * across K (0 and 3 sum in the same order).  The grouped GEMMs of the MoE
 * block are not affected.  Returns LLAMA_ERR_ARG for any other value. */
int llama_set_gemm_schedule(int schedule);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_LAYER_H_ */
