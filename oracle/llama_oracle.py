"""CPU oracle for the Llama decoder-layer forward over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers or tables) and it
does not import the ``llama_decoder_layer_gb300`` package.

It is deliberately plain and slow: NumPy arrays, one library matmul per
projection, explicit loops over sequences, tokens and heads for attention, and
no blocking, fusion or reordering beyond what the definitions state.  Floating
point runs in ``dtype`` (float64 by default, float32 for the large subsets)
over the exact bf16 input values.  The layer-level functions model the pages'
modules in the model's dtype (R3): every tensor a module returns is stored in
bf16 (``bf16_tensors=True``, the default there), while the arithmetic inside a
module is exact in ``dtype``.  ``bf16_tensors=False`` gives exact arithmetic
end to end (used by the pins of the mathematics).

Sources (three web pages on vLLM's ``llama.py``), cited below by tag:

* [LLAMA-70B]    page "LLama — DeepSeek-R1-Distill-Llama-70B" (hotelren.com
                 vLLM walk-through): the model config, §3 input_layernorm
                 (RMSNorm), §4 LlamaAttention, LlamaMLP / SiluAndMul, the final
                 RMSNorm and the Sampler.
* [WALKTHROUGH]  page "模型库与算子层 — 代码走读" (vllm-learning code
                 walkthrough): LlamaModel, LlamaDecoderLayer (unfused pre-norm
                 form), Attention (separate q/k/v, _update_kv_cache,
                 attn_backend with block_table), Linear layers (F.linear).
* [CODE-READING] page "vLLM Llama 代码解析" (yeyulingfeng.com): §1
                 LlamaForCausalLM (packed_modules_mapping, compute_logits),
                 §2.1 LlamaModel.forward (layer loop with residual, final
                 norm), §4 LlamaAttention (qkv split, RoPE on q/k only), §5
                 LlamaMLP.

Where the pages leave a step open, the reading taken is stated at the function
(readings R1..R20; the same numbering is used in the design notes).

Parity status of each function:

* rms_norm, fused_add_rms_norm, linear, silu_and_mul, paged_attention,
  kv_cache_write, slot_mapping, greedy_argmax: pinned (library special cases,
  closed forms, invariants and brute force in tests/test_oracle_pins.py).
* rope_inv_freq: the plain and llama3 band edges are pinned by closed forms; the
  interior of the llama3 smooth band follows the published Llama 3.1 rule only
  (the pages give the parameters, not the formula).
* apply_rope: norm preservation, relative-position dependence and the identity
  at position 0 are pinned; the rotate-half pairing itself is a reading (R4)
  that no invariant on the pages separates from the interleaved pairing:
  parity unpinned for the pairing choice.
* sample: pinned (argmax limits, inverse-CDF frequencies over a grid of
  draws, closed-form temperature and hand-worked top-k / top-p sets with ties,
  scipy's log_softmax for the logprob); R21..R25 are readings of a page that
  names the steps without their formulas.
* moe_route, moe_expert, moe_combine, moe_block: pinned (the page's worked
  combine example, a single expert with k = 1 equal to the dense MLP, expert
  relabelling invariance, weights summing to one, brute-force top-k);
  R26..R29 are readings of pages that name the steps without their
  precision.
* moe_decoder_layer: the decoder layer with the sparse MoE block in place of
  the dense MLP; pinned by its reduction to decoder_layer (one expert, k = 1,
  the dense MLP's weights), bit for bit.
* decoder_layer / stack_forward: compositions of the pinned parts, cross-checked
  against the unfused form and brute force; no value on the pages fixes an
  end-to-end number, so end-to-end parity beyond composition is unpinned.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# bf16 storage helpers (the cache's storage format; R11)
# ---------------------------------------------------------------------------


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and
    return the bit patterns as uint16.  NaN is not expected in this method."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Value of ``x`` after storage as bf16, returned as float32."""
    return bf16_bits_to_float(float_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def store(x, bf16_tensors: bool, dtype=np.float64):
    """A module's output tensor as the next module sees it.

    R3: [LLAMA-70B] config.json gives torch_dtype bfloat16, and in the pages'
    code each module call (the fused RMSNorm, qkv_proj, rotary_emb, attn,
    o_proj, gate_up_proj, the SiluAndMul act_fn, down_proj) returns a tensor of
    the model's dtype; so every module output is stored in bf16 (round to
    nearest even, through fp32)."""
    if not bf16_tensors:
        return x
    return round_to_bf16(np.asarray(x)).astype(dtype)


# ---------------------------------------------------------------------------
# Configuration
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class LayerShape:
    """Shape and constants of one decoder layer.

    [LLAMA-70B] config.json gives, for the 70B model: hidden_size 8192,
    num_attention_heads 64, num_key_value_heads 8, head_dim 128,
    intermediate_size 28672, rms_norm_eps 1e-5, rope_theta 500000 and the
    llama3 rope_scaling block; hidden_act "silu".
    """

    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    rms_eps: float
    rope_theta: float
    rope_scaling: Optional[dict] = None  # llama3 block or None
    block_size: int = 16
    hidden_act: str = "silu"

    @property
    def q_size(self) -> int:
        # [CODE-READING] §4: q_size / kv_size come from the head counts (GQA).
        return self.n_heads * self.head_dim

    @property
    def kv_size(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads


# ---------------------------------------------------------------------------
# Normalisation
# ---------------------------------------------------------------------------


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float, dtype=np.float64) -> np.ndarray:
    """RMSNorm over the last axis.

    R1 (the pages name RMSNorm but print no formula; [LLAMA-70B] §3): the
    standard definition  y = x / sqrt(mean(x^2) + eps) * gamma, with eps inside
    the square root and the mean over the hidden dimension.
    """
    x = np.asarray(x, dtype=dtype)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + dtype(eps)) * np.asarray(gamma, dtype=dtype)


def fused_add_rms_norm(x, residual, gamma, eps, dtype=np.float64, bf16_tensors=False):
    """The residual-fused RMSNorm of vLLM's decoder layer.

    [LLAMA-70B] §3 input_layernorm: when residual is None the residual becomes
    the (un-normed) input and the hidden states are normalised; otherwise the
    sum hidden + residual becomes the new residual and is normalised (R2).
    [CODE-READING] §4 uses the same call after attention
    (post_attention_layernorm) and §2.1 for the final norm.
    With ``bf16_tensors`` both outputs are stored in bf16 and the norm is taken
    of the stored residual (R3: the residual is a module output).
    Returns (normed, new_residual).
    """
    x = np.asarray(x, dtype=dtype)
    if residual is None:
        r = x.copy()
    else:
        r = x + np.asarray(residual, dtype=dtype)
    r = store(r, bf16_tensors, dtype)
    return store(rms_norm(r, gamma, eps, dtype), bf16_tensors, dtype), r


# ---------------------------------------------------------------------------
# Projections and the MLP activation
# ---------------------------------------------------------------------------


def linear(x, weight, dtype=np.float64):
    """y = x @ W^T with W stored [out, in].

    [WALKTHROUGH] Linear layers: every parallel linear holds
    ``Parameter(out, in)`` and calls ``F.linear(x, self.weight)``; with one GPU
    there is no all-reduce.
    """
    return np.asarray(x, dtype=dtype) @ np.asarray(weight, dtype=dtype).T


def silu(z, dtype=np.float64):
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=dtype)
    with np.errstate(over="ignore"):
        return z / (dtype(1.0) + np.exp(-z))


def silu_and_mul(x, dtype=np.float64):
    """[LLAMA-70B] LlamaMLP, SiluAndMul: x -> silu(x[:d]) * x[d:] with
    d = x.shape[-1] // 2, '*' the elementwise (Hadamard) product.  The first
    half is the gate (R15; also the [gate_proj, up_proj] packing order of
    [CODE-READING] §1)."""
    x = np.asarray(x, dtype=dtype)
    d = x.shape[-1] // 2
    return silu(x[..., :d], dtype) * x[..., d:]


# ---------------------------------------------------------------------------
# Rotary embedding
# ---------------------------------------------------------------------------


def rope_inv_freq(head_dim: int, theta: float, scaling: Optional[dict] = None) -> np.ndarray:
    """Per-pair inverse frequencies (float64), length head_dim // 2.

    R5: inv_freq_i = theta ** (-2 i / head_dim), i = 0 .. head_dim/2 - 1
    (only rope_theta is on the pages: [LLAMA-70B] config.json).

    R6: with rope_type "llama3" ([LLAMA-70B] config.json gives factor 8,
    low_freq_factor 1, high_freq_factor 4, original_max_position_embeddings
    8192 but not the rule) the published Llama 3.1 frequency rule is applied,
    stated from its mathematics: with wavelength lam = 2 pi / inv_freq,
      lam < orig / high          -> unchanged (high-frequency band)
      lam > orig / low           -> inv_freq / factor (low-frequency band)
      otherwise, s = (orig / lam - low) / (high - low), the blend
                 (1 - s) * inv_freq / factor + s * inv_freq.
    """
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv = float(theta) ** (-2.0 * i / head_dim)
    if scaling is None:
        return inv
    if scaling.get("rope_type", "llama3") != "llama3":
        raise ValueError("only llama3 rope scaling is defined")
    factor = float(scaling["factor"])
    low = float(scaling["low_freq_factor"])
    high = float(scaling["high_freq_factor"])
    orig = float(scaling["original_max_position_embeddings"])
    out = np.empty_like(inv)
    for j, f in enumerate(inv):
        lam = 2.0 * math.pi / f
        if lam < orig / high:
            out[j] = f
        elif lam > orig / low:
            out[j] = f / factor
        else:
            s = (orig / lam - low) / (high - low)
            out[j] = (1.0 - s) * f / factor + s * f
    return out


def apply_rope(x, positions, inv_freq, dtype=np.float64):
    """Rotate every head of ``x`` ([T, n_heads, head_dim]) by its token's
    position.

    [LLAMA-70B] §4 and [CODE-READING] §4: rotary_emb(positions, q, k) rotates
    q and k only; v is untouched.  R4: the rotate-half ("neox") pairing of
    element i with element i + head_dim/2, over the full head_dim.  Angles
    pos * inv_freq and their cos/sin are taken in float64.
    """
    x = np.asarray(x, dtype=dtype)
    T, nh, d = x.shape
    half = d // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * np.asarray(inv_freq, dtype=np.float64)[None, :]
    cos = np.cos(ang).astype(dtype)[:, None, :]
    sin = np.sin(ang).astype(dtype)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = x1 * cos - x2 * sin
    out[..., half:] = x2 * cos + x1 * sin
    return out


# ---------------------------------------------------------------------------
# Paged KV cache
# ---------------------------------------------------------------------------


def token_sequence(query_start_loc: Sequence[int]) -> np.ndarray:
    """Sequence index of every token of the flat batch."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    seq = np.empty(int(qsl[-1]), dtype=np.int64)
    for b in range(len(qsl) - 1):
        seq[qsl[b]:qsl[b + 1]] = b
    return seq


def slot_mapping(positions, query_start_loc, block_table, block_size: int) -> np.ndarray:
    """Cache slot of every token: block_table[b][pos // bs] * bs + pos % bs.

    [WALKTHROUGH] Attention: _update_kv_cache writes this step's k, v into the
    block-paged cache addressed through kv_cache.block_table (R11 layout).
    Integer arithmetic, exact.
    """
    seq = token_sequence(query_start_loc)
    bt = np.asarray(block_table, dtype=np.int64)
    out = np.empty(len(seq), dtype=np.int64)
    for t, (b, p) in enumerate(zip(seq, np.asarray(positions, dtype=np.int64))):
        out[t] = bt[b, p // block_size] * block_size + p % block_size
    return out


def kv_cache_write(k, v, slots, k_cache_bits, v_cache_bits, block_size: int) -> None:
    """Store k, v ([T, n_kv, d] values) into the caches in place.

    The caches hold bf16 bit patterns, laid out [num_blocks, n_kv, block_size,
    d] (R11).  A slot < 0 means "skip this token".  Values are rounded to bf16,
    the cache's storage type (R3, R11).
    """
    kb = float_to_bf16_bits(np.asarray(k, dtype=np.float32))
    vb = float_to_bf16_bits(np.asarray(v, dtype=np.float32))
    for t, s in enumerate(np.asarray(slots, dtype=np.int64)):
        if s < 0:
            continue
        blk, off = divmod(int(s), block_size)
        k_cache_bits[blk, :, off, :] = kb[t]
        v_cache_bits[blk, :, off, :] = vb[t]


def gather_kv(cache_bits, block_table_row, n_tokens: int, block_size: int) -> np.ndarray:
    """Read the first ``n_tokens`` cached tokens of one sequence through its
    block table: returns float32 [n_tokens, n_kv, d]."""
    out = []
    for j in range(n_tokens):
        blk = int(block_table_row[j // block_size])
        out.append(bf16_bits_to_float(cache_bits[blk, :, j % block_size, :]))
    if not out:
        return np.zeros((0,) + cache_bits.shape[1:2] + cache_bits.shape[3:], np.float32)
    return np.stack(out, axis=0)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------


def paged_attention(q, k_cache_bits, v_cache_bits, block_table, seq_lens, query_start_loc, positions,
                    n_kv_heads: int, block_size: int, rows: Optional[Sequence[int]] = None,
                    dtype=np.float64) -> np.ndarray:
    """Causal GQA attention of every selected token against its own sequence's
    paged cache.

    [WALKTHROUGH] Attention: attn_backend.forward(q, k, v, block_table, ...)
    after the cache update; [LLAMA-70B] config / §4: grouped-query attention
    (64 q heads share 8 kv heads).
    R7: scale 1 / sqrt(head_dim).  R8: q head h reads kv head h // (nq/nkv).
    R9: a token at position p sees cache positions 0..p of its sequence (the
    new tokens are already in the cache, so a token sees itself).
    Softmax subtracts the row maximum.  ``q`` is [T, nq, d]; the result is
    [T, nq, d] (rows not selected stay zero).
    """
    q = np.asarray(q, dtype=dtype)
    T, nq, d = q.shape
    g = nq // n_kv_heads
    scale = dtype(1.0 / math.sqrt(d))
    seq = token_sequence(query_start_loc)
    pos = np.asarray(positions, dtype=np.int64)
    out = np.zeros_like(q)
    wanted = range(T) if rows is None else rows
    cache_rows = {}
    for t in wanted:
        b = int(seq[t])
        if b not in cache_rows:
            n = int(seq_lens[b])
            cache_rows[b] = (gather_kv(k_cache_bits, block_table[b], n, block_size).astype(dtype),
                             gather_kv(v_cache_bits, block_table[b], n, block_size).astype(dtype))
        K, V = cache_rows[b]
        p = int(pos[t])
        for h in range(nq):
            kh = h // g
            s = (K[:p + 1, kh, :] @ q[t, h, :]) * scale
            w = np.exp(s - np.max(s))
            w = w / np.sum(w)
            out[t, h, :] = w @ V[:p + 1, kh, :]
    return out


# ---------------------------------------------------------------------------
# Decoder layer and stack
# ---------------------------------------------------------------------------


@dataclass
class LayerWeights:
    """Weights of one layer as float32 arrays holding exact bf16 values.

    w_qkv rows are [q; k; v] and w_gate_up rows are [gate; up]
    ([CODE-READING] §1 packed_modules_mapping); every projection is stored
    [out, in] ([WALKTHROUGH] Linear layers)."""

    ln1: np.ndarray
    w_qkv: np.ndarray
    w_o: np.ndarray
    ln2: np.ndarray
    w_gate_up: np.ndarray
    w_down: np.ndarray


@dataclass
class Batch:
    """Flat batch of tokens from many sequences ([CODE-READING] §2.1)."""

    positions: np.ndarray        # [T]
    query_start_loc: np.ndarray  # [B+1]
    seq_lens: np.ndarray         # [B], context including this step's tokens
    block_table: np.ndarray      # [B, max_blocks]


def attention_block(shape: LayerShape, w: LayerWeights, batch: Batch, h, k_cache_bits, v_cache_bits,
                    rows=None, dtype=np.float64, bf16_tensors=True):
    """LlamaAttention.forward: qkv_proj -> split -> rotary_emb -> attn -> o_proj.

    [LLAMA-70B] §4 / [CODE-READING] §4: one merged projection, split into
    [q_size, kv_size, kv_size]; RoPE on q and k; v untouched; the cache update
    precedes attention ([WALKTHROUGH] Attention).  K/V for every token are
    written; attention and o_proj are evaluated on ``rows`` (all if None).
    Module outputs (qkv, rotated q and k, attention output, o_proj output) are
    stored in bf16 when ``bf16_tensors`` (R3).
    Returns y [T, hidden] (zero outside ``rows``).
    """
    T = h.shape[0]
    qkv = store(linear(h, w.w_qkv, dtype), bf16_tensors, dtype)
    q = qkv[:, :shape.q_size].reshape(T, shape.n_heads, shape.head_dim)
    k = qkv[:, shape.q_size:shape.q_size + shape.kv_size].reshape(T, shape.n_kv_heads, shape.head_dim)
    v = qkv[:, shape.q_size + shape.kv_size:].reshape(T, shape.n_kv_heads, shape.head_dim)
    inv = rope_inv_freq(shape.head_dim, shape.rope_theta, shape.rope_scaling)
    q = store(apply_rope(q, batch.positions, inv, dtype), bf16_tensors, dtype)
    k = apply_rope(k, batch.positions, inv, dtype)
    slots = slot_mapping(batch.positions, batch.query_start_loc, batch.block_table, shape.block_size)
    kv_cache_write(k, v, slots, k_cache_bits, v_cache_bits, shape.block_size)
    o = paged_attention(q, k_cache_bits, v_cache_bits, batch.block_table, batch.seq_lens,
                        batch.query_start_loc, batch.positions, shape.n_kv_heads, shape.block_size,
                        rows=rows, dtype=dtype)
    y = np.zeros((T, shape.hidden), dtype=dtype)
    sel = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    o_sel = store(o[sel].reshape(len(sel), shape.q_size), bf16_tensors, dtype)
    y[sel] = store(linear(o_sel, w.w_o, dtype), bf16_tensors, dtype)
    return y


def mlp_block(shape: LayerShape, w: LayerWeights, h2, dtype=np.float64, bf16_tensors=True):
    """LlamaMLP.forward: gate_up_proj -> SiluAndMul -> down_proj.

    [LLAMA-70B] LlamaMLP: FFN(x) = down_proj(up_proj(x) * Act(gate_proj(x)))
    with Act = SiLU; any other activation is rejected.  [CODE-READING] §5.
    The three module outputs are stored in bf16 when ``bf16_tensors`` (R3).
    """
    if shape.hidden_act != "silu":
        raise ValueError(f"unsupported activation {shape.hidden_act}: only silu")
    gu = store(linear(h2, w.w_gate_up, dtype), bf16_tensors, dtype)
    a = store(silu_and_mul(gu, dtype), bf16_tensors, dtype)
    return store(linear(a, w.w_down, dtype), bf16_tensors, dtype)


def decoder_layer(shape: LayerShape, w: LayerWeights, batch: Batch, hidden, residual,
                  k_cache_bits, v_cache_bits, rows=None, dtype=np.float64, bf16_tensors=True):
    """One decoder layer: (hidden, residual) -> (hidden, residual).

    [CODE-READING] §2.1 / §3 / §4: input_layernorm (fused add) -> attention ->
    post_attention_layernorm (fused add) -> MLP; the residual is threaded out
    of the layer.  ``residual=None`` is the first layer ([LLAMA-70B] §3).
    The caches are updated in place for every token; the returned arrays are
    meaningful on ``rows`` (all rows if None).  ``bf16_tensors``: module
    outputs stored in bf16 (R3).
    """
    h, r = fused_add_rms_norm(hidden, residual, w.ln1, shape.rms_eps, dtype, bf16_tensors)
    y = attention_block(shape, w, batch, h, k_cache_bits, v_cache_bits, rows=rows, dtype=dtype,
                        bf16_tensors=bf16_tensors)
    sel = np.arange(h.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    h2, r2 = fused_add_rms_norm(y[sel], r[sel], w.ln2, shape.rms_eps, dtype, bf16_tensors)
    out = np.zeros_like(r)
    res = np.zeros_like(r)
    out[sel] = mlp_block(shape, w, h2, dtype, bf16_tensors)
    res[sel] = r2
    return out, res


def decoder_layer_unfused(shape: LayerShape, w: LayerWeights, batch: Batch, hidden,
                          k_cache_bits, v_cache_bits, dtype=np.float64):
    """The same layer in the pre-norm form with the residual kept inside.

    [WALKTHROUGH] LlamaDecoderLayer: residual = h; h = norm(h); h = attn(h);
    h = residual + h; residual = h; h = norm(h); h = mlp(h); h = residual + h.
    Used only as a cross-check of the fused form in exact arithmetic: for the
    same input (hidden + residual of the fused form) it returns out + residual.
    """
    x = np.asarray(hidden, dtype=dtype)
    a_in = rms_norm(x, w.ln1, shape.rms_eps, dtype)
    x = x + attention_block(shape, w, batch, a_in, k_cache_bits, v_cache_bits, dtype=dtype, bf16_tensors=False)
    m_in = rms_norm(x, w.ln2, shape.rms_eps, dtype)
    return x + mlp_block(shape, w, m_in, dtype, bf16_tensors=False)


def last_token_rows(query_start_loc) -> np.ndarray:
    """R13: logits are computed for the last token of every sequence
    ([CODE-READING] §1: compute_logits is separate from forward)."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    return qsl[1:] - 1


def greedy_argmax(logits):
    """[LLAMA-70B] Sampler: when every request is greedy, the sampled token is
    the argmax.  R14: ties go to the lowest index.  Returns (tokens, top-2
    gap) per row; the gap decides which rows a greedy comparison is defined
    on."""
    logits = np.asarray(logits)
    tok = np.argmax(logits, axis=-1)
    part = np.sort(logits, axis=-1)
    gap = part[..., -1] - part[..., -2]
    return tok.astype(np.int64), gap


# ---------------------------------------------------------------------------
# Sampler beyond greedy
# ---------------------------------------------------------------------------
GREEDY_TEMPERATURE = 1e-5  # R21


def sample(logits, temperature, top_k, top_p, uniform, dtype=np.float64):
    """[LLAMA-70B] Sampler, sample(): greedy rows take the argmax; the others
    are scaled by their temperature, cut by top-k and top-p, and drawn at
    random; logprobs are gathered from the raw log-softmax.  Readings:

    * R21: a row is greedy when its temperature is below 1e-5 (the page merges
      greedy results below a temperature threshold without giving it).
    * R22: top-k keeps every token whose logit is at least the k-th largest
      (ties at the boundary are kept); k <= 0 or k >= vocab keeps all.
    * R23: top-p, applied after top-k to the temperature-scaled probabilities,
      keeps every token whose probability is at least tau, the largest value
      for which the kept mass is >= p times the mass of the top-k set (ties
      kept); p >= 1 keeps all.
    * R24: the random draw is an input, one uniform u in [0, 1) per row: the
      token is the first kept token in index order at which the cumulative
      kept probability exceeds u times the total kept probability (inverse
      CDF).
    * R25: the returned logprob is the raw log-softmax of the unscaled logits
      at the sampled token (the page's raw_logprobs mode).

    Returns (tokens [B] int64, logprobs [B], margins [B]): a margin is the
    smaller of the distance of the draw u * total from the nearest CDF
    boundary (relative to the total) and the distance of the top-p target
    from the nearest cumulative sum of the sorted kept probabilities
    (relative to the top-k mass); inf for greedy rows.  It tells a comparison
    how close the integer decision was."""
    logits = np.asarray(logits, dtype=dtype)
    B, V = logits.shape
    tokens = np.empty(B, dtype=np.int64)
    logprobs = np.empty(B, dtype=dtype)
    margins = np.empty(B, dtype=dtype)
    for b in range(B):
        lrow = logits[b]
        lmax = lrow.max()
        log_z = lmax + np.log(np.sum(np.exp(lrow - lmax)))
        t = float(temperature[b])
        if t < GREEDY_TEMPERATURE:
            tok = int(np.argmax(lrow))
            margin = np.inf
        else:
            w = np.exp((lrow - lmax) / t)  # unnormalised tempered probabilities
            keep = np.ones(V, dtype=bool)
            k = int(top_k[b])
            if 0 < k < V:
                kth = np.sort(lrow)[V - k]
                keep &= lrow >= kth
            p = float(top_p[b])
            p_margin = np.inf
            if p < 1.0:
                mass_k = np.sum(w[keep])
                vals = np.sort(w[keep])[::-1]
                csum = np.cumsum(vals)
                idx = int(np.searchsorted(csum, p * mass_k, side="left"))
                tau = vals[min(idx, vals.size - 1)]
                keep &= w >= tau
                near = np.abs(csum - p * mass_k)
                p_margin = near.min() / mass_k if p > 0 else np.inf
            wk = np.where(keep, w, 0.0)
            c = np.cumsum(wk)
            total = c[-1]
            target = float(uniform[b]) * total
            tok = int(np.searchsorted(c, target, side="right"))
            lo = c[tok - 1] if tok > 0 else 0.0
            margin = min((c[tok] - target) / total, (target - lo) / total, p_margin)
        tokens[b] = tok
        logprobs[b] = lrow[tok] - log_z
        margins[b] = margin
    return tokens, logprobs, margins


# ---------------------------------------------------------------------------
# Sparse MoE block (Qwen3MoeSparseMoeBlock / FusedMoE)
# ---------------------------------------------------------------------------


def moe_route(router_logits, top_k: int):
    """[LLAMA-70B] Qwen3MoeSparseMoeBlock: the gate gives one logit per expert
    and every token picks its top-k experts; [WALKTHROUGH] FusedMoE:
    torch.topk(router_logits, top_k).  Readings:

    * R26: the router logits are the gate's fp32-accumulated outputs, kept in
      fp32 for routing (like the Sampler's logits.float()); ties between equal
      logits go to the lower expert index.
    * R27: norm_topk_prob (true in the page's config) renormalises the top-k
      probabilities to sum to one, i.e. the weights are the softmax of the k
      selected logits.

    Returns (ids [T, k] int64 in descending logit order, weights [T, k], gap
    [T]): gap is the distance between the k-th and (k+1)-th largest logits,
    which tells a comparison how close the expert choice was."""
    x = np.asarray(router_logits, dtype=np.float64)
    T, E = x.shape
    order = np.argsort(-x, axis=1, kind="stable")  # stable: equal logits keep index order
    ids = order[:, :top_k]
    sel = np.take_along_axis(x, ids, axis=1)
    w = np.exp(sel - sel[:, :1])
    w = w / w.sum(axis=1, keepdims=True)
    if top_k < E:
        nxt = np.take_along_axis(x, order[:, top_k:top_k + 1], axis=1)[:, 0]
        gap = sel[:, -1] - nxt
    else:
        gap = np.full(T, np.inf)
    return ids.astype(np.int64), w, gap


def moe_expert(x, w13_e, w2_e, dtype=np.float64, bf16_tensors=True):
    """One expert: a two-layer FFN with SiluAndMul, w13_e [2I, H] holding the
    gate rows then the up rows ([WALKTHROUGH] FusedMoE w13 / w2; [LLAMA-70B]
    每个专家是双层FFN 2048 -> 768 -> 2048).  R28: as for the dense MLP (R3) the
    merged projection, SiluAndMul and the expert output are stored in bf16."""
    gu = store(linear(x, w13_e, dtype), bf16_tensors, dtype)
    act = store(silu_and_mul(gu, dtype), bf16_tensors, dtype)
    return store(linear(act, w2_e, dtype), bf16_tensors, dtype)


def moe_combine(expert_outputs, weights, dtype=np.float64):
    """[LLAMA-70B] the token's MoE output is the sum of its experts' outputs,
    each multiplied by its routing weight.  R29: the sum runs in ``dtype``
    over the k experts in routing order."""
    out = np.zeros_like(np.asarray(expert_outputs[0], dtype=dtype))
    for y, w in zip(expert_outputs, weights):
        out = out + np.asarray(w, dtype=dtype) * np.asarray(y, dtype=dtype)
    return out


def moe_block(h, w_router, w13, w2, top_k: int, dtype=np.float64, bf16_tensors=True):
    """Qwen3MoeSparseMoeBlock forward over tokens h [T, H]: router logits
    (R26), top-k routing with renormalised weights (R27), the selected experts
    (R28) and the weighted sum (R29), no shared expert; the block's output is
    stored in bf16 (R3).  w_router [E, H], w13 [E, 2I, H], w2 [E, H, I].
    Returns (out [T, H], ids, weights, gap)."""
    h = np.asarray(h, dtype=dtype)
    logits = linear(h, w_router, dtype)
    ids, wts, gap = moe_route(logits, top_k)
    T = h.shape[0]
    out = np.zeros((T, np.asarray(w2).shape[1]), dtype=dtype)
    for t in range(T):
        ys = [moe_expert(h[t:t + 1], w13[e], w2[e], dtype, bf16_tensors)[0] for e in ids[t]]
        out[t] = moe_combine(ys, wts[t], dtype)
    return store(out, bf16_tensors, dtype), ids, wts, gap


def moe_decoder_layer(shape: LayerShape, w: LayerWeights, w_router, w13, w2, top_k: int, batch: Batch, hidden,
                      residual, k_cache_bits, v_cache_bits, rows=None, dtype=np.float64, bf16_tensors=True):
    """A Qwen3-MoE decoder layer as the pages describe it: the Llama layer's
    input_layernorm, attention and post_attention_layernorm, then the sparse
    MoE block ([LLAMA-70B] Qwen3MoeSparseMoeBlock, decoder_sparse_step 1 and
    no mlp_only_layers: every layer is sparse) where the dense MLP was.  The
    pages describe no other difference (R30).  ``w`` supplies ln1, w_qkv, w_o
    and ln2; its MLP weights are unused.  Returns (hidden, residual, expert
    ids, top-k gap) on ``rows`` (all rows if None)."""
    h, r = fused_add_rms_norm(hidden, residual, w.ln1, shape.rms_eps, dtype, bf16_tensors)
    y = attention_block(shape, w, batch, h, k_cache_bits, v_cache_bits, rows=rows, dtype=dtype,
                        bf16_tensors=bf16_tensors)
    sel = np.arange(h.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    h2, r2 = fused_add_rms_norm(y[sel], r[sel], w.ln2, shape.rms_eps, dtype, bf16_tensors)
    out = np.zeros_like(r)
    res = np.zeros_like(r)
    moe_out, ids, _, gap = moe_block(h2, w_router, w13, w2, top_k, dtype, bf16_tensors)
    out[sel] = moe_out
    res[sel] = r2
    ids_all = np.full((h.shape[0], top_k), -1, dtype=np.int64)
    gap_all = np.full(h.shape[0], np.nan)
    ids_all[sel] = ids
    gap_all[sel] = gap
    return out, res, ids_all, gap_all


def stack_forward(shape: LayerShape, layers: Sequence[LayerWeights], final_norm, lm_head, batch: Batch,
                  hidden, k_caches, v_caches, dtype=np.float64, bf16_tensors=True):
    """The model body and head over one flat batch.

    [CODE-READING] §2.1: for layer in layers: hidden, residual =
    layer(positions, hidden, residual), starting from residual None, then
    hidden, _ = norm(hidden, residual); [LLAMA-70B] final RMSNorm and Sampler;
    R13 logits only for the last row of each sequence.  Logits are kept in
    ``dtype`` (the Sampler works on logits.float()).
    Returns (tokens, top-2 gap, logits [B, vocab], final normed rows [B, H]).
    """
    x = np.asarray(hidden, dtype=dtype)
    r = None
    for li, w in enumerate(layers):
        x, r = decoder_layer(shape, w, batch, x, r, k_caches[li], v_caches[li], dtype=dtype,
                             bf16_tensors=bf16_tensors)
    sel = last_token_rows(batch.query_start_loc)
    hf, _ = fused_add_rms_norm(x[sel], r[sel], final_norm, shape.rms_eps, dtype, bf16_tensors)
    logits = linear(hf, lm_head, dtype)
    tok, gap = greedy_argmax(logits)
    return tok, gap, logits, hf


def embed(embedding, input_ids):
    """[WALKTHROUGH] LlamaModel / [CODE-READING] §2: input_ids become vectors
    by a row lookup of the embedding table (one GPU: no vocabulary shards)."""
    return np.asarray(embedding)[np.asarray(input_ids, dtype=np.int64)]
