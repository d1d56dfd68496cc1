"""Seeded synthetic workloads for the Llama decoder-layer forward.

This module only draws numbers and lays out batch structure (sequence lengths,
positions, shuffled block tables); it holds none of the layer's arithmetic, so
both the CUDA path and the CPU oracle can take their inputs from it.

Workloads (all sizes as the layer sees them):

* ``tiny``        hidden 512, 8 q heads x 64, 2 kv heads, intermediate 1376,
                  theta 1e4 unscaled; 2 sequences x 32 prefill tokens,
                  residual None.
* ``decode_8b``   Llama-3-8B shape (4096, 32/8 x 128, 14336, theta 5e5, no
                  scaling); 64 sequences x 1 new token, 2048 cached tokens each.
* ``decode_70b``  70B shape (8192, 64/8 x 128, 28672, llama3 scaling);
                  128 sequences x 1 new token, cached context uniform in
                  [512, 8192].
* ``prefill_70b`` 70B shape; 8 sequences x 4096 prefill tokens at positions
                  0..4095 into an empty cache; residual ~N(0,1).
* ``stack_70b``   8 layers of the 70B shape + final norm + lm_head (vocab
                  128256) + greedy argmax; 32 decode sequences (context uniform
                  in [1024, 16384]) then 2 prefill chunks of 2048 tokens.
* ``small_mixed`` hidden 1024, 8 q heads x 128, 2 kv heads, intermediate
                  2048, llama3 scaling; 3 decode sequences (context uniform in
                  [1500, 2100], one or two split-KV chunks) and one 80-token
                  prefill chunk after a 32-token cached prefix: the head_dim-128
                  kernels of every path at a size the oracle runs in seconds.

Value recipe: projection, lm_head weights ~N(0, 0.02) in bf16; norm weights
1 + N(0, 0.02) (the reading that keeps the norms' scale); hidden states,
residuals, embeddings and prior cache contents ~N(0, 1) in bf16.  Every tensor
has its own seed offset so a tensor's values do not depend on which others are
drawn.  Block tables are a seeded random permutation of the physical blocks,
with a few spare blocks no sequence owns (they must stay untouched).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

BLOCK = 16

LLAMA3_SCALING = {
    "rope_type": "llama3",
    "factor": 8.0,
    "low_freq_factor": 1.0,
    "high_freq_factor": 4.0,
    "original_max_position_embeddings": 8192,
}


@dataclass(frozen=True)
class Spec:
    name: str
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    rms_eps: float
    rope_theta: float
    rope_scaling: Optional[dict]
    # batch structure: list of (kind, count, new_tokens, ctx_lo, ctx_hi)
    #   kind "decode": new_tokens=1 at position ctx, ctx ~ U[ctx_lo, ctx_hi]
    #   kind "prefill": new_tokens tokens at positions ctx..ctx+new-1
    groups: tuple
    residual_none: bool = False
    num_layers: int = 1
    vocab: int = 0
    block_size: int = BLOCK
    spare_blocks: int = 8
    literal_gamma: bool = False
    extra: dict = field(default_factory=dict)


SPECS = {
    "tiny": Spec("tiny", 512, 8, 2, 64, 1376, 1e-5, 10000.0, None,
                 groups=(("prefill", 2, 32, 0, 0),), residual_none=True),
    "small_mixed": Spec("small_mixed", 1024, 8, 2, 128, 2048, 1e-5, 500000.0, LLAMA3_SCALING,
                        groups=(("decode", 3, 1, 1500, 2100), ("prefill", 1, 80, 32, 32))),
    "decode_8b": Spec("decode_8b", 4096, 32, 8, 128, 14336, 1e-5, 500000.0, None,
                      groups=(("decode", 64, 1, 2048, 2048),)),
    "decode_70b": Spec("decode_70b", 8192, 64, 8, 128, 28672, 1e-5, 500000.0, LLAMA3_SCALING,
                       groups=(("decode", 128, 1, 512, 8192),)),
    "prefill_70b": Spec("prefill_70b", 8192, 64, 8, 128, 28672, 1e-5, 500000.0, LLAMA3_SCALING,
                        groups=(("prefill", 8, 4096, 0, 0),)),
    "stack_70b": Spec("stack_70b", 8192, 64, 8, 128, 28672, 1e-5, 500000.0, LLAMA3_SCALING,
                      groups=(("decode", 32, 1, 1024, 16384), ("prefill", 2, 2048, 0, 0)),
                      residual_none=True, num_layers=8, vocab=128256),
    # the full-depth 70B decode step (all 80 layers, embedding to sampled
    # token) at a batch that fits one GPU next to 137 GB of layer weights
    "decode_70b_80l": Spec("decode_70b_80l", 8192, 64, 8, 128, 28672, 1e-5, 500000.0, LLAMA3_SCALING,
                           groups=(("decode", 64, 1, 512, 4096),), residual_none=True, num_layers=80,
                           vocab=128256),
    # Qwen3-30B-A3B (Qwen3MoeForCausalLM config): hidden 2048, 32 q heads, 4 KV
    # heads, head_dim 128, rms_eps 1e-6, rope_theta 1e7 without scaling,
    # 128 experts, top-8, moe_intermediate 768 (intermediate_size 6144 is the
    # dense size, unused: every layer is sparse)
    "qwen3_moe": Spec("qwen3_moe", 2048, 32, 4, 128, 6144, 1e-6, 10000000.0, None,
                      groups=(("decode", 16, 1, 512, 4096), ("prefill", 1, 256, 0, 0)),
                      extra={"num_experts": 128, "top_k": 8, "moe_intermediate": 768}),
    "qwen3_moe_decode": Spec("qwen3_moe_decode", 2048, 32, 4, 128, 6144, 1e-6, 10000000.0, None,
                             groups=(("decode", 64, 1, 512, 4096),),
                             extra={"num_experts": 128, "top_k": 8, "moe_intermediate": 768}),
    "qwen3_moe_prefill": Spec("qwen3_moe_prefill", 2048, 32, 4, 128, 6144, 1e-6, 10000000.0, None,
                              groups=(("prefill", 4, 2048, 0, 0),),
                              extra={"num_experts": 128, "top_k": 8, "moe_intermediate": 768}),
}

# seed offsets per tensor kind
_OFF = {"ln1": 1, "w_qkv": 2, "w_o": 3, "ln2": 4, "w_gate_up": 5, "w_down": 6, "w_router": 7, "w13": 8, "w2": 9,
        "hidden": 20, "residual": 21, "k_cache": 22, "v_cache": 23, "ctx": 24, "perm": 25,
        "embed": 30, "ids": 31, "lm_head": 32, "final_norm": 33}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal_bf16(shape, std: float, mean: float, seed: int, device) -> torch.Tensor:
    """N(mean, std^2) drawn in fp32 with a seeded generator, rounded to bf16."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def make_layer_weights(spec: Spec, seed: int = 0, layer: int = 0, device="cpu") -> dict:
    """bf16 weights of one layer, [out, in] row-major; qkv rows [q; k; v],
    gate_up rows [gate; up]."""
    base = seed * 1000003 + layer * 101
    H, d = spec.hidden, spec.head_dim
    nqkv = (spec.n_heads + 2 * spec.n_kv_heads) * d
    gmean = 0.0 if spec.literal_gamma else 1.0
    return {
        "ln1": normal_bf16((H,), 0.02, gmean, base + _OFF["ln1"], device),
        "w_qkv": normal_bf16((nqkv, H), 0.02, 0.0, base + _OFF["w_qkv"], device),
        "w_o": normal_bf16((H, spec.n_heads * d), 0.02, 0.0, base + _OFF["w_o"], device),
        "ln2": normal_bf16((H,), 0.02, gmean, base + _OFF["ln2"], device),
        "w_gate_up": normal_bf16((2 * spec.intermediate, H), 0.02, 0.0, base + _OFF["w_gate_up"], device),
        "w_down": normal_bf16((H, spec.intermediate), 0.02, 0.0, base + _OFF["w_down"], device),
    }


def make_moe_layer_weights(spec: Spec, seed: int = 0, layer: int = 0, device="cpu") -> dict:
    """bf16 weights of one Qwen3-MoE layer: the attention half of
    make_layer_weights plus w_router [E, H], w13 [E, 2I, H] (gate rows then
    up rows per expert) and w2 [E, H, I], all N(0, 0.02)."""
    base = seed * 1000003 + layer * 101
    H, d = spec.hidden, spec.head_dim
    E, Im = spec.extra["num_experts"], spec.extra["moe_intermediate"]
    nqkv = (spec.n_heads + 2 * spec.n_kv_heads) * d
    gmean = 0.0 if spec.literal_gamma else 1.0
    return {
        "ln1": normal_bf16((H,), 0.02, gmean, base + _OFF["ln1"], device),
        "w_qkv": normal_bf16((nqkv, H), 0.02, 0.0, base + _OFF["w_qkv"], device),
        "w_o": normal_bf16((H, spec.n_heads * d), 0.02, 0.0, base + _OFF["w_o"], device),
        "ln2": normal_bf16((H,), 0.02, gmean, base + _OFF["ln2"], device),
        "w_router": normal_bf16((E, H), 0.02, 0.0, base + _OFF["w_router"], device),
        "w13": normal_bf16((E, 2 * Im, H), 0.02, 0.0, base + _OFF["w13"], device),
        "w2": normal_bf16((E, H, Im), 0.02, 0.0, base + _OFF["w2"], device),
    }


@dataclass
class BatchLayout:
    """Batch structure on the host (python ints / int lists) plus device copies."""

    positions: torch.Tensor        # int32 [T]
    query_start_loc: torch.Tensor  # int32 [B+1]
    seq_lens: torch.Tensor         # int32 [B]
    block_table: torch.Tensor      # int32 [B, max_blocks]; unused entries -1
    num_tokens: int
    num_seqs: int
    max_blocks_per_seq: int
    num_blocks: int
    q_lens: list
    ctx_lens: list                 # cached tokens before this step


def make_batch(spec: Spec, seed: int = 0, device="cpu") -> BatchLayout:
    """Flat batch: sequences in the order of ``spec.groups``.  Decode
    sequences get one new token at position ctx (ctx cached tokens before it);
    prefill sequences get their tokens at positions ctx..ctx+n-1."""
    g = _gen("cpu", seed * 7919 + _OFF["ctx"])
    q_lens, ctx_lens = [], []
    for kind, count, new, lo, hi in spec.groups:
        for _ in range(count):
            ctx = int(torch.randint(lo, hi + 1, (1,), generator=g).item()) if hi > lo else int(lo)
            q_lens.append(int(new))
            ctx_lens.append(ctx)
    B = len(q_lens)
    bs = spec.block_size
    seq_lens = [c + q for c, q in zip(ctx_lens, q_lens)]
    nblk = [(s + bs - 1) // bs for s in seq_lens]
    used = sum(nblk)
    num_blocks = used + spec.spare_blocks
    perm = torch.randperm(num_blocks, generator=_gen("cpu", seed * 7919 + _OFF["perm"]))
    maxb = max(nblk)
    bt = torch.full((B, maxb), -1, dtype=torch.int32)
    cur = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[cur:cur + nblk[b]].to(torch.int32)
        cur += nblk[b]
    positions, qsl = [], [0]
    for c, q in zip(ctx_lens, q_lens):
        positions.extend(range(c, c + q))
        qsl.append(qsl[-1] + q)
    return BatchLayout(
        positions=torch.tensor(positions, dtype=torch.int32, device=device),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32, device=device),
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
        block_table=bt.to(device),
        num_tokens=qsl[-1], num_seqs=B, max_blocks_per_seq=maxb, num_blocks=num_blocks,
        q_lens=q_lens, ctx_lens=ctx_lens)


def make_activations(spec: Spec, num_tokens: int, seed: int = 0, device="cpu"):
    """hidden_states and residual (None when the workload starts a stack)."""
    H = spec.hidden
    x = normal_bf16((num_tokens, H), 1.0, 0.0, seed * 31 + _OFF["hidden"], device)
    r = None if spec.residual_none else normal_bf16((num_tokens, H), 1.0, 0.0, seed * 31 + _OFF["residual"], device)
    return x, r


def make_kv_cache(spec: Spec, num_blocks: int, seed: int = 0, layer: int = 0, device="cpu"):
    """K and V caches [num_blocks, n_kv, block, head_dim] bf16 ~N(0,1): the
    prior context of decode sequences (slots a step writes are overwritten)."""
    shape = (num_blocks, spec.n_kv_heads, spec.block_size, spec.head_dim)
    base = seed * 1000003 + layer * 101
    return (normal_bf16(shape, 1.0, 0.0, base + _OFF["k_cache"], device),
            normal_bf16(shape, 1.0, 0.0, base + _OFF["v_cache"], device))


def make_stack_extras(spec: Spec, num_tokens: int, seed: int = 0, device="cpu"):
    """Embedding table ~N(0,1), token ids uniform in [0, vocab), lm_head
    ~N(0,0.02) and the final norm weight."""
    V, H = spec.vocab, spec.hidden
    gmean = 0.0 if spec.literal_gamma else 1.0
    emb = normal_bf16((V, H), 1.0, 0.0, seed * 31 + _OFF["embed"], device)
    ids = torch.randint(0, V, (num_tokens,), generator=_gen("cpu", seed * 31 + _OFF["ids"]),
                        dtype=torch.int64).to(torch.int32).to(device)
    lm = normal_bf16((V, H), 0.02, 0.0, seed * 31 + _OFF["lm_head"], device)
    fn = normal_bf16((H,), 0.02, gmean, seed * 31 + _OFF["final_norm"], device)
    return emb, ids, lm, fn


def random_slots(num_tokens: int, num_blocks: int, block_size: int, seed: int = 0, skip_every: int = 0):
    """Distinct random cache slots (int32) for standalone cache-write tests;
    every ``skip_every``-th token gets -1 (skip)."""
    perm = torch.randperm(num_blocks * block_size, generator=_gen("cpu", seed * 17 + 5))[:num_tokens]
    s = perm.to(torch.int32)
    if skip_every:
        s[::skip_every] = -1
    return s
