"""How far two equally valid evaluations of the stack drift apart with depth
(CPU, no GPU).

The stack threads hidden_states and residual through its layers
([CODE-READING] "vLLM Llama 代码解析" §2.1, the layer loop), and every module
output is a bf16 tensor (the model's dtype, [LLAMA-70B] "LLama —
DeepSeek-R1-Distill-Llama-70B" config.json).  A tiny difference in how a
module accumulates (fp32 against fp64 here, or the tensor cores' order on the
GPU) moves some outputs across a bf16 rounding boundary; the next layers carry
that one-ulp change forward and it grows with depth.

These tests pin that behaviour with two oracles that differ only in the
precision of their accumulation, on an 8-layer stack of the 70B layer's
structure at hidden 4096 (32 q heads / 4 KV heads x 128, intermediate 14336,
llama3 RoPE), 4 decode sequences and one 256-token prefill chunk:

* given the same inputs, one layer of the two agrees far inside the 2e-2
  bar (the teacher-forced comparison the GPU tests make per layer);
* run free through 8 layers, the two exceed the 2e-2 bar.

So a free-running comparison of the 8-layer stack against the oracle cannot be
held to the per-tensor bar by any implementation, the oracle's own fp32 mode
included; the stack is checked by its composition (bit for bit), per layer on
each layer's inputs, and by the head on its inputs.
"""

import dataclasses

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O

TOL = 2e-2
NL = 8


def _f32(t):
    return t.float().numpy()


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rel(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - b)) / np.max(np.abs(b)))


@pytest.fixture(scope="module")
def drift():
    spec = dataclasses.replace(I.SPECS["stack_70b"], name="stack_h4096", hidden=4096, n_heads=32, n_kv_heads=4,
                               intermediate=14336, vocab=0,
                               groups=(("decode", 4, 1, 256, 2048), ("prefill", 1, 256, 0, 0)))
    bl = I.make_batch(spec, 0)
    sh = O.LayerShape(spec.hidden, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.intermediate, spec.rms_eps,
                      spec.rope_theta, spec.rope_scaling, spec.block_size)
    ob = O.Batch(bl.positions.numpy().astype(np.int64), bl.query_start_loc.numpy().astype(np.int64),
                 bl.seq_lens.numpy().astype(np.int64), bl.block_table.numpy().astype(np.int64))
    x0 = _f32(I.normal_bf16((bl.num_tokens, spec.hidden), 1.0, 0.0, 5, "cpu"))
    x32, r32, x64, r64 = x0, None, x0, None
    same_input, free = [], []
    for layer in range(NL):
        w = I.make_layer_weights(spec, 0, layer)
        ow = O.LayerWeights(*(_f32(w[k]) for k in ("ln1", "w_qkv", "w_o", "ln2", "w_gate_up", "w_down")))
        kc, vc = I.make_kv_cache(spec, bl.num_blocks, 0, layer)
        kb, vb = _bits(kc), _bits(vc)
        # the fp64 evaluation carries the stack; the fp32 one runs once on its
        # inputs (teacher forced) and once on its own previous outputs (free)
        t32, tr32 = O.decoder_layer(sh, ow, ob, x64, r64, kb.copy(), vb.copy(), dtype=np.float32)
        x32, r32 = O.decoder_layer(sh, ow, ob, x32, r32, kb.copy(), vb.copy(), dtype=np.float32)
        x64, r64 = O.decoder_layer(sh, ow, ob, x64, r64, kb.copy(), vb.copy(), dtype=np.float64)
        same_input.append(max(_rel(t32, x64), _rel(tr32, r64)))
        free.append(max(_rel(x32, x64), _rel(r32, r64)))
    return same_input, free


def test_same_inputs_one_layer_within_the_bar(drift):
    same_input, _ = drift
    print("fp32 vs fp64, same inputs, per layer:", " ".join(f"{e:.2e}" for e in same_input))
    assert max(same_input) < TOL / 2


def test_free_running_exceeds_the_bar_by_depth_8(drift):
    same_input, free = drift
    print("fp32 vs fp64, free running, per layer:", " ".join(f"{e:.2e}" for e in free))
    assert free[0] < TOL / 2, "one layer from the same input must agree well inside the bar"
    assert max(free) > TOL, "the two evaluations were expected to drift past the bar within 8 layers"
    # the drift is the depth, not a single bad layer: it grows past what any
    # one layer contributes
    assert max(free[NL // 2:]) > 2 * max(same_input[:1])
