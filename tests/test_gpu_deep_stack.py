"""The full-depth stack (GPU): 80 decoder layers, the depth of the 70B model
([LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B", config.json: 80 hidden
layers), through one llama_stack_forward call with embedding, final norm,
lm_head and greedy argmax ([CODE-READING] "vLLM Llama 代码解析" §2.1, the layer
loop with the residual threaded from None), on the tiny layer shape so the
oracle can follow it.  Every layer has its own weights and KV cache; the batch
mixes decode sequences with prefill chunks, one on a cached prefix.

Pinned as the 8-layer stack is:
(a) the eager call equals its composition (80 layer calls, the final norm of
    each sequence's last row and lm_head) bit for bit: tokens, logits, caches;
(b) the call captured in a CUDA graph and replayed equals the eager call bit
    for bit;
(c) seeded layers (the first, the second, two in the middle, the last) match
    the oracle given that layer's inputs;
(d) the head matches the oracle given the final hidden and residual rows of
    every sequence: logits within tolerance, greedy tokens identical wherever
    the oracle's top-2 gap exceeds 0.05.
"""

import dataclasses

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O
from tests.helpers import SubBatch, assert_close, bits, f32, oracle_shape, oracle_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"
NL = 80


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


def test_80_layer_stack_eager_graph_composition_and_oracle():
    spec = dataclasses.replace(I.SPECS["tiny"], num_layers=NL, vocab=4096, residual_none=True,
                               rope_theta=500000.0, rope_scaling=I.LLAMA3_SCALING,
                               groups=(("decode", 6, 1, 64, 3500), ("prefill", 1, 40, 0, 0),
                                       ("prefill", 1, 24, 50, 50)))
    bl = I.make_batch(spec, 5, DEV)
    layers = [I.make_layer_weights(spec, 5, l, DEV) for l in range(NL)]
    caches0 = [I.make_kv_cache(spec, bl.num_blocks, 5, l, DEV) for l in range(NL)]
    emb, ids, lm, fn = I.make_stack_extras(spec, bl.num_tokens, 5, DEV)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    T, B = bl.num_tokens, bl.num_seqs
    ws = lb.alloc_workspace(lb.workspace_size(cfg, T, B, batch.max_seq_len, spec.vocab), DEV)
    hidden = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device=DEV)
    residual = torch.empty_like(hidden)
    tokens = torch.empty(B, dtype=torch.int32, device=DEV)
    logits = torch.empty((B, spec.vocab), dtype=torch.float32, device=DEV)
    caches = [(k.clone(), v.clone()) for k, v in caches0]

    def reset():
        for (k, v), (k0, v0) in zip(caches, caches0):
            k.copy_(k0)
            v.copy_(v0)
        tokens.fill_(-1)
        logits.zero_()
        hidden.zero_()
        residual.zero_()

    def call(stream):
        lb.stack_forward(cfg, layers, fn, lm, batch, hidden, residual, [c[0] for c in caches],
                         [c[1] for c in caches], tokens, ws, embed=emb, input_ids=ids, out_logits=logits,
                         stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        reset()
        call(s)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    eager = (tokens.clone(), logits.clone(), hidden.clone(), residual.clone(),
             [(k.clone(), v.clone()) for k, v in caches])

    # (b) the same call from a CUDA graph
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    torch.cuda.synchronize()
    reset()
    g.replay()
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    assert torch.equal(tokens, eager[0]) and torch.equal(logits, eager[1]), "graph replay: head differs"
    assert torch.equal(hidden, eager[2]) and torch.equal(residual, eager[3]), "graph replay: hidden differs"
    for l, ((k, v), (ke, ve)) in enumerate(zip(caches, eager[4])):
        assert torch.equal(k.view(torch.int16), ke.view(torch.int16)), f"graph replay: layer {l} k cache"
        assert torch.equal(v.view(torch.int16), ve.view(torch.int16)), f"graph replay: layer {l} v cache"
    del g

    # (a) the composition, keeping every layer's inputs
    comp = [(k.clone(), v.clone()) for k, v in caches0]
    h2 = emb[ids.long()].contiguous()
    r2 = torch.empty_like(h2)
    layer_in = []
    for l in range(NL):
        layer_in.append((f32(h2), None if l == 0 else f32(r2)))
        lb.layer_forward(cfg, layers[l], batch, h2, None if l == 0 else r2, r2, comp[l][0], comp[l][1], ws)
    last = bl.query_start_loc[1:].long() - 1
    hf = torch.empty((B, spec.hidden), dtype=torch.bfloat16, device=DEV)
    lb.fused_add_rmsnorm(h2[last].contiguous(), r2[last].contiguous(), None, hf, fn, spec.rms_eps)
    logits2 = torch.empty_like(logits)
    lb.linear(hf, lm, logits2, lb.alloc_workspace(lb.linear_workspace_size(), DEV))
    torch.cuda.synchronize()
    assert torch.equal(eager[2], h2) and torch.equal(eager[3], r2), "stack differs from its layer composition"
    assert torch.equal(eager[1], logits2), "stack logits differ from the composition's"
    for l in range(NL):
        assert torch.equal(eager[4][l][0].view(torch.int16), comp[l][0].view(torch.int16)), f"layer {l} k cache"
        assert torch.equal(eager[4][l][1].view(torch.int16), comp[l][1].view(torch.int16)), f"layer {l} v cache"

    # (c) seeded layers against the oracle on their own inputs
    sh = oracle_shape(spec)
    everyone = list(range(B))
    for l in (0, 1, 39, 40, NL - 1):
        sub = SubBatch(bl, everyone, caches0[l][0], caches0[l][1])
        kref, vref = sub.kc.copy(), sub.vc.copy()
        xo, ro = O.decoder_layer(sh, oracle_weights(layers[l]), sub.batch, layer_in[l][0], layer_in[l][1], kref,
                                 vref)
        after = layer_in[l + 1] if l + 1 < NL else (f32(eager[2]), f32(eager[3]))
        eh = assert_close(after[0], xo, f"layer {l} hidden (same inputs)")
        er = assert_close(after[1], ro, f"layer {l} residual (same inputs)")
        ek = assert_close(O.bf16_bits_to_float(sub.gpu_written(bits(eager[4][l][0]))),
                          O.bf16_bits_to_float(sub.oracle_written(kref)), f"layer {l} k written")
        print(f"deep stack layer {l}: same-input rel err hidden {eh:.2e} residual {er:.2e} k {ek:.2e}")

    # (d) the head on every sequence's final rows
    lrows = last.cpu().numpy()
    hf_ref, _ = O.fused_add_rms_norm(f32(eager[2])[lrows], f32(eager[3])[lrows], f32(fn), sh.rms_eps,
                                     bf16_tensors=True)
    ref_logits = O.linear(hf_ref, f32(lm))
    ref_tok, gap = O.greedy_argmax(ref_logits)
    e = assert_close(f32(eager[1]), ref_logits, "deep stack logits")
    tok = eager[0].cpu().numpy()
    decided = gap > 0.05
    assert np.array_equal(tok[decided], ref_tok[decided]), f"greedy tokens differ: {tok} vs {ref_tok}"
    assert np.array_equal(tok, np.argmax(f32(eager[1]), axis=-1))
    print(f"deep stack head: logits rel err {e:.2e}, tokens compared on {int(decided.sum())}/{B} rows")
