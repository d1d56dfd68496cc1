"""The layer call captured in a CUDA graph and replayed.

The call must be capture-safe: lazy set-up happens on the first (eager)
calls, and a batch with prefill sequences forks the decode kernels onto the
library's side stream and joins it again, which the capture turns into graph
edges.  Every reduction in the layer has a fixed order, so the replay must
reproduce the eager result bit for bit (hidden states, residual and the
written cache)."""

import dataclasses

import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


@pytest.mark.parametrize("name,groups", [
    ("tiny", (("prefill", 2, 24, 0, 0), ("decode", 3, 1, 40, 2000), ("prefill", 1, 9, 30, 30))),  # mixed: side stream
    ("decode_8b", (("decode", 16, 1, 100, 3000),)),                                                  # cluster split-K
])
def test_layer_graph_replay_matches_eager(name, groups):
    spec = dataclasses.replace(I.SPECS[name], groups=groups)
    bl = I.make_batch(spec, 7, DEV)
    w = I.make_layer_weights(spec, 7, 0, DEV)
    x, r = I.make_activations(spec, bl.num_tokens, 7, DEV)
    kc0, vc0 = I.make_kv_cache(spec, bl.num_blocks, 7, 0, DEV)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), DEV)
    hidden, res_out = x.clone(), torch.empty_like(x)
    kc, vc = kc0.clone(), vc0.clone()

    def reset():
        hidden.copy_(x)
        kc.copy_(kc0)
        vc.copy_(vc0)
        res_out.zero_()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        reset()
        lb.layer_forward(cfg, w, batch, hidden, r, res_out, kc, vc, ws, stream=s)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    eager = (hidden.clone(), res_out.clone(), kc.clone(), vc.clone())

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lb.layer_forward(cfg, w, batch, hidden, r, res_out, kc, vc, ws, stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        reset()
        g.replay()
        torch.cuda.synchronize()
        assert lb.get_device_error()[0] == lb.LLAMA_OK
        for a, b, what in zip((hidden, res_out, kc, vc), eager, ("hidden", "residual", "k cache", "v cache")):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what} differs after graph replay"


def test_stack_graph_replay_matches_eager():
    # a 2-layer stack with embedding, final norm, lm_head and argmax over a
    # mixed batch, captured as one call
    spec = dataclasses.replace(I.SPECS["tiny"], num_layers=2, vocab=1024, residual_none=True,
                               groups=(("decode", 3, 1, 10, 1800), ("prefill", 2, 20, 0, 0)))
    bl = I.make_batch(spec, 11, DEV)
    layers = [I.make_layer_weights(spec, 11, l, DEV) for l in range(spec.num_layers)]
    caches0 = [I.make_kv_cache(spec, bl.num_blocks, 11, l, DEV) for l in range(spec.num_layers)]
    emb, ids, lm, fn = I.make_stack_extras(spec, bl.num_tokens, 11, DEV)
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
    eager = (tokens.clone(), logits.clone(), [c[0].clone() for c in caches])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    torch.cuda.synchronize()
    reset()
    g.replay()
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    assert torch.equal(tokens, eager[0])
    assert torch.equal(logits, eager[1])
    for k, k_eager in zip([c[0] for c in caches], eager[2]):
        assert torch.equal(k.view(torch.int16), k_eager.view(torch.int16))
