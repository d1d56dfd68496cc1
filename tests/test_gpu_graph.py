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
