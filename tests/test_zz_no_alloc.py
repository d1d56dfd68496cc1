"""llama_paged_attention_noalloc: the paged attention call for callers that
cannot allocate device memory where they run attention.  Examples are a plugin
that gets only input and output buffers, and a process whose memory pool
another runtime owns.  Its split-KV scratch is a fixed array inside the
library.

Checked through the C ABI against llama_paged_attention (which takes a caller
workspace), on two calls in a row so the second one meets the array as the
first one left it.  The oversized-batch rejection is checked too.  This file
is collected last; it also passes when run alone in a fresh process.
"""

import dataclasses

import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from tests.helpers import assert_close, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


def _case(nq, nkv, d, groups, seed):
    spec = dataclasses.replace(I.SPECS["tiny"], n_heads=nq, n_kv_heads=nkv, head_dim=d, hidden=nq * d,
                               groups=groups)
    bl = I.make_batch(spec, seed, DEV)
    q = I.normal_bf16((bl.num_tokens, nq, d), 1.0, 0.0, seed + 1, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, DEV)
    return lb.LayerConfig.from_spec(spec), lb.Batch.from_layout(bl), q, kc, vc, bl


def test_noalloc_matches_workspace_entry_point_twice():
    # decode contexts up to 5000 keys (four 1536-key chunks: the scratch is
    # used) plus prefill sequences with and without a cached prefix
    groups = (("decode", 6, 1, 20, 5000), ("prefill", 2, 40, 0, 0), ("decode", 2, 1, 0, 30),
              ("prefill", 1, 17, 30, 30))
    cfg, batch, q, kc, vc, bl = _case(64, 8, 128, groups, 51)
    ref = torch.empty((bl.num_tokens, 64 * 128), dtype=torch.bfloat16, device=DEV)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), DEV)
    lb.paged_attention(cfg, batch, q, kc, vc, ref, ws)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lb.paged_attention_noalloc(cfg, batch, q, kc, vc, out)
        torch.cuda.synchronize()
        assert lb.get_device_error()[0] == lb.LLAMA_OK
        assert_close(f32(out), f32(ref), f"no-alloc call {call + 1}")


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    limit = int(lb.lib().llama_paged_attention_noalloc_limit())
    assert limit == 32 << 20
    # 128 sequences x 16385-token contexts (11 split-KV chunks each) x 64 heads
    # need 47 MB of partials, more than the 32 MiB array
    spec = I.SPECS["decode_70b"]
    cfg = lb.LayerConfig.from_spec(spec)
    z = torch.zeros(1, dtype=torch.int32, device=DEV)
    batch = lb.Batch(torch.zeros(128, dtype=torch.int32, device=DEV), torch.arange(129, dtype=torch.int32, device=DEV),
                     torch.full((128,), 16385, dtype=torch.int32, device=DEV),
                     torch.zeros((128, 1025), dtype=torch.int32, device=DEV), 1, 1, 16385)
    with pytest.raises(lb.LlamaError) as e:
        lb.paged_attention_noalloc(cfg, batch, z, z, z, z)
    assert e.value.status == lb.LLAMA_ERR_SCRATCH_LIMIT
