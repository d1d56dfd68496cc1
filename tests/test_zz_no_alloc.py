"""llama_paged_attention_noalloc: the paged attention call for callers that
cannot allocate device memory where they run attention.  Examples are a plugin
that gets only input and output buffers, and a process whose memory pool
another runtime owns.  Its split-KV scratch is a fixed array inside the
library.

Checked through the C ABI on two calls in a row with different batches: the
second call meets the array as the first one left it, laid out for another
batch (other contexts, chunk counts and work-list offset).  Each call must
equal llama_paged_attention (which takes a caller workspace) bit for bit, as
both run the same deterministic kernels, and the second also matches the
oracle's attention within the tolerance.  The oversized-batch rejection and
the order of the argument checks are checked too.  This file is collected
last; it also passes when run alone in a fresh process.
"""

import dataclasses

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O
from tests.helpers import assert_close, bits, f32, oracle_batch

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


def _both_entry_points(case):
    cfg, batch, q, kc, vc, bl = case
    ref = torch.empty((bl.num_tokens, cfg.n_heads * cfg.head_dim), dtype=torch.bfloat16, device=DEV)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), DEV)
    lb.paged_attention(cfg, batch, q, kc, vc, ref, ws)
    out = torch.full_like(ref, float("nan"))
    lb.paged_attention_noalloc(cfg, batch, q, kc, vc, out)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    return out, ref


def test_noalloc_matches_workspace_entry_point_twice():
    # first call: long decode contexts (up to 9000 keys, six 1536-key chunks)
    # and a long prefill, so the array is left full of another batch's
    # partials and work list
    first = _case(64, 8, 128, (("decode", 9, 1, 3000, 9000), ("prefill", 1, 300, 100, 100)), 41)
    # second call: decode contexts up to 5000 keys (up to four chunks) plus
    # prefill sequences with and without a cached prefix
    second = _case(64, 8, 128, (("decode", 6, 1, 20, 5000), ("prefill", 2, 40, 0, 0), ("decode", 2, 1, 0, 30),
                                ("prefill", 1, 17, 30, 30)), 51)
    for call, case in enumerate((first, second), start=1):
        out, ref = _both_entry_points(case)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"no-alloc call {call} differs from llama_paged_attention"
    cfg, batch, q, kc, vc, bl = second
    ob = oracle_batch(bl)
    want = O.paged_attention(f32(q), bits(kc), bits(vc), ob.block_table, ob.seq_lens, ob.query_start_loc,
                             ob.positions, cfg.n_kv_heads, 16)
    assert_close(f32(out).reshape(want.shape), want, "no-alloc call 2 against the oracle")


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    limit = int(lb.lib().llama_paged_attention_noalloc_limit())
    assert limit == 32 << 20
    # 128 decode sequences, one token each at position 16384 (16385-token
    # contexts, 11 split-KV chunks each) x 64 heads need 47 MB of partials,
    # more than the 32 MiB array
    spec = I.SPECS["decode_70b"]
    cfg = lb.LayerConfig.from_spec(spec)
    z = torch.zeros(1, dtype=torch.int32, device=DEV)
    nblk = 16385 // 16 + 1
    batch = lb.Batch(torch.full((128,), 16384, dtype=torch.int32, device=DEV),
                     torch.arange(129, dtype=torch.int32, device=DEV),
                     torch.full((128,), 16385, dtype=torch.int32, device=DEV),
                     torch.arange(128 * nblk, dtype=torch.int32, device=DEV).view(128, nblk), 128 * nblk, 1, 16385)
    with pytest.raises(lb.LlamaError) as e:
        lb.paged_attention_noalloc(cfg, batch, z, z, z, z)
    assert e.value.status == lb.LLAMA_ERR_SCRATCH_LIMIT
    # an invalid batch (more sequences than tokens) is an argument error
    # first, whatever its scratch would be
    bad = dataclasses.replace(batch, positions=batch.positions[:1])
    with pytest.raises(lb.LlamaError) as e:
        lb.paged_attention_noalloc(cfg, bad, z, z, z, z)
    assert e.value.status == lb.LLAMA_ERR_ARG
    assert lb.get_device_error()[0] == lb.LLAMA_OK
