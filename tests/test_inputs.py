"""The synthetic input recipe on the CPU: every workload's batch has the
structure its parity tests and the benchmark assume (block tables that are a
permutation of the used blocks plus unowned spares, decode tokens at position
= context, fresh prefill chunks at positions 0..n-1, seq_lens = context + new
tokens), and the generators are reproducible from their seeds."""

import pytest
import torch

from llama_decoder_layer_gb300 import inputs as I


@pytest.mark.parametrize("name", ["tiny", "decode_8b", "decode_70b", "stack_70b", "decode_70b_80l", "qwen3_moe",
                                  "qwen3_moe_decode"])
def test_batch_structure(name):
    spec = I.SPECS[name]
    bl = I.make_batch(spec, 3, "cpu")
    qsl = bl.query_start_loc.tolist()
    pos = bl.positions.tolist()
    sl = bl.seq_lens.tolist()
    bt = bl.block_table
    assert qsl[0] == 0 and qsl[-1] == bl.num_tokens == len(pos)
    owned = []
    for b in range(bl.num_seqs):
        q, c = bl.q_lens[b], bl.ctx_lens[b]
        assert qsl[b + 1] - qsl[b] == q and sl[b] == c + q
        assert pos[qsl[b]:qsl[b + 1]] == list(range(c, c + q))  # decode: position = context
        n = (sl[b] + spec.block_size - 1) // spec.block_size
        row = bt[b].tolist()
        assert all(x >= 0 for x in row[:n]) and all(x == -1 for x in row[n:])
        owned += row[:n]
    # a permutation of the used blocks, with the spare blocks owned by no sequence
    assert len(owned) == len(set(owned)) == bl.num_blocks - spec.spare_blocks
    assert set(owned) <= set(range(bl.num_blocks))
    # contexts within the ranges of the workload's groups
    i = 0
    for kind, count, new, lo, hi in spec.groups:
        for _ in range(count):
            assert lo <= bl.ctx_lens[i] <= hi and bl.q_lens[i] == new
            if kind == "prefill":
                assert bl.ctx_lens[i] == 0 == pos[qsl[i]]  # fresh chunks start at position 0
            i += 1


def test_generators_are_reproducible_and_seeded():
    spec = I.SPECS["tiny"]
    a, b, c = (I.make_batch(spec, s, "cpu") for s in (5, 5, 6))
    assert torch.equal(a.block_table, b.block_table) and torch.equal(a.positions, b.positions)
    w1, w2 = I.make_layer_weights(spec, 1, 0, "cpu"), I.make_layer_weights(spec, 1, 0, "cpu")
    w3 = I.make_layer_weights(spec, 1, 1, "cpu")  # another layer
    for k in w1:
        assert torch.equal(w1[k], w2[k])
        assert not torch.equal(w1[k], w3[k])
    x = I.normal_bf16((64, 256), 0.02, 1.0, 9, "cpu").float()
    assert abs(float(x.mean()) - 1.0) < 0.01 and abs(float(x.std()) - 0.02) < 0.005
    assert x.dtype == torch.float32 and I.normal_bf16((4,), 1.0, 0.0, 9, "cpu").dtype == torch.bfloat16


def test_moe_weights_shapes():
    spec = I.SPECS["qwen3_moe"]
    w = I.make_moe_layer_weights(spec, 0, 0, "cpu")
    E, H, Im = spec.extra["num_experts"], spec.hidden, spec.extra["moe_intermediate"]
    assert w["w_router"].shape == (E, H) and w["w13"].shape == (E, 2 * Im, H) and w["w2"].shape == (E, H, Im)
    assert w["w_qkv"].shape == ((spec.n_heads + 2 * spec.n_kv_heads) * spec.head_dim, H)
