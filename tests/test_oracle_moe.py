"""Pins of the oracle's MoE block against what the pages and the mathematics
fix: the page's worked combine example (tests/golden/moe_combine_example.json),
a single expert with k = 1 reducing to the dense MLP (already pinned), the
routing weights summing to one and equal to the softmax of the selected
logits, brute-force top-k with index-order ties, and invariance under a
relabelling of the experts."""

import json
import os

import numpy as np
from scipy.special import softmax

from oracle import llama_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "moe_combine_example.json")


def _experts(rng, E, H, I):
    w13 = rng.normal(size=(E, 2 * I, H)) * 0.1
    w2 = rng.normal(size=(E, H, I)) * 0.1
    return w13, w2


def test_page_worked_combine_example():
    ex = json.load(open(GOLDEN))
    ids, w = ex["expert_ids"], np.array(ex["weights"])
    rng = np.random.default_rng(0)
    H, I, E = 16, 12, 128
    w13, w2 = _experts(rng, E, H, I)
    x = rng.normal(size=(1, H))
    ys = [O.moe_expert(x, w13[e], w2[e], bf16_tensors=False)[0] for e in ids]
    got = O.moe_combine(ys, w)
    # written out term by term: 0.1*y0 + 0.2*y7 + 0.2*y9 + 0.1*y34 + 0.05*y77 + 0.05*y89 + 0.1*y110 + 0.1*y127
    by_id = dict(zip(ids, ys))
    ref = (0.1 * by_id[0] + 0.2 * by_id[7] + 0.2 * by_id[9] + 0.1 * by_id[34] + 0.05 * by_id[77]
           + 0.05 * by_id[89] + 0.1 * by_id[110] + 0.1 * by_id[127])
    assert np.max(np.abs(got - ref)) < 1e-12


def test_single_expert_is_the_dense_mlp():
    rng = np.random.default_rng(1)
    T, H, I = 5, 32, 24
    w13, w2 = _experts(rng, 1, H, I)
    wr = rng.normal(size=(1, H))
    h = rng.normal(size=(T, H))
    out, ids, w, _ = O.moe_block(h, wr, w13, w2, top_k=1, bf16_tensors=False)
    assert np.all(ids == 0) and np.allclose(w, 1.0)
    dense = O.linear(O.silu_and_mul(O.linear(h, w13[0])), w2[0])
    assert np.max(np.abs(out - dense)) < 1e-12


def test_routing_weights_are_the_softmax_of_the_selected_logits():
    rng = np.random.default_rng(2)
    logits = rng.normal(size=(40, 128)) * 3
    ids, w, gap = O.moe_route(logits, 8)
    assert np.allclose(w.sum(axis=1), 1.0)
    for t in range(40):
        brute = sorted(range(128), key=lambda e: (-logits[t, e], e))[:8]  # value, then index
        assert list(ids[t]) == brute
        assert np.allclose(w[t], softmax(logits[t, brute]))
        # renormalised full softmax: the same weights
        p = softmax(logits[t])
        assert np.allclose(w[t], p[brute] / p[brute].sum())
        assert gap[t] == logits[t, brute[7]] - logits[t, sorted(range(128), key=lambda e: (-logits[t, e], e))[8]]


def test_ties_go_to_the_lower_expert_index():
    logits = np.zeros((1, 16))
    logits[0, [3, 9, 12]] = 2.0
    ids, _, gap = O.moe_route(logits, 4)
    assert list(ids[0]) == [3, 9, 12, 0] and gap[0] == 0.0


def test_relabelling_the_experts_changes_nothing():
    rng = np.random.default_rng(3)
    T, H, I, E = 6, 16, 8, 10
    w13, w2 = _experts(rng, E, H, I)
    wr = rng.normal(size=(E, H))
    h = rng.normal(size=(T, H))
    perm = rng.permutation(E)
    a, _, _, _ = O.moe_block(h, wr, w13, w2, 3, bf16_tensors=False)
    b, _, _, _ = O.moe_block(h, wr[perm], w13[perm], w2[perm], 3, bf16_tensors=False)
    assert np.max(np.abs(a - b)) < 1e-12


def test_block_equals_the_per_token_sum_over_its_experts():
    rng = np.random.default_rng(4)
    T, H, I, E, k = 7, 16, 12, 20, 4
    w13, w2 = _experts(rng, E, H, I)
    wr = rng.normal(size=(E, H))
    h = rng.normal(size=(T, H))
    out, ids, w, _ = O.moe_block(h, wr, w13, w2, k, bf16_tensors=False)
    for t in range(T):
        acc = np.zeros(H)
        for j in range(k):
            e = ids[t, j]
            g = h[t] @ w13[e, :I].T
            u = h[t] @ w13[e, I:].T
            acc += w[t, j] * ((g / (1 + np.exp(-g)) * u) @ w2[e].T)
        assert np.max(np.abs(out[t] - acc)) < 1e-10


def _moe_layer_case(seed=51, residual=True):
    from tests.test_oracle_pins import _paged_setup, tiny_shape, tiny_weights
    sh = tiny_shape()
    rng = np.random.default_rng(seed)
    w = tiny_weights(sh, rng)
    s = _paged_setup([6, 0, 3], [1, 7, 4], sh.n_kv_heads, sh.head_dim, bs=sh.block_size, seed=13)
    batch = O.Batch(s["positions"], s["qsl"], s["seq_lens"], s["block_table"])
    T = int(s["qsl"][-1])
    x = O.round_to_bf16(rng.standard_normal((T, sh.hidden)))
    res = O.round_to_bf16(rng.standard_normal((T, sh.hidden))) if residual else None
    return sh, w, s, batch, x, res


def test_moe_layer_with_one_expert_is_the_dense_layer():
    """The Qwen3-MoE layer with a single expert, k = 1 and the dense MLP's
    weights as that expert is the Llama layer, bit for bit (the routing weight
    is exactly 1), with the module outputs stored in bf16."""
    for residual in (True, False):
        sh, w, s, batch, x, res = _moe_layer_case(residual=residual)
        kc1, vc1 = s["k"].copy(), s["v"].copy()
        want, want_r = O.decoder_layer(sh, w, batch, x, res, kc1, vc1)
        kc2, vc2 = s["k"].copy(), s["v"].copy()
        wr = np.ones((1, sh.hidden))
        got, got_r, ids, _ = O.moe_decoder_layer(sh, w, wr, w.w_gate_up[None], w.w_down[None], 1, batch, x, res,
                                                 kc2, vc2)
        assert np.all(ids == 0)
        assert np.array_equal(got, want) and np.array_equal(got_r, want_r)
        assert np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2)


def test_moe_layer_rows_subset_matches_the_full_layer():
    sh, w, s, batch, x, res = _moe_layer_case(seed=52)
    rng = np.random.default_rng(5)
    E, I = 6, 20
    w13, w2 = _experts(rng, E, sh.hidden, I)
    wr = rng.normal(size=(E, sh.hidden))
    full = O.moe_decoder_layer(sh, w, wr, w13, w2, 2, batch, x, res, s["k"].copy(), s["v"].copy())
    rows = [0, 5, 11]
    part = O.moe_decoder_layer(sh, w, wr, w13, w2, 2, batch, x, res, s["k"].copy(), s["v"].copy(), rows=rows)
    assert np.array_equal(part[0][rows], full[0][rows]) and np.array_equal(part[1][rows], full[1][rows])
    assert np.array_equal(part[2][rows], full[2][rows])


# ----------------------------------------------------------- planted mistakes

def _route_not_renormalised(router_logits, top_k):
    x = np.asarray(router_logits, dtype=np.float64)
    ids = np.argsort(-x, axis=1, kind="stable")[:, :top_k]
    w = np.take_along_axis(softmax(x, axis=1), ids, axis=1)  # top-k of the full softmax, not renormalised
    return ids, w, np.zeros(x.shape[0])


def _route_ties_high(router_logits, top_k):
    x = np.asarray(router_logits, dtype=np.float64)
    order = np.argsort(-x[:, ::-1], axis=1, kind="stable")
    ids = (x.shape[1] - 1 - order)[:, :top_k]
    sel = np.take_along_axis(x, ids, axis=1)
    w = softmax(sel, axis=1)
    return ids, w, np.zeros(x.shape[0])


def _combine_unweighted(expert_outputs, weights, dtype=np.float64):
    return np.sum(np.asarray(expert_outputs, dtype=dtype), axis=0)


def _expert_gate_up_swapped(x, w13_e, w2_e, dtype=np.float64, bf16_tensors=True):
    I = w13_e.shape[0] // 2
    sw = np.concatenate([w13_e[I:], w13_e[:I]])
    return O.store(O.linear(O.silu_and_mul(O.linear(x, sw, dtype), dtype), w2_e, dtype), bf16_tensors, dtype)


PINS = [test_page_worked_combine_example, test_single_expert_is_the_dense_mlp,
        test_routing_weights_are_the_softmax_of_the_selected_logits, test_ties_go_to_the_lower_expert_index,
        test_relabelling_the_experts_changes_nothing, test_block_equals_the_per_token_sum_over_its_experts,
        test_moe_layer_with_one_expert_is_the_dense_layer]


import pytest  # noqa: E402


def _layer_moe_on_first_norm(shape, w, w_router, w13, w2, top_k, batch, hidden, residual, k_cache_bits,
                             v_cache_bits, rows=None, dtype=np.float64, bf16_tensors=True):
    # the MoE block fed from the input norm instead of the post-attention norm
    h, r = O.fused_add_rms_norm(hidden, residual, w.ln1, shape.rms_eps, dtype, bf16_tensors)
    y = O.attention_block(shape, w, batch, h, k_cache_bits, v_cache_bits, dtype=dtype, bf16_tensors=bf16_tensors)
    _, r2 = O.fused_add_rms_norm(y, r, w.ln2, shape.rms_eps, dtype, bf16_tensors)
    out, ids, _, gap = O.moe_block(h, w_router, w13, w2, top_k, dtype, bf16_tensors)
    return out, r2, ids, gap


@pytest.mark.parametrize("name,mutant", [("moe_route", _route_not_renormalised), ("moe_route", _route_ties_high),
                                         ("moe_combine", _combine_unweighted),
                                         ("moe_expert", _expert_gate_up_swapped),
                                         ("moe_decoder_layer", _layer_moe_on_first_norm)],
                         ids=["not_renormalised", "ties_high", "combine_unweighted", "gate_up_swapped",
                              "layer_moe_on_first_norm"])
def test_planted_moe_mistake_is_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(O, name, mutant)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0
