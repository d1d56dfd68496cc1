"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each check ties one oracle function to what the pages and mathematics fix:
library routines on special cases, closed forms, invariants the pages state,
and brute force on tiny inputs.  ``tests/test_oracle_mutations.py`` plants
mistakes in the oracle and shows that these checks catch them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import llama_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def bf16_vals(shape, std=1.0, rng=RNG):
    return O.round_to_bf16(rng.standard_normal(shape).astype(np.float32) * std).astype(np.float64)


# --------------------------------------------------------------------------- bf16 storage

def check_bf16_rounding():
    x = np.concatenate([RNG.standard_normal(5000).astype(np.float32) * 10.0 ** RNG.integers(-6, 6, 5000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0, -0.0,
                                  65504.0, 3.0e38], np.float32)])
    ours = O.float_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = O.bf16_bits_to_float(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_bf16_rounding_matches_torch():
    check_bf16_rounding()


# --------------------------------------------------------------------------- RMSNorm

def check_rms_norm():
    x = RNG.standard_normal((7, 96)) * 3.0
    g = 1.0 + 0.02 * RNG.standard_normal(96)
    ours = O.rms_norm(x, g, 1e-5)
    ref = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.max(np.abs(ours - ref)) < 1e-12
    # closed form with gamma = 1: mean(h^2) = m / (m + eps), m = mean(x^2)
    eps = 0.3
    h = O.rms_norm(x, np.ones(96), eps)
    m = np.mean(x * x, axis=-1)
    assert np.allclose(np.mean(h * h, axis=-1), m / (m + eps), rtol=1e-13, atol=0)


def test_rms_norm_library_and_closed_form():
    check_rms_norm()


def check_fused_add_norm():
    x = RNG.standard_normal((5, 64))
    res = RNG.standard_normal((5, 64))
    g = 1.0 + 0.02 * RNG.standard_normal(64)
    # residual None: residual becomes the un-normed input, hidden = norm(input)
    h, r = O.fused_add_rms_norm(x, None, g, 1e-5)
    assert np.array_equal(r, x)
    assert np.array_equal(h, O.rms_norm(x, g, 1e-5))
    # with residual: add then norm
    h, r = O.fused_add_rms_norm(x, res, g, 1e-5)
    assert np.array_equal(r, x + res)
    ref = F.rms_norm(torch.from_numpy(x + res), (64,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.max(np.abs(h - ref)) < 1e-12


def test_fused_add_rms_norm_equals_add_then_norm():
    check_fused_add_norm()


# --------------------------------------------------------------------------- linear / SiluAndMul

def check_linear():
    x = RNG.standard_normal((6, 40))
    w = RNG.standard_normal((24, 40))
    assert np.max(np.abs(O.linear(x, w) - F.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy())) < 1e-12


def test_linear_is_f_linear():
    check_linear()


def check_silu_and_mul():
    x = RNG.standard_normal((9, 2 * 33)) * 4
    ours = O.silu_and_mul(x)
    t = torch.from_numpy(x)
    ref = (F.silu(t[:, :33]) * t[:, 33:]).numpy()
    assert np.max(np.abs(ours - ref)) < 1e-12
    # special values of SiLU: silu(0) = 0, silu(z) -> z for large z, -> 0 for very negative z
    z = np.array([0.0, 40.0, -40.0])
    s = O.silu(z)
    assert s[0] == 0.0 and abs(s[1] - 40.0) < 1e-12 and abs(s[2]) < 1e-15
    # gate is the FIRST half: gate = 0 gives zero output whatever up is
    x2 = np.concatenate([np.zeros((3, 8)), RNG.standard_normal((3, 8))], axis=1)
    assert np.all(O.silu_and_mul(x2) == 0.0)


def test_silu_and_mul_definition():
    check_silu_and_mul()


# --------------------------------------------------------------------------- RoPE

def check_rope_invariants(theta=500000.0, scaling=None, d=128):
    inv = O.rope_inv_freq(d, theta, scaling)
    x = RNG.standard_normal((1, 3, d))
    # position 0 is the identity
    assert np.max(np.abs(O.apply_rope(x, [0], inv) - x)) == 0.0
    # norm of every (i, i + d/2) pair is preserved
    pos = [1234]
    y = O.apply_rope(x, pos, inv)
    h = d // 2
    assert np.allclose(x[..., :h] ** 2 + x[..., h:] ** 2, y[..., :h] ** 2 + y[..., h:] ** 2, rtol=1e-12, atol=1e-12)
    # q(m) . k(n) depends on m - n only
    q = RNG.standard_normal((1, 1, d))
    k = RNG.standard_normal((1, 1, d))
    for m, n, c in [(10, 3, 500), (7000, 6999, 12345), (0, 100, 1)]:
        a = np.sum(O.apply_rope(q, [m], inv) * O.apply_rope(k, [n], inv))
        b = np.sum(O.apply_rope(q, [m + c], inv) * O.apply_rope(k, [n + c], inv))
        assert abs(a - b) < 1e-9 * max(1.0, abs(a))
    # rotating by p then by -p is the identity
    z = O.apply_rope(O.apply_rope(x, [777], inv), [-777], inv)
    assert np.max(np.abs(z - x)) < 1e-12


def test_rope_invariants_plain():
    check_rope_invariants(10000.0, None, 64)
    check_rope_invariants(500000.0, None, 128)


def test_rope_invariants_llama3():
    check_rope_invariants(500000.0, O_LLAMA3, 128)


O_LLAMA3 = {"rope_type": "llama3", "factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
            "original_max_position_embeddings": 8192}


def check_rope_rotation_closed_form():
    # reading R4: element i pairs with i + d/2; unit vector e_i at position p
    d, theta = 16, 10000.0
    inv = O.rope_inv_freq(d, theta)
    assert inv[0] == 1.0 and abs(inv[1] - theta ** (-2.0 / d)) < 1e-15
    assert np.allclose(inv[1:] / inv[:-1], theta ** (-2.0 / d), rtol=1e-13)
    p = 37
    for i in range(d // 2):
        e = np.zeros((1, 1, d))
        e[0, 0, i] = 1.0
        y = O.apply_rope(e, [p], inv)[0, 0]
        want = np.zeros(d)
        want[i] = math.cos(p * inv[i])
        want[i + d // 2] = math.sin(p * inv[i])
        assert np.max(np.abs(y - want)) < 1e-14


def test_rope_rotation_closed_form():
    check_rope_rotation_closed_form()


def check_llama3_bands():
    d, theta = 128, 500000.0
    plain = O.rope_inv_freq(d, theta)
    sc = O.rope_inv_freq(d, theta, O_LLAMA3)
    lam = 2 * math.pi / plain
    hi_band = lam < 8192 / 4.0
    lo_band = lam > 8192 / 1.0
    assert hi_band.any() and lo_band.any() and (~hi_band & ~lo_band).any()
    assert np.array_equal(sc[hi_band], plain[hi_band])
    assert np.array_equal(sc[lo_band], plain[lo_band] / 8.0)
    mid = ~hi_band & ~lo_band
    # the blend lies between inv/8 and inv
    assert np.all(sc[mid] <= plain[mid]) and np.all(sc[mid] >= plain[mid] / 8.0)
    # continuity of the smooth band at both edges: evaluate the rule as a
    # function of wavelength right at the band edges
    cfg1 = dict(O_LLAMA3)
    for edge, want_ratio in [(8192.0, 1 / 8.0), (2048.0, 1.0)]:
        f = 2 * math.pi / edge
        # theta chosen so that inv_freq[1] == f exactly: theta^(-2/d) = f
        th = f ** (-d / 2.0)
        got = O.rope_inv_freq(d, th, cfg1)[1]
        assert abs(got / f - want_ratio) < 1e-12
    # factor 1 and equal band edges reduce to plain RoPE frequencies
    ident = {"rope_type": "llama3", "factor": 1.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
             "original_max_position_embeddings": 8192}
    assert np.allclose(O.rope_inv_freq(d, theta, ident), plain, rtol=1e-15, atol=0)
    # monotone decreasing in i
    assert np.all(np.diff(sc) < 0)


def test_llama3_band_edges():
    check_llama3_bands()


# --------------------------------------------------------------------------- paged attention

def _paged_setup(seq_ctx, seq_new, nkv, d, bs=4, seed=0, spare=3):
    rng = np.random.default_rng(seed)
    B = len(seq_ctx)
    seq_lens = [c + n for c, n in zip(seq_ctx, seq_new)]
    nblk = [(s + bs - 1) // bs for s in seq_lens]
    nb = sum(nblk) + spare
    perm = rng.permutation(nb)
    bt = -np.ones((B, max(nblk)), np.int64)
    cur = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[cur:cur + nblk[b]]
        cur += nblk[b]
    kc = O.float_to_bf16_bits(rng.standard_normal((nb, nkv, bs, d)).astype(np.float32))
    vc = O.float_to_bf16_bits(rng.standard_normal((nb, nkv, bs, d)).astype(np.float32))
    pos, qsl = [], [0]
    for c, n in zip(seq_ctx, seq_new):
        pos += list(range(c, c + n))
        qsl.append(qsl[-1] + n)
    return dict(seq_lens=np.array(seq_lens), block_table=bt, k=kc, v=vc, positions=np.array(pos),
                qsl=np.array(qsl), bs=bs)


def contiguous_kv(setup, b, n):
    return (O.gather_kv(setup["k"], setup["block_table"][b], n, setup["bs"]).astype(np.float64),
            O.gather_kv(setup["v"], setup["block_table"][b], n, setup["bs"]).astype(np.float64))


def check_attention_vs_sdpa():
    nq, nkv, d = 8, 2, 16
    s = _paged_setup([5, 0, 13], [1, 9, 4], nkv, d, seed=3)
    T = int(s["qsl"][-1])
    q = RNG.standard_normal((T, nq, d))
    out = O.paged_attention(q, s["k"], s["v"], s["block_table"], s["seq_lens"], s["qsl"], s["positions"],
                            nkv, s["bs"])
    for b in range(3):
        lo, hi = s["qsl"][b], s["qsl"][b + 1]
        n = int(s["seq_lens"][b])
        K, V = contiguous_kv(s, b, n)
        qb = torch.from_numpy(q[lo:hi]).permute(1, 0, 2)[None]      # [1, nq, L, d]
        kb = torch.from_numpy(K).permute(1, 0, 2)[None]             # [1, nkv, n, d]
        vb = torch.from_numpy(V).permute(1, 0, 2)[None]
        mask = torch.from_numpy(np.arange(n)[None, :] <= s["positions"][lo:hi][:, None])
        ref = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, enable_gqa=True)[0].permute(1, 0, 2)
        assert np.max(np.abs(out[lo:hi] - ref.numpy())) < 1e-12
    # fresh prefill (no prior context) is exactly is_causal=True
    b = 1
    lo, hi = s["qsl"][b], s["qsl"][b + 1]
    K, V = contiguous_kv(s, b, int(s["seq_lens"][b]))
    ref = F.scaled_dot_product_attention(torch.from_numpy(q[lo:hi]).permute(1, 0, 2)[None],
                                         torch.from_numpy(K).permute(1, 0, 2)[None],
                                         torch.from_numpy(V).permute(1, 0, 2)[None],
                                         is_causal=True, enable_gqa=True)[0].permute(1, 0, 2)
    assert np.max(np.abs(out[lo:hi] - ref.numpy())) < 1e-12


def test_attention_matches_sdpa():
    check_attention_vs_sdpa()


def check_gqa_equals_mha():
    nq, nkv, d = 8, 2, 8
    s = _paged_setup([6, 2], [3, 1], nkv, d, seed=5)
    T = int(s["qsl"][-1])
    q = RNG.standard_normal((T, nq, d))
    gqa = O.paged_attention(q, s["k"], s["v"], s["block_table"], s["seq_lens"], s["qsl"], s["positions"], nkv, s["bs"])
    # replicate every kv head nq/nkv times (consecutive groups) -> MHA
    g = nq // nkv
    k_rep = np.repeat(s["k"], g, axis=1)
    v_rep = np.repeat(s["v"], g, axis=1)
    mha = O.paged_attention(q, k_rep, v_rep, s["block_table"], s["seq_lens"], s["qsl"], s["positions"], nq, s["bs"])
    assert np.max(np.abs(gqa - mha)) == 0.0


def test_gqa_equals_mha_with_replicated_kv():
    check_gqa_equals_mha()


def check_paged_equals_contiguous():
    nq, nkv, d, bs = 4, 2, 8, 4
    s = _paged_setup([9, 3], [2, 5], nkv, d, bs=bs, seed=11)
    T = int(s["qsl"][-1])
    q = RNG.standard_normal((T, nq, d))
    base = O.paged_attention(q, s["k"], s["v"], s["block_table"], s["seq_lens"], s["qsl"], s["positions"], nkv, bs)
    # relocate every block to a new random physical index: same result
    for seed in range(3):
        rng = np.random.default_rng(100 + seed)
        nb = s["k"].shape[0]
        new_of_old = rng.permutation(nb)
        k2 = np.empty_like(s["k"])
        v2 = np.empty_like(s["v"])
        k2[new_of_old] = s["k"]
        v2[new_of_old] = s["v"]
        bt2 = np.where(s["block_table"] >= 0, new_of_old[np.maximum(s["block_table"], 0)], -1)
        got = O.paged_attention(q, k2, v2, bt2, s["seq_lens"], s["qsl"], s["positions"], nkv, bs)
        assert np.array_equal(got, base)
    # a contiguous cache (identity block table over an unshuffled copy) gives the same result
    B = 2
    kc, vc, rows = [], [], []
    for b in range(B):
        n = int(s["seq_lens"][b])
        nblk = (n + bs - 1) // bs
        rows.append(list(range(len(kc), len(kc) + nblk)))
        for j in range(nblk):
            kc.append(s["k"][s["block_table"][b, j]])
            vc.append(s["v"][s["block_table"][b, j]])
    bt3 = -np.ones_like(s["block_table"])
    for b in range(B):
        bt3[b, :len(rows[b])] = rows[b]
    got = O.paged_attention(q, np.stack(kc), np.stack(vc), bt3, s["seq_lens"], s["qsl"], s["positions"], nkv, bs)
    assert np.array_equal(got, base)


def test_paged_equals_contiguous():
    check_paged_equals_contiguous()


def check_attention_closed_forms():
    nq, nkv, d = 4, 1, 8
    # context 1: the single visible value is the output
    s = _paged_setup([0], [1], nkv, d, seed=7)
    q = RNG.standard_normal((1, nq, d)) * 5
    out = O.paged_attention(q, s["k"], s["v"], s["block_table"], s["seq_lens"], s["qsl"], s["positions"], nkv, s["bs"])
    _, V = contiguous_kv(s, 0, 1)
    for h in range(nq):
        assert np.max(np.abs(out[0, h] - V[0, 0])) < 1e-15
    # identical keys: uniform weights, output = mean of the visible values
    s = _paged_setup([10], [1], nkv, d, seed=8)
    kc = s["k"].copy()
    kc[...] = kc[s["block_table"][0, 0], 0, 0]
    out = O.paged_attention(q, kc, s["v"], s["block_table"], s["seq_lens"], s["qsl"], s["positions"], nkv, s["bs"])
    _, V = contiguous_kv(s, 0, 11)
    assert np.max(np.abs(out[0, 0] - V[:, 0].mean(axis=0))) < 1e-13


def test_attention_closed_forms():
    check_attention_closed_forms()


def brute_attention(q, K, V, p, scale):
    """Scalar loops: one query vector against keys 0..p."""
    s = []
    for j in range(p + 1):
        acc = 0.0
        for i in range(len(q)):
            acc += q[i] * K[j][i]
        s.append(acc * scale)
    mx = max(s)
    e = [math.exp(x - mx) for x in s]
    z = sum(e)
    return [sum(e[j] / z * V[j][i] for j in range(p + 1)) for i in range(len(q))]


def check_attention_brute_force():
    nq, nkv, d = 4, 2, 4
    s = _paged_setup([3, 0], [2, 3], nkv, d, bs=2, seed=9)
    T = int(s["qsl"][-1])
    q = RNG.standard_normal((T, nq, d))
    out = O.paged_attention(q, s["k"], s["v"], s["block_table"], s["seq_lens"], s["qsl"], s["positions"], nkv, s["bs"])
    seq = [0, 0, 1, 1, 1]
    for t in range(T):
        b = seq[t]
        K, V = contiguous_kv(s, b, int(s["seq_lens"][b]))
        for h in range(nq):
            kh = h // (nq // nkv)
            want = brute_attention(q[t, h].tolist(), K[:, kh].tolist(), V[:, kh].tolist(), int(s["positions"][t]),
                                   1 / math.sqrt(d))
            assert np.max(np.abs(out[t, h] - np.array(want))) < 1e-12


def test_attention_brute_force():
    check_attention_brute_force()


# --------------------------------------------------------------------------- cache indexing

def test_slot_mapping_and_cache_write_roundtrip():
    nkv, d, bs = 2, 4, 4
    s = _paged_setup([5, 0], [3, 6], nkv, d, bs=bs, seed=21)
    slots = O.slot_mapping(s["positions"], s["qsl"], s["block_table"], bs)
    assert len(set(slots.tolist())) == len(slots)
    T = len(slots)
    k = RNG.standard_normal((T, nkv, d)).astype(np.float32)
    v = RNG.standard_normal((T, nkv, d)).astype(np.float32)
    kc, vc = s["k"].copy(), s["v"].copy()
    O.kv_cache_write(k, v, slots, kc, vc, bs)
    # reading each sequence back through its block table returns the written rows in order
    for b in range(2):
        lo, hi = s["qsl"][b], s["qsl"][b + 1]
        Kb = O.gather_kv(kc, s["block_table"][b], int(s["seq_lens"][b]), bs)
        Vb = O.gather_kv(vc, s["block_table"][b], int(s["seq_lens"][b]), bs)
        p = s["positions"][lo:hi]
        assert np.array_equal(Kb[p], O.round_to_bf16(k[lo:hi]))
        assert np.array_equal(Vb[p], O.round_to_bf16(v[lo:hi]))
    # exactly T*nkv*d elements changed per cache; skipped tokens (slot < 0) write nothing
    slots2 = slots.copy()
    slots2[1] = -1
    kc2, vc2 = s["k"].copy(), s["v"].copy()
    O.kv_cache_write(k, v, slots2, kc2, vc2, bs)
    blk, off = divmod(int(slots[1]), bs)
    assert np.array_equal(kc2[blk, :, off], s["k"][blk, :, off])


def test_greedy_argmax_ties_and_gap():
    lg = np.array([[0.0, 3.0, 3.0, 1.0], [5.0, -1.0, 4.5, 4.9]])
    tok, gap = O.greedy_argmax(lg)
    assert tok.tolist() == [1, 0]
    assert gap.tolist() == [0.0, pytest.approx(0.1)]
    x = RNG.standard_normal((6, 1000))
    assert np.array_equal(O.greedy_argmax(x)[0], np.argmax(x, axis=-1))


# --------------------------------------------------------------------------- whole layer

def tiny_shape(hidden=64, nq=4, nkv=2, d=16, inter=48, scaling=None, theta=10000.0, bs=4):
    return O.LayerShape(hidden=hidden, n_heads=nq, n_kv_heads=nkv, head_dim=d, intermediate=inter, rms_eps=1e-5,
                        rope_theta=theta, rope_scaling=scaling, block_size=bs)


def tiny_weights(sh, rng, std=0.2):
    qkv = (sh.n_heads + 2 * sh.n_kv_heads) * sh.head_dim
    return O.LayerWeights(
        ln1=1 + 0.1 * rng.standard_normal(sh.hidden), w_qkv=std * rng.standard_normal((qkv, sh.hidden)),
        w_o=std * rng.standard_normal((sh.hidden, sh.q_size)), ln2=1 + 0.1 * rng.standard_normal(sh.hidden),
        w_gate_up=std * rng.standard_normal((2 * sh.intermediate, sh.hidden)),
        w_down=std * rng.standard_normal((sh.hidden, sh.intermediate)))


def check_fused_equals_unfused(scaling=None):
    sh = tiny_shape(scaling=scaling, theta=500000.0 if scaling else 10000.0)
    rng = np.random.default_rng(41)
    w = tiny_weights(sh, rng)
    s = _paged_setup([6, 0, 3], [1, 7, 4], sh.n_kv_heads, sh.head_dim, bs=sh.block_size, seed=13)
    batch = O.Batch(s["positions"], s["qsl"], s["seq_lens"], s["block_table"])
    T = int(s["qsl"][-1])
    x = rng.standard_normal((T, sh.hidden))
    res = rng.standard_normal((T, sh.hidden))
    kc1, vc1 = s["k"].copy(), s["v"].copy()
    out, r2 = O.decoder_layer(sh, w, batch, x, res, kc1, vc1, bf16_tensors=False)
    kc2, vc2 = s["k"].copy(), s["v"].copy()
    want = O.decoder_layer_unfused(sh, w, batch, x + res, kc2, vc2)
    assert np.max(np.abs(out + r2 - want)) < 1e-10
    assert np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2)
    # residual None: the layer's residual output starts from the raw input
    kc3, vc3 = s["k"].copy(), s["v"].copy()
    out3, r3 = O.decoder_layer(sh, w, batch, x, None, kc3, vc3, bf16_tensors=False)
    want3 = O.decoder_layer_unfused(sh, w, batch, x, s["k"].copy(), s["v"].copy())
    assert np.max(np.abs(out3 + r3 - want3)) < 1e-10
    # rows subset gives the same rows as the full evaluation
    kc4, vc4 = s["k"].copy(), s["v"].copy()
    rows = [0, 4, 9]
    out4, r4 = O.decoder_layer(sh, w, batch, x, res, kc4, vc4, rows=rows, bf16_tensors=False)
    assert np.max(np.abs(out4[rows] - out[rows])) < 1e-12 and np.array_equal(r4[rows], r2[rows])


def test_fused_layer_equals_unfused_prenorm():
    check_fused_equals_unfused(None)
    check_fused_equals_unfused(O_LLAMA3)


def test_merged_qkv_equals_separate_projections():
    sh = tiny_shape()
    rng = np.random.default_rng(3)
    w = tiny_weights(sh, rng)
    h = rng.standard_normal((5, sh.hidden))
    qkv = O.linear(h, w.w_qkv)
    wq = w.w_qkv[:sh.q_size]
    wk = w.w_qkv[sh.q_size:sh.q_size + sh.kv_size]
    wv = w.w_qkv[sh.q_size + sh.kv_size:]
    assert np.max(np.abs(qkv - np.concatenate([O.linear(h, wq), O.linear(h, wk), O.linear(h, wv)], 1))) < 1e-12
    gu = O.linear(h, w.w_gate_up)
    I = sh.intermediate
    sep = O.silu(O.linear(h, w.w_gate_up[:I])) * O.linear(h, w.w_gate_up[I:])
    assert np.max(np.abs(O.silu_and_mul(gu) - sep)) < 1e-12


def _bf16_scalar(v):
    """bf16 value of a Python float (round to nearest even), by integer
    arithmetic on the float32 bit pattern."""
    import struct
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def brute_layer(sh, w, positions, seq_of, seq_lens, x, res, kcache, vcache, bt, bf16=False):
    """Scalar-loop restatement of the layer on tiny shapes (contiguous per-token
    K/V lists are rebuilt from a dict of written positions).  ``bf16`` stores
    every module output in bf16, as the layer-level oracle does by default."""
    T, H = len(x), sh.hidden
    rn = (lambda vec: [_bf16_scalar(e) for e in vec]) if bf16 else (lambda vec: vec)
    d, nq, nkv = sh.head_dim, sh.n_heads, sh.n_kv_heads

    def rms(v, g):
        ms = sum(e * e for e in v) / len(v)
        return [e / math.sqrt(ms + sh.rms_eps) * gg for e, gg in zip(v, g)]

    def mv(W, v):
        return [sum(W[o][i] * v[i] for i in range(len(v))) for o in range(len(W))]

    inv = O.rope_inv_freq(d, sh.rope_theta, sh.rope_scaling).tolist()

    def rot(vec, p):
        half = d // 2
        out = list(vec)
        for i in range(half):
            c, s_ = math.cos(p * inv[i]), math.sin(p * inv[i])
            out[i] = vec[i] * c - vec[i + half] * s_
            out[i + half] = vec[i + half] * c + vec[i] * s_
        return out

    r = [rn([x[t][i] + (res[t][i] if res is not None else 0.0) for i in range(H)]) for t in range(T)]
    hs = [rn(rms(r[t], w.ln1.tolist())) for t in range(T)]
    Wqkv, q_all = w.w_qkv.tolist(), []
    kv_new = {}
    for t in range(T):
        qkv = rn(mv(Wqkv, hs[t]))
        q = [rn(rot(qkv[h * d:(h + 1) * d], positions[t])) for h in range(nq)]
        k = [rot(qkv[sh.q_size + h * d: sh.q_size + (h + 1) * d], positions[t]) for h in range(nkv)]
        v = [qkv[sh.q_size + sh.kv_size + h * d: sh.q_size + sh.kv_size + (h + 1) * d] for h in range(nkv)]
        q_all.append(q)
        # bf16 storage of the cache
        kv_new[(seq_of[t], positions[t])] = ([O.round_to_bf16(np.array(e, np.float32)).astype(float).tolist() for e in k],
                                             [O.round_to_bf16(np.array(e, np.float32)).astype(float).tolist() for e in v])
    outs, r2s = [], []
    for t in range(T):
        b, p = seq_of[t], positions[t]
        o = []
        for h in range(nq):
            kh = h // (nq // nkv)
            K, V = [], []
            for j in range(p + 1):
                if (b, j) in kv_new:
                    K.append(kv_new[(b, j)][0][kh])
                    V.append(kv_new[(b, j)][1][kh])
                else:
                    blk = bt[b][j // sh.block_size]
                    K.append(O.bf16_bits_to_float(kcache[blk, kh, j % sh.block_size]).astype(float).tolist())
                    V.append(O.bf16_bits_to_float(vcache[blk, kh, j % sh.block_size]).astype(float).tolist())
            o += brute_attention(q_all[t][h], K, V, p, 1 / math.sqrt(d))
        o = rn(o)
        y = rn(mv(w.w_o.tolist(), o))
        r2 = rn([y[i] + r[t][i] for i in range(H)])
        h2 = rn(rms(r2, w.ln2.tolist()))
        gu = rn(mv(w.w_gate_up.tolist(), h2))
        I = sh.intermediate
        a = rn([gu[i] / (1 + math.exp(-gu[i])) * gu[I + i] for i in range(I)])
        outs.append(rn(mv(w.w_down.tolist(), a)))
        r2s.append(r2)
    return np.array(outs), np.array(r2s)


def check_layer_brute_force(scaling=None, residual=True, bf16=False):
    sh = tiny_shape(hidden=32, nq=4, nkv=2, d=8, inter=24, scaling=scaling,
                    theta=500000.0 if scaling else 10000.0, bs=2)
    rng = np.random.default_rng(77)
    w = tiny_weights(sh, rng, std=0.3)
    s = _paged_setup([3, 0], [2, 3], sh.n_kv_heads, sh.head_dim, bs=sh.block_size, seed=17)
    batch = O.Batch(s["positions"], s["qsl"], s["seq_lens"], s["block_table"])
    T = int(s["qsl"][-1])
    x = rng.standard_normal((T, sh.hidden))
    res = rng.standard_normal((T, sh.hidden)) if residual else None
    kc, vc = s["k"].copy(), s["v"].copy()
    out, r2 = O.decoder_layer(sh, w, batch, x, res, kc, vc, bf16_tensors=bf16)
    seq_of = O.token_sequence(s["qsl"]).tolist()
    bo, br = brute_layer(sh, w, s["positions"].tolist(), seq_of, s["seq_lens"].tolist(), x.tolist(),
                         None if res is None else res.tolist(), s["k"], s["v"], s["block_table"].tolist(), bf16=bf16)
    if bf16:
        # both sides store module outputs in bf16; the fp64 arithmetic inside may
        # put a value on the other side of a bf16 rounding boundary in rare
        # cases: allow one bf16 ulp on a few elements, exact elsewhere
        ulp = np.abs(bo) * 2.0 ** -7 + 1e-30
        bad = np.abs(out - bo) > 1e-9 * np.maximum(1.0, np.abs(bo))
        assert np.all(np.abs(out - bo)[bad] <= ulp[bad] * 1.01) and bad.mean() < 0.02
        assert np.max(np.abs(r2 - br)) <= 2.0 ** -7 * np.max(np.abs(br))
    else:
        assert np.max(np.abs(out - bo)) < 1e-9 * max(1.0, np.max(np.abs(bo)))
        assert np.max(np.abs(r2 - br)) < 1e-12


def test_layer_brute_force():
    check_layer_brute_force(None, True)
    check_layer_brute_force(O_LLAMA3, False)


def test_layer_brute_force_bf16_module_outputs():
    check_layer_brute_force(None, True, bf16=True)
    check_layer_brute_force(O_LLAMA3, False, bf16=True)


def check_stack_composition():
    sh = tiny_shape()
    rng = np.random.default_rng(5)
    layers = [tiny_weights(sh, rng) for _ in range(3)]
    fnorm = 1 + 0.1 * rng.standard_normal(sh.hidden)
    lm = 0.2 * rng.standard_normal((50, sh.hidden))
    s = _paged_setup([4, 0], [1, 6], sh.n_kv_heads, sh.head_dim, bs=sh.block_size, seed=19)
    batch = O.Batch(s["positions"], s["qsl"], s["seq_lens"], s["block_table"])
    T = int(s["qsl"][-1])
    x = rng.standard_normal((T, sh.hidden))
    kcs = [s["k"].copy() for _ in range(3)]
    vcs = [s["v"].copy() for _ in range(3)]
    tok, gap, logits, hf = O.stack_forward(sh, layers, fnorm, lm, batch, x, kcs, vcs, bf16_tensors=False)
    # unfused model: hidden = layer(hidden) with the residual inside, then norm(hidden)
    hid = x.copy()
    for li in range(3):
        hid = O.decoder_layer_unfused(sh, layers[li], batch, hid, s["k"].copy(), s["v"].copy())
    rows = O.last_token_rows(s["qsl"])
    want = O.rms_norm(hid[rows], fnorm, sh.rms_eps)
    assert np.max(np.abs(hf - want)) < 1e-10
    assert np.max(np.abs(logits - want @ lm.T)) < 1e-9
    assert np.array_equal(tok, np.argmax(want @ lm.T, axis=-1))


def test_stack_composition():
    check_stack_composition()


def test_activation_guard():
    sh = O.LayerShape(64, 4, 2, 16, 48, 1e-5, 1e4, None, hidden_act="gelu")
    with pytest.raises(ValueError):
        O.mlp_block(sh, tiny_weights(tiny_shape(), np.random.default_rng(0)), np.zeros((1, 64)))


# --------------------------------------------------------------------------- golden config

def test_golden_config_matches_workloads():
    """Values printed on the 70B page (model config and the q/kv head split)
    against the workload definitions used by tests and the bench."""
    from llama_decoder_layer_gb300.inputs import SPECS
    with open(os.path.join(GOLDEN, "llama70b_config.json")) as f:
        g = json.load(f)
    assert g["num_attention_heads"] * g["head_dim"] == g["q_size"] == 8192
    assert g["num_key_value_heads"] * g["head_dim"] == g["kv_size"] == 1024
    for name in ("decode_70b", "prefill_70b", "stack_70b"):
        sp = SPECS[name]
        assert sp.hidden == g["hidden_size"] and sp.intermediate == g["intermediate_size"]
        assert sp.n_heads == g["num_attention_heads"] and sp.n_kv_heads == g["num_key_value_heads"]
        assert sp.head_dim == g["head_dim"] and sp.rms_eps == g["rms_norm_eps"]
        assert sp.rope_theta == g["rope_theta"]
        sc = dict(sp.rope_scaling)
        for k_, v_ in g["rope_scaling"].items():
            assert sc[k_] == v_
    assert SPECS["stack_70b"].vocab == g["vocab_size"]


def test_golden_qwen3_moe_config_matches_workloads():
    """Values printed on the 70B page's Qwen3MoeForCausalLM section against the
    MoE workload definitions (every layer sparse, no rope scaling)."""
    from llama_decoder_layer_gb300.inputs import SPECS
    with open(os.path.join(GOLDEN, "qwen3_30b_a3b_config.json")) as f:
        g = json.load(f)
    assert g["num_attention_heads"] * g["head_dim"] == g["q_size"] == 4096
    assert g["num_key_value_heads"] * g["head_dim"] == g["kv_size"] == 512
    assert g["decoder_sparse_step"] == 1 and g["mlp_only_layers"] == [] and g["norm_topk_prob"] is True
    for name in ("qwen3_moe", "qwen3_moe_decode", "qwen3_moe_prefill"):
        sp = SPECS[name]
        assert sp.hidden == g["hidden_size"] and sp.intermediate == g["intermediate_size"]
        assert sp.n_heads == g["num_attention_heads"] and sp.n_kv_heads == g["num_key_value_heads"]
        assert sp.head_dim == g["head_dim"] and sp.rms_eps == g["rms_norm_eps"]
        assert sp.rope_theta == g["rope_theta"] and sp.rope_scaling is None and g["rope_scaling"] is None
        assert sp.extra["num_experts"] == g["num_experts"]
        assert sp.extra["top_k"] == g["num_experts_per_tok"]
        assert sp.extra["moe_intermediate"] == g["moe_intermediate_size"]
