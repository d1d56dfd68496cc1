"""Plant plausible mistakes in the oracle (on the CPU) and show that the pins in
``test_oracle_pins.py`` catch each of them: a dropped term, a wrong sign or
index, a transposed operand, a swapped half."""

import math

import numpy as np
import pytest

import tests.test_oracle_pins as P
from oracle import llama_oracle as O


def _mut_rms_eps_outside(x, gamma, eps, dtype=np.float64):
    x = np.asarray(x, dtype=dtype)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * gamma


def _mut_rms_sum(x, gamma, eps, dtype=np.float64):
    x = np.asarray(x, dtype=dtype)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * gamma


def _mut_fused_returns_normed(x, residual, gamma, eps, dtype=np.float64):
    r = np.asarray(x, dtype=dtype) + (0 if residual is None else np.asarray(residual, dtype=dtype))
    h = O.rms_norm(r, gamma, eps, dtype)
    return h, h


def _mut_silu_swapped(x, dtype=np.float64):
    x = np.asarray(x, dtype=dtype)
    d = x.shape[-1] // 2
    return O.silu(x[..., d:], dtype) * x[..., :d]


def _mut_linear_transposed(x, weight, dtype=np.float64):
    w = np.asarray(weight, dtype=dtype)
    return np.asarray(x, dtype=dtype) @ (w.T if w.shape[0] == w.shape[1] else w.T[:, ::-1])


def _mut_rope_sign(x, positions, inv_freq, dtype=np.float64):
    x = np.asarray(x, dtype=dtype)
    half = x.shape[-1] // 2
    ang = np.asarray(positions, np.float64)[:, None] * np.asarray(inv_freq)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    out = np.empty_like(x)
    out[..., :half] = x[..., :half] * c + x[..., half:] * s
    out[..., half:] = x[..., half:] * c + x[..., :half] * s
    return out


def _mut_rope_interleaved(x, positions, inv_freq, dtype=np.float64):
    x = np.asarray(x, dtype=dtype)
    ang = np.asarray(positions, np.float64)[:, None] * np.asarray(inv_freq)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return out


_orig_inv = O.rope_inv_freq


def _mut_llama3_bands_swapped(head_dim, theta, scaling=None):
    base = _orig_inv(head_dim, theta, None)
    if scaling is None:
        return base
    out = base.copy()
    lam = 2 * math.pi / base
    orig = scaling["original_max_position_embeddings"]
    out[lam < orig / scaling["high_freq_factor"]] /= scaling["factor"]
    return out


_orig_attn = O.paged_attention


def _mut_attn_gqa_modulo(q, k_cache_bits, v_cache_bits, block_table, seq_lens, query_start_loc, positions,
                         n_kv_heads, block_size, rows=None, dtype=np.float64):
    q = np.asarray(q, dtype=dtype)
    T, nq, d = q.shape
    seq = O.token_sequence(query_start_loc)
    out = np.zeros_like(q)
    for t in range(T):
        b = int(seq[t])
        n = int(seq_lens[b])
        K = O.gather_kv(k_cache_bits, block_table[b], n, block_size).astype(dtype)
        V = O.gather_kv(v_cache_bits, block_table[b], n, block_size).astype(dtype)
        p = int(positions[t])
        for h in range(nq):
            kh = h % n_kv_heads
            s = K[:p + 1, kh] @ q[t, h] / math.sqrt(d)
            w = np.exp(s - s.max())
            out[t, h] = (w / w.sum()) @ V[:p + 1, kh]
    return out


def _mut_attn_no_causal(q, k_cache_bits, v_cache_bits, block_table, seq_lens, query_start_loc, positions,
                        n_kv_heads, block_size, rows=None, dtype=np.float64):
    seq = O.token_sequence(query_start_loc)
    last = np.array([int(seq_lens[b]) - 1 for b in seq])
    return _orig_attn(q, k_cache_bits, v_cache_bits, block_table, seq_lens, query_start_loc, last,
                      n_kv_heads, block_size, rows=rows, dtype=dtype)


def _mut_attn_scale(q, *a, **kw):
    d = np.asarray(q).shape[-1]
    return _orig_attn(np.asarray(q) / math.sqrt(d), *a, **kw)


def _mut_slot_off_by_one(positions, query_start_loc, block_table, block_size):
    seq = O.token_sequence(query_start_loc)
    bt = np.asarray(block_table)
    return np.array([bt[b, (p + 1) // block_size] * block_size + (p + 1) % block_size
                     if (p + 1) // block_size < bt.shape[1] and bt[b, (p + 1) // block_size] >= 0
                     else bt[b, p // block_size] * block_size
                     for b, p in zip(seq, np.asarray(positions))])


_orig_layer = O.decoder_layer


def _mut_layer_residual_dropped(shape, w, batch, hidden, residual, kc, vc, rows=None, dtype=np.float64,
                                bf16_tensors=True):
    h, r = O.fused_add_rms_norm(hidden, residual, w.ln1, shape.rms_eps, dtype, bf16_tensors)
    y = O.attention_block(shape, w, batch, h, kc, vc, rows=rows, dtype=dtype, bf16_tensors=bf16_tensors)
    h2, r2 = O.fused_add_rms_norm(y, None, w.ln2, shape.rms_eps, dtype, bf16_tensors)
    return O.mlp_block(shape, w, h2, dtype, bf16_tensors), r2


MUTANTS = [
    ("rms_norm", _mut_rms_eps_outside, P.check_rms_norm),
    ("rms_norm", _mut_rms_sum, P.check_rms_norm),
    ("fused_add_rms_norm", _mut_fused_returns_normed, P.check_fused_add_norm),
    ("silu_and_mul", _mut_silu_swapped, P.check_silu_and_mul),
    ("linear", _mut_linear_transposed, P.check_linear),
    ("apply_rope", _mut_rope_sign, P.check_rope_invariants),
    ("apply_rope", _mut_rope_interleaved, P.check_rope_rotation_closed_form),
    ("rope_inv_freq", _mut_llama3_bands_swapped, P.check_llama3_bands),
    ("paged_attention", _mut_attn_gqa_modulo, P.check_gqa_equals_mha),
    ("paged_attention", _mut_attn_no_causal, P.check_attention_vs_sdpa),
    ("paged_attention", _mut_attn_scale, P.check_attention_vs_sdpa),
    ("paged_attention", _mut_attn_scale, P.check_attention_brute_force),
    ("slot_mapping", _mut_slot_off_by_one, P.test_slot_mapping_and_cache_write_roundtrip),
    ("decoder_layer", _mut_layer_residual_dropped, lambda: P.check_fused_equals_unfused(None)),
    ("rms_norm", _mut_rms_eps_outside, lambda: P.check_layer_brute_force(None, True)),
    ("silu_and_mul", _mut_silu_swapped, lambda: P.check_layer_brute_force(None, True)),
    ("apply_rope", _mut_rope_sign, lambda: P.check_layer_brute_force(None, True)),
    ("silu_and_mul", _mut_silu_swapped, lambda: P.check_layer_brute_force(None, True, bf16=True)),
]


@pytest.mark.parametrize("name,mutant,check", MUTANTS,
                         ids=[f"{n}-{m.__name__}" for n, m, _ in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, mutant, check):
    monkeypatch.setattr(O, name, mutant)
    with pytest.raises(Exception):
        check()


def test_unmutated_checks_pass():
    for _, _, check in MUTANTS:
        check()
