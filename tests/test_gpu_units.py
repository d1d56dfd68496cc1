"""Parity of each CUDA kernel against the oracle on small seeded inputs that
span several tiles and ragged tails (GPU)."""

import dataclasses

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O
from tests.helpers import (assert_close, bits, check_cache, f32, oracle_batch, oracle_shape, oracle_weights,
                           written_slot_mask)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


def _ws(n):
    return torch.empty(n, dtype=torch.uint8, device=DEV)


# ----------------------------------------------------------------- GEMM


# tiles = ceil(M/128) * ceil(N/256) against the SM count (152 on GB300): at most
# half of it -> split-K over a cluster, below it -> stream-K + fixup, from it
# on -> data-parallel.  Ragged M, N and K tails throughout.
@pytest.mark.parametrize("M,N,K", [
    (37, 768, 512), (128, 1024, 1376), (300, 1000, 512),      # cluster split-K (S = 4, 8, 4)
    (1, 256, 64), (64, 30720, 512), (200, 15360, 256),        # stream-K (one k-block; 120 tiles; 2 M-tiles)
    (1500, 2304, 192),                                        # stream-K, 108 tiles of 12 M-tiles
    (64, 40960, 512), (4096, 4096, 256),                      # data-parallel (160 tiles: one and a bit waves)
])
def test_linear_bf16(M, N, K):
    x = I.normal_bf16((M, K), 1.0, 0.0, 11 + M, DEV)
    w = I.normal_bf16((N, K), 0.02, 0.0, 12 + N, DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    lb.linear(x, w, y, _ws(lb.linear_workspace_size()))
    torch.cuda.synchronize()
    ref = O.linear(f32(x), f32(w))
    assert_close(f32(y), ref, f"linear {M}x{N}x{K}")


def test_linear_fp32_out_and_repeat():
    M, N, K = 34, 2048, 1024
    x = I.normal_bf16((M, K), 1.0, 0.0, 5, DEV)
    w = I.normal_bf16((N, K), 0.02, 0.0, 6, DEV)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = _ws(lb.linear_workspace_size())
    lb.linear(x, w, y, ws)
    y1 = y.clone()
    lb.linear(x, w, y, ws)
    torch.cuda.synchronize()
    assert torch.equal(y, y1), "split-K reduction is not deterministic"
    ref = O.linear(f32(x), f32(w))
    e = assert_close(f32(y), ref, "linear fp32")
    assert e < 1e-3  # fp32 output: only accumulation-order differences


# ----------------------------------------------------------------- RMSNorm


@pytest.mark.parametrize("H,rows", [(512, 7), (4096, 33), (8192, 130)])
def test_fused_add_rmsnorm(H, rows):
    x = I.normal_bf16((rows, H), 1.0, 0.0, 1, DEV)
    r = I.normal_bf16((rows, H), 1.0, 0.0, 2, DEV)
    g = I.normal_bf16((H,), 0.02, 1.0, 3, DEV)
    h = torch.empty_like(x)
    ro = torch.empty_like(x)
    lb.fused_add_rmsnorm(x, r, ro, h, g, 1e-5)
    h0 = torch.empty_like(x)
    ro0 = torch.empty_like(x)
    lb.fused_add_rmsnorm(x, None, ro0, h0, g, 1e-5)
    # in place: residual_out aliases residual_in and h aliases x
    x2, r2 = x.clone(), r.clone()
    lb.fused_add_rmsnorm(x2, r2, r2, x2, g, 1e-5)
    torch.cuda.synchronize()
    hr, rr = O.fused_add_rms_norm(f32(x), f32(r), f32(g), 1e-5)
    assert_close(f32(h), hr, "h")
    assert_close(f32(ro), rr, "residual")
    hr0, rr0 = O.fused_add_rms_norm(f32(x), None, f32(g), 1e-5)
    assert_close(f32(h0), hr0, "h (residual None)")
    assert np.array_equal(bits(ro0), bits(x)), "residual None must pass the input through unchanged"
    assert torch.equal(x2, h) and torch.equal(r2, ro), "in-place result differs"


# ----------------------------------------------------------------- cache write


def test_kv_cache_write_bit_exact():
    T, nkv, d, nb, bs = 300, 8, 128, 40, 16
    k = I.normal_bf16((T, nkv, d), 1.0, 0.0, 7, DEV)
    v = I.normal_bf16((T, nkv, d), 1.0, 0.0, 8, DEV)
    slots = I.random_slots(T, nb, bs, seed=3, skip_every=7).to(DEV)
    kc = I.normal_bf16((nb, nkv, bs, d), 1.0, 0.0, 9, DEV)
    vc = I.normal_bf16((nb, nkv, bs, d), 1.0, 0.0, 10, DEV)
    kb, vb = bits(kc), bits(vc)
    lb.kv_cache_write(k, v, slots, kc, vc, bs)
    torch.cuda.synchronize()
    O.kv_cache_write(f32(k), f32(v), slots.cpu().numpy(), kb, vb, bs)
    assert np.array_equal(bits(kc), kb) and np.array_equal(bits(vc), vb)
    assert lb.get_device_error()[0] == lb.LLAMA_OK


def test_kv_cache_write_guard():
    T, nkv, d, nb, bs = 4, 2, 64, 3, 16
    k = I.normal_bf16((T, nkv, d), 1.0, 0.0, 7, DEV)
    v = I.normal_bf16((T, nkv, d), 1.0, 0.0, 8, DEV)
    slots = torch.tensor([0, 5, nb * bs + 3, 17], dtype=torch.int32, device=DEV)
    kc = torch.zeros((nb, nkv, bs, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    lb.kv_cache_write(k, v, slots, kc, vc, bs)
    st, where = lb.get_device_error()
    assert st == lb.LLAMA_ERR_DEVICE_GUARD
    assert torch.equal(kc[0, :, 0], k[0]) and torch.equal(kc[1, :, 1], k[3])
    assert lb.get_device_error()[0] == lb.LLAMA_OK  # cleared


# ----------------------------------------------------------------- attention


def _attn_case(nq, nkv, d, groups, seed):
    spec = dataclasses.replace(I.SPECS["tiny"], n_heads=nq, n_kv_heads=nkv, head_dim=d, hidden=nq * d,
                               groups=groups)
    bl = I.make_batch(spec, seed, DEV)
    q = I.normal_bf16((bl.num_tokens, nq, d), 1.0, 0.0, seed + 1, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, DEV)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    out = torch.empty((bl.num_tokens, nq * d), dtype=torch.bfloat16, device=DEV)
    ws = _ws(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len))
    lb.paged_attention(cfg, batch, q, kc, vc, out, ws)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    ob = oracle_batch(bl)
    ref = O.paged_attention(f32(q), bits(kc), bits(vc), ob.block_table, ob.seq_lens, ob.query_start_loc,
                            ob.positions, nkv, 16)
    return f32(out).reshape(ref.shape), ref


@pytest.mark.parametrize("nq,nkv,d", [(8, 2, 64), (16, 2, 128), (64, 8, 128)])
def test_attention_decode(nq, nkv, d):
    # contexts 0 (one visible key), 15, 16 (block edges), 1535/1536 (where a sequence goes from one
    # split-KV chunk to two), up to 5000 (4 chunks of decreasing length)
    groups = (("decode", 1, 1, 0, 0), ("decode", 1, 1, 15, 15), ("decode", 1, 1, 16, 16),
              ("decode", 1, 1, 1535, 1535), ("decode", 1, 1, 1536, 1536), ("decode", 5, 1, 1, 5000))
    g, r = _attn_case(nq, nkv, d, groups, 21)
    assert_close(g, r, "decode attention")


@pytest.mark.parametrize("nq,nkv,d", [(8, 2, 64), (16, 2, 128), (64, 8, 128)])
def test_attention_prefill(nq, nkv, d):
    # fresh prefill with ragged lengths, and chunked prefill on top of a cached prefix
    groups = (("prefill", 1, 2, 0, 0), ("prefill", 1, 37, 0, 0), ("prefill", 1, 130, 0, 0),
              ("prefill", 2, 21, 3, 90))
    g, r = _attn_case(nq, nkv, d, groups, 31)
    assert_close(g, r, "prefill attention")


def test_attention_mixed_batch():
    groups = (("decode", 4, 1, 20, 4000), ("prefill", 2, 50, 0, 0), ("decode", 2, 1, 0, 40),
              ("prefill", 1, 17, 30, 30))
    g, r = _attn_case(16, 2, 128, groups, 41)
    assert_close(g, r, "mixed attention")


# ----------------------------------------------------------------- whole layer (tiny)


def _run_layer(spec, seed=0, residual_none=None):
    bl = I.make_batch(spec, seed, DEV)
    w = I.make_layer_weights(spec, seed, 0, DEV)
    x, r = I.make_activations(spec, bl.num_tokens, seed, DEV)
    if residual_none is not None:
        r = None if residual_none else I.normal_bf16(x.shape, 1.0, 0.0, seed + 99, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, DEV)
    kb0, vb0 = bits(kc), bits(vc)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    ws = _ws(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len))
    hid = x.clone()
    res_out = torch.empty_like(x)
    lb.layer_forward(cfg, w, batch, hid, r, res_out, kc, vc, ws)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    kref, vref = kb0.copy(), vb0.copy()
    out, res = O.decoder_layer(oracle_shape(spec), oracle_weights(w), oracle_batch(bl), f32(x),
                               None if r is None else f32(r), kref, vref)
    wm = written_slot_mask(bl, bl.num_blocks)
    assert_close(f32(hid), out, "hidden_states")
    assert_close(f32(res_out), res, "residual")
    check_cache(bits(kc), kref, kb0, wm, "k_cache")
    check_cache(bits(vc), vref, vb0, wm, "v_cache")


def test_layer_tiny():
    _run_layer(I.SPECS["tiny"])


def test_layer_tiny_literal_gamma():
    _run_layer(dataclasses.replace(I.SPECS["tiny"], literal_gamma=True))


def test_layer_tiny_chunked_prefill_with_residual():
    spec = dataclasses.replace(I.SPECS["tiny"], groups=(("prefill", 2, 20, 5, 40), ("decode", 3, 1, 10, 600)))
    _run_layer(spec, seed=3, residual_none=False)


def test_layer_tiny_llama3_rope():
    spec = dataclasses.replace(I.SPECS["tiny"], rope_theta=500000.0, rope_scaling=I.LLAMA3_SCALING,
                               groups=(("decode", 4, 1, 3000, 9000), ("prefill", 1, 40, 8000, 8000)))
    _run_layer(spec, seed=5, residual_none=False)


def test_layer_device_guard_bad_block_table():
    spec = I.SPECS["tiny"]
    bl = I.make_batch(spec, 0, DEV)
    w = I.make_layer_weights(spec, 0, 0, DEV)
    x, _ = I.make_activations(spec, bl.num_tokens, 0, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, 0, 0, DEV)
    bl.block_table[1, 0] = bl.num_blocks + 7  # out of range
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    ws = _ws(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len))
    res = torch.empty_like(x)
    lb.layer_forward(cfg, w, batch, x, None, res, kc, vc, ws)
    st, where = lb.get_device_error()
    assert st == lb.LLAMA_ERR_DEVICE_GUARD
    # the context stays usable
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    y = torch.ones(4, device=DEV) * 2
    assert float(y.sum()) == 8.0


def test_host_argument_errors():
    spec = I.SPECS["tiny"]
    cfg = lb.LayerConfig.from_spec(spec)
    bl = I.make_batch(spec, 0, DEV)
    w = I.make_layer_weights(spec, 0, 0, DEV)
    x, _ = I.make_activations(spec, bl.num_tokens, 0, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, 0, 0, DEV)
    batch = lb.Batch.from_layout(bl)
    ws = _ws(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len))
    res = torch.empty_like(x)
    with pytest.raises(lb.LlamaError) as e:
        lb.layer_forward(cfg, w, batch, x, None, res, kc, vc, ws[:1000])
    assert e.value.status == lb.LLAMA_ERR_WORKSPACE
    bad = dataclasses.replace(cfg, hidden_act="gelu")
    with pytest.raises(lb.LlamaError) as e:
        lb.layer_forward(bad, w, batch, x, None, res, kc, vc, ws)
    assert e.value.status == lb.LLAMA_ERR_ARG
    bad = dataclasses.replace(cfg, n_kv_heads=3)
    with pytest.raises(lb.LlamaError) as e:
        lb.layer_forward(bad, w, batch, x, None, res, kc, vc, ws)
    assert e.value.status == lb.LLAMA_ERR_ARG
