"""The projection GEMM under each of its schedules (GPU): whole 128 x 256 tiles
on single SMs, 256 x 256 tiles on SM pairs (tcgen05 pair MMAs from a 2-CTA
cluster), stream-K and cluster split-K, forced through llama_set_gemm_schedule.

Every schedule must match the oracle's product within the tolerance, on shapes
with ragged M, N and K tails (M tails that leave the second CTA of a pair
without a valid row, or with only part of one); the single-SM and SM-pair
schedules sum K in the same order and must agree bit for bit.  Each of the
four epilogues (bf16, fp32, SwiGLU, and the qkv epilogue with RoPE and the
paged-cache scatter, through a whole decoder layer) runs on SM pairs.
[WALKTHROUGH] "模型库与算子层 — 代码走读", Linear layers (F.linear with
Parameter(out, in)); [LLAMA-70B] "LLama — DeepSeek-R1-Distill-Llama-70B",
LlamaMLP / SiluAndMul.
"""

import dataclasses

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O
from tests.helpers import assert_close, bits, f32, oracle_batch, oracle_shape, oracle_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"
SINGLE, STREAM_K, CLUSTER, PAIR = 0, 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


@pytest.fixture(autouse=True)
def _automatic_schedule_after():
    yield
    lb.set_gemm_schedule(-1)


def _ws():
    return torch.empty(lb.linear_workspace_size(), dtype=torch.uint8, device=DEV)


def _linear(x, w, out_dtype, schedule):
    lb.set_gemm_schedule(schedule)
    y = torch.empty((x.shape[0], w.shape[0]), dtype=out_dtype, device=DEV)
    lb.linear(x, w, y, _ws())
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    return y


@pytest.mark.parametrize("M,N,K", [
    (300, 1000, 520),    # ragged everything; 2 pair rows, the second CTA of the last one 44 rows
    (129, 512, 64),      # one valid row in the second CTA of the pair
    (128, 768, 192),     # the second CTA of the pair has no valid row
    (1, 256, 64),        # a single row
    (4128, 2304, 256),   # the stack's row count: 16 full pair rows and a 32-row tail
])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_pair_and_single_sm_tiles_agree_and_match_the_oracle(M, N, K, out_dtype):
    x = I.normal_bf16((M, K), 1.0, 0.0, 21 + M, DEV)
    w = I.normal_bf16((N, K), 0.02, 0.0, 22 + N, DEV)
    y_pair = _linear(x, w, out_dtype, PAIR)
    y_single = _linear(x, w, out_dtype, SINGLE)
    assert torch.equal(y_pair, y_single), "SM-pair tiles differ from single-SM tiles"
    ref = O.linear(f32(x), f32(w))
    if out_dtype == torch.bfloat16:
        ref = O.round_to_bf16(ref)
    assert_close(f32(y_pair), ref, f"pair linear {M}x{N}x{K}")


@pytest.mark.parametrize("schedule", [STREAM_K, CLUSTER])
def test_other_schedules_match_the_oracle(schedule):
    M, N, K = 300, 1000, 520
    x = I.normal_bf16((M, K), 1.0, 0.0, 31, DEV)
    w = I.normal_bf16((N, K), 0.02, 0.0, 32, DEV)
    y = _linear(x, w, torch.float32, schedule)
    assert_close(f32(y), O.linear(f32(x), f32(w)), f"schedule {schedule}")


@pytest.mark.parametrize("M,I_,K", [(300, 1376, 512), (4128, 1536, 256), (129, 256, 128)])
def test_pair_swiglu_epilogue(M, I_, K):
    x = I.normal_bf16((M, K), 1.0, 0.0, 41 + M, DEV)
    w = I.normal_bf16((2 * I_, K), 0.02, 0.0, 42 + I_, DEV)
    outs = {}
    for schedule in (PAIR, SINGLE):
        lb.set_gemm_schedule(schedule)
        a = torch.empty((M, I_), dtype=torch.bfloat16, device=DEV)
        lb.gate_up_silu(x, w, a, _ws())
        torch.cuda.synchronize()
        assert lb.get_device_error()[0] == lb.LLAMA_OK
        outs[schedule] = a
    assert torch.equal(outs[PAIR], outs[SINGLE]), "SM-pair SwiGLU differs from single-SM tiles"
    # gate_up_proj's bf16 output, then SiluAndMul's bf16 output
    gu = O.store(O.linear(f32(x), f32(w)), True)
    ref = O.store(O.silu_and_mul(gu), True)
    assert_close(f32(outs[PAIR]), ref, f"pair SwiGLU {M}x{2 * I_}x{K}")


def test_pair_schedule_through_a_decoder_layer():
    """The qkv epilogue (RoPE, q store, paged K/V scatter) and the other three
    projections of a prefill layer on SM pairs, against the oracle layer; the
    caches and outputs equal those of single-SM tiles bit for bit."""
    spec = dataclasses.replace(I.SPECS["tiny"], groups=(("prefill", 2, 150, 0, 0), ("prefill", 1, 70, 30, 30)))
    bl = I.make_batch(spec, 3, DEV)
    w = I.make_layer_weights(spec, 3, 0, DEV)
    x, r = I.make_activations(spec, bl.num_tokens, 3, DEV)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), DEV)
    kc0, vc0 = I.make_kv_cache(spec, bl.num_blocks, 3, 0, DEV)
    results = {}
    for schedule in (PAIR, SINGLE):
        lb.set_gemm_schedule(schedule)
        kc, vc = kc0.clone(), vc0.clone()
        hid = x.clone()
        res = torch.empty_like(x)
        lb.layer_forward(cfg, w, batch, hid, r, res, kc, vc, ws)
        torch.cuda.synchronize()
        assert lb.get_device_error()[0] == lb.LLAMA_OK
        results[schedule] = (hid, res, kc, vc)
    for a, b, name in zip(results[PAIR], results[SINGLE], ("hidden", "residual", "k cache", "v cache")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name}: SM pairs differ from single SMs"
    hid, res, kc, vc = results[PAIR]
    kref, vref = bits(kc0), bits(vc0)
    out, res_ref = O.decoder_layer(oracle_shape(spec), oracle_weights(w), oracle_batch(bl), f32(x),
                                   None if r is None else f32(r), kref, vref)
    assert_close(f32(hid), out, "pair layer hidden")
    assert_close(f32(res), res_ref, "pair layer residual")
    assert_close(O.bf16_bits_to_float(bits(kc)), O.bf16_bits_to_float(kref), "pair layer k cache")
    assert_close(O.bf16_bits_to_float(bits(vc)), O.bf16_bits_to_float(vref), "pair layer v cache")


def test_schedule_override_rejects_unknown_values():
    with pytest.raises(lb.LlamaError):
        lb.set_gemm_schedule(4)
    with pytest.raises(lb.LlamaError):
        lb.set_gemm_schedule(-2)


def test_gate_up_timer_counts_the_layer_launches():
    """llama_gate_up_timer_*: one timed launch per layer of each stack call,
    with a positive duration; none once stopped."""
    spec = dataclasses.replace(I.SPECS["tiny"], num_layers=3, vocab=512, residual_none=True,
                               groups=(("decode", 2, 1, 10, 40), ("prefill", 1, 30, 0, 0)))
    bl = I.make_batch(spec, 2, DEV)
    layers = [I.make_layer_weights(spec, 2, l, DEV) for l in range(spec.num_layers)]
    caches = [I.make_kv_cache(spec, bl.num_blocks, 2, l, DEV) for l in range(spec.num_layers)]
    emb, ids, lm, fn = I.make_stack_extras(spec, bl.num_tokens, 2, DEV)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    T, B = bl.num_tokens, bl.num_seqs
    ws = lb.alloc_workspace(lb.workspace_size(cfg, T, B, batch.max_seq_len, spec.vocab), DEV)
    hidden = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device=DEV)
    residual = torch.empty_like(hidden)
    tokens = torch.empty(B, dtype=torch.int32, device=DEV)

    def call():
        lb.stack_forward(cfg, layers, fn, lm, batch, hidden, residual, [c[0] for c in caches],
                         [c[1] for c in caches], tokens, ws, embed=emb, input_ids=ids)

    call()
    lb.gate_up_timer_start(100)
    for _ in range(2):
        call()
    ms, n = lb.gate_up_timer_stop()
    assert n == 2 * spec.num_layers and ms > 0
    call()  # not timed
    lb.gate_up_timer_start(1)  # the cap: further launches go untimed
    call()
    ms1, n1 = lb.gate_up_timer_stop()
    assert n1 == 1 and ms1 > 0
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK


@pytest.mark.parametrize("M,I_,K", [
    (64, 14336, 256),   # the 8B decode gate_up's tile grid: 150 narrow tiles in one wave
    (128, 28672, 128),  # the 70B decode gate_up's: 299 narrow tiles in two waves
    (37, 10000, 192),   # ragged M and a last tile with 16 of its 96 columns valid
])
def test_narrow_swiglu_tiles_for_one_row_block(M, I_, K):
    """SwiGLU at decode-sized M with more than sms / 2 wide tiles runs on
    192-column tiles (96 gate + 96 up rows of B); compared with the oracle
    and with 256-column tiles (forced single-SM schedule)."""
    x = I.normal_bf16((M, K), 1.0, 0.0, 51 + M, DEV)
    w = I.normal_bf16((2 * I_, K), 0.02, 0.0, 52 + K, DEV)
    outs = {}
    for schedule in (-1, SINGLE):
        lb.set_gemm_schedule(schedule)
        a = torch.full((M, I_), float("nan"), dtype=torch.bfloat16, device=DEV)
        lb.gate_up_silu(x, w, a, _ws())
        torch.cuda.synchronize()
        assert lb.get_device_error()[0] == lb.LLAMA_OK
        outs[schedule] = a
    gu = O.store(O.linear(f32(x), f32(w)), True)
    ref = O.store(O.silu_and_mul(gu), True)
    assert_close(f32(outs[-1]), ref, f"narrow SwiGLU {M}x{2 * I_}x{K}")
    assert_close(f32(outs[SINGLE]), ref, f"wide SwiGLU {M}x{2 * I_}x{K}")
    print(f"narrow vs wide tiles bit-identical: {torch.equal(outs[-1], outs[SINGLE])}")
