"""Parity at the full sizes of the five workloads, in the launch configuration
the benchmark times (GPU).  The GPU runs the whole batch; the oracle runs on a
seeded subset of sequences (exact: sequences are independent) and, for the
70B prefill, on a seeded subset of rows after the cache update."""

import dataclasses

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from llama_decoder_layer_gb300 import inputs as I
from oracle import llama_oracle as O
from tests.helpers import (SubBatch, assert_close, bits, f32, oracle_batch, oracle_shape, oracle_weights,
                           rel_err, written_slot_mask)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


def _untouched_on_device(before: torch.Tensor, after: torch.Tensor, written: np.ndarray, name: str):
    keep = torch.as_tensor(~written, device=before.device)  # [num_blocks, 16]
    b = before.permute(0, 2, 1, 3)[keep]
    a = after.permute(0, 2, 1, 3)[keep]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{name}: slots outside the batch changed"


def _layer_case(name, sample_seqs, rows_in_seq=None, seed=0, dtype=np.float64, folded=False):
    spec = I.SPECS[name]
    bl = I.make_batch(spec, seed, DEV)
    w = I.make_layer_weights(spec, seed, 0, DEV)
    # folded norms: the GPU runs gamma folded into w_qkv / w_gate_up; the
    # oracle runs the unfolded layer (the same mathematics, rounded elsewhere)
    w_gpu = lb.folded_layer_weights(w) if folded else w
    x, r = I.make_activations(spec, bl.num_tokens, seed, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, DEV)
    kc0, vc0 = kc.clone(), vc.clone()
    sub = SubBatch(bl, sample_seqs, kc, vc)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), DEV)
    hid = x.clone()
    res = torch.empty_like(x)
    lb.layer_forward(cfg, w_gpu, batch, hid, r, res, kc, vc, ws)
    torch.cuda.synchronize()
    st, where = lb.get_device_error()
    assert st == lb.LLAMA_OK, f"device error {st} at {where}"
    # indexing: every slot outside the batch is untouched, bit for bit
    wm = written_slot_mask(bl, bl.num_blocks)
    _untouched_on_device(kc0, kc, wm, "k_cache")
    _untouched_on_device(vc0, vc, wm, "v_cache")
    del kc0, vc0
    rows_sel = None if rows_in_seq is None else list(rows_in_seq)
    xs = f32(x)[sub.rows]
    rs = None if r is None else f32(r)[sub.rows]
    kref, vref = sub.kc.copy(), sub.vc.copy()
    out, res_ref = O.decoder_layer(oracle_shape(spec), oracle_weights(w), sub.batch, xs, rs, kref, vref,
                                   rows=rows_sel, dtype=dtype)
    sel = np.arange(len(sub.rows)) if rows_sel is None else np.asarray(rows_sel)
    e1 = assert_close(f32(hid)[sub.rows][sel], out[sel], f"{name} hidden_states")
    e2 = assert_close(f32(res)[sub.rows][sel], res_ref[sel], f"{name} residual")
    e3 = assert_close(O.bf16_bits_to_float(sub.gpu_written(bits(kc))),
                      O.bf16_bits_to_float(sub.oracle_written(kref)), f"{name} k written")
    e4 = assert_close(O.bf16_bits_to_float(sub.gpu_written(bits(vc))),
                      O.bf16_bits_to_float(sub.oracle_written(vref)), f"{name} v written")
    print(f"{name}{' (folded norms)' if folded else ''}: rel err hidden {e1:.2e} residual {e2:.2e} k {e3:.2e} "
          f"v {e4:.2e}")


def test_tiny_full_config():
    _layer_case("tiny", sample_seqs=range(2))


def test_decode_8b_all_sequences():
    _layer_case("decode_8b", sample_seqs=range(64))


def test_decode_70b_seeded_subset():
    rng = np.random.default_rng(2024)
    _layer_case("decode_70b", sample_seqs=sorted(rng.choice(128, size=8, replace=False).tolist()))


def test_prefill_70b_one_sequence_seeded_rows():
    rng = np.random.default_rng(7)
    seq = int(rng.integers(0, 8))
    rows = sorted(set(rng.choice(4096, size=254, replace=False).tolist()) | {0, 4095})
    _layer_case("prefill_70b", sample_seqs=[seq], rows_in_seq=rows)


def test_folded_norms_tiny_and_decode_70b():
    """Folded norms (ln1/ln2 None, gamma in w_qkv / w_gate_up) against the
    unfolded oracle layer, on the tiny config and a seeded 70B decode subset."""
    _layer_case("tiny", sample_seqs=range(2), folded=True)
    rng = np.random.default_rng(2025)
    _layer_case("decode_70b", sample_seqs=sorted(rng.choice(128, size=4, replace=False).tolist()), folded=True)


def test_folded_norms_prefill_70b_seeded_rows():
    rng = np.random.default_rng(8)
    seq = int(rng.integers(0, 8))
    rows = sorted(set(rng.choice(4096, size=126, replace=False).tolist()) | {0, 4095})
    _layer_case("prefill_70b", sample_seqs=[seq], rows_in_seq=rows, folded=True)


def test_fold_norm_weights_is_the_rounded_product():
    """llama_fold_norm_weights: bf16(w * gamma) column-wise, bit for bit
    against the oracle's bf16 rounding of the product (ragged row count)."""
    g = I.normal_bf16((520,), 0.02, 1.0, 91, DEV)
    w = I.normal_bf16((37, 520), 0.02, 0.0, 92, DEV)
    got = lb.fold_norm_weights(g, w)
    torch.cuda.synchronize()
    want = O.round_to_bf16(f32(w).astype(np.float64) * f32(g).astype(np.float64)[None, :])
    # the product of two bf16 values is exact in fp64 and in fp32 (8-bit significands)
    assert np.array_equal(f32(got), want.astype(np.float32))


def test_stack_70b_subset_tokens_and_logits():
    """The 8-layer stack, pinned in four parts:
    (a) the stack call equals the composition of its layer calls, the final
        norm and lm_head, bit for bit (caches, logits, tokens);
    (b) every layer matches the oracle given that layer's inputs (teacher
        forcing), on 4 seeded decode sequences and one prefill chunk;
    (c) the head matches the oracle given the final hidden/residual rows of
        all 34 sequences: logits within tolerance, greedy tokens identical
        wherever the oracle's top-2 gap exceeds 0.05;
    (d) free running, the oracle's own 8-layer pass over the sampled
        sequences picks the GPU's greedy token wherever its top-2 gap
        exceeds 0.05.
    The free-running difference of hidden_states across the 8 layers is
    printed, not held to the 2e-2 bar: two oracles that differ only in fp32
    vs fp64 accumulation drift past that bar by depth 8
    (tests/test_oracle_depth_drift.py)."""
    spec = I.SPECS["stack_70b"]
    seed = 0
    bl = I.make_batch(spec, seed, DEV)
    NL = spec.num_layers
    layers = [I.make_layer_weights(spec, seed, l, DEV) for l in range(NL)]
    emb, ids, lm, fn = I.make_stack_extras(spec, bl.num_tokens, seed, DEV)
    caches = [I.make_kv_cache(spec, bl.num_blocks, seed, l, DEV) for l in range(NL)]
    caches2 = [(kc.clone(), vc.clone()) for kc, vc in caches]
    rng = np.random.default_rng(11)
    sample = sorted(rng.choice(32, size=4, replace=False).tolist()) + [32 + int(rng.integers(0, 2))]
    subs = [SubBatch(bl, sample, kc, vc) for kc, vc in caches]
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    T, B = bl.num_tokens, bl.num_seqs
    ws = lb.alloc_workspace(lb.workspace_size(cfg, T, B, batch.max_seq_len, spec.vocab), DEV)
    hid = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device=DEV)
    res = torch.empty_like(hid)
    tokens = torch.empty(B, dtype=torch.int32, device=DEV)
    logits = torch.empty((B, spec.vocab), dtype=torch.float32, device=DEV)
    lb.stack_forward(cfg, layers, fn, lm, batch, hid, res, [c[0] for c in caches], [c[1] for c in caches], tokens, ws,
                     embed=emb, input_ids=ids, out_logits=logits)
    torch.cuda.synchronize()
    st, where = lb.get_device_error()
    assert st == lb.LLAMA_OK, f"device error {st} at {where}"

    # (a) the same step as separate layer calls; keep every layer's inputs
    h2 = emb[ids.long()].contiguous()
    r2 = torch.empty_like(h2)
    layer_in = []
    for l in range(NL):
        layer_in.append((f32(h2)[subs[0].rows], None if l == 0 else f32(r2)[subs[0].rows]))
        lb.layer_forward(cfg, layers[l], batch, h2, None if l == 0 else r2, r2, caches2[l][0], caches2[l][1], ws)
    last = bl.query_start_loc[1:].long() - 1
    hf = torch.empty((B, spec.hidden), dtype=torch.bfloat16, device=DEV)
    lb.fused_add_rmsnorm(h2[last].contiguous(), r2[last].contiguous(), None, hf, fn, spec.rms_eps)
    logits2 = torch.empty_like(logits)
    lb.linear(hf, lm, logits2, lb.alloc_workspace(lb.linear_workspace_size(), DEV))
    torch.cuda.synchronize()
    assert torch.equal(hid, h2) and torch.equal(res, r2), "stack hidden/residual differ from the layer composition"
    for l in range(NL):
        assert torch.equal(caches[l][0].view(torch.int16), caches2[l][0].view(torch.int16)), f"layer {l} k cache"
        assert torch.equal(caches[l][1].view(torch.int16), caches2[l][1].view(torch.int16)), f"layer {l} v cache"
    assert torch.equal(logits, logits2), "stack logits differ from norm + lm_head of the composition"
    del caches2

    # (b) every layer against the oracle on the same inputs (fp32 oracle for this size)
    sh = oracle_shape(spec)
    x_free = f32(emb)[ids.cpu().numpy().astype(np.int64)[subs[0].rows]]
    r_free = None
    gpu_after = [(layer_in[l + 1] if l + 1 < NL else (f32(hid)[subs[0].rows], f32(res)[subs[0].rows]))
                 for l in range(NL)]
    for l in range(NL):
        ow = oracle_weights(layers[l])
        kref, vref = subs[l].kc.copy(), subs[l].vc.copy()
        xo, ro = O.decoder_layer(sh, ow, subs[l].batch, layer_in[l][0], layer_in[l][1], kref, vref,
                                 dtype=np.float32)
        eh = assert_close(gpu_after[l][0], xo, f"layer {l} hidden (same inputs)")
        er = assert_close(gpu_after[l][1], ro, f"layer {l} residual (same inputs)")
        ek = assert_close(O.bf16_bits_to_float(subs[l].gpu_written(bits(caches[l][0]))),
                          O.bf16_bits_to_float(subs[l].oracle_written(kref)), f"layer {l} k written")
        ev = assert_close(O.bf16_bits_to_float(subs[l].gpu_written(bits(caches[l][1]))),
                          O.bf16_bits_to_float(subs[l].oracle_written(vref)), f"layer {l} v written")
        kf, vf = subs[l].kc.copy(), subs[l].vc.copy()
        x_free, r_free = O.decoder_layer(sh, ow, subs[l].batch, x_free, r_free, kf, vf, dtype=np.float32)
        print(f"stack layer {l}: same-input rel err hidden {eh:.2e} residual {er:.2e} k {ek:.2e} v {ev:.2e}; "
              f"free-running hidden {rel_err(gpu_after[l][0], x_free):.2e}")

    # (c) the head on the same inputs, all sequences
    last_all = bl.query_start_loc[1:].long().cpu().numpy() - 1
    hf_ref, _ = O.fused_add_rms_norm(f32(hid)[last_all], f32(res)[last_all], f32(fn), sh.rms_eps, np.float32,
                                     bf16_tensors=True)
    lm_f = f32(lm)
    ref_logits = O.linear(hf_ref, lm_f, np.float32)
    ref_tok, gap = O.greedy_argmax(ref_logits)
    e = assert_close(f32(logits), ref_logits, "logits (all rows)")
    g_tok_all = tokens.cpu().numpy()
    decided = gap > 0.05
    assert np.array_equal(g_tok_all[decided], ref_tok[decided]), \
        f"greedy tokens differ: {g_tok_all} vs {ref_tok} gap {gap}"
    assert np.array_equal(g_tok_all, np.argmax(f32(logits), axis=-1))
    print(f"stack head: logits rel err {e:.2e} on {B} rows, tokens compared on {int(decided.sum())}/{B} rows")

    # (d) free running: the oracle's own pass through all 8 layers and the head
    lrows = O.last_token_rows(subs[0].batch.query_start_loc)
    hf_free, _ = O.fused_add_rms_norm(x_free[lrows], r_free[lrows], f32(fn), sh.rms_eps, np.float32,
                                      bf16_tensors=True)
    free_logits = O.linear(hf_free, lm_f, np.float32)
    free_tok, free_gap = O.greedy_argmax(free_logits)
    g_tok = g_tok_all[sample]
    free_decided = free_gap > 0.05
    print(f"stack free running: logits rel err {rel_err(f32(logits)[sample], free_logits):.2e}, gaps "
          f"{np.round(free_gap, 3).tolist()}, tokens gpu {g_tok.tolist()} oracle {free_tok.tolist()}")
    assert np.array_equal(g_tok[free_decided], free_tok[free_decided]), \
        f"free-running greedy tokens differ: {g_tok} vs {free_tok} gap {free_gap}"


def test_max_position_decode():
    """One decode token at position 131071 (max_position_embeddings - 1) over a
    131072-token context, tiny shape with llama3 RoPE."""
    spec = dataclasses.replace(I.SPECS["tiny"], rope_theta=500000.0, rope_scaling=I.LLAMA3_SCALING,
                               groups=(("decode", 1, 1, 131071, 131071), ("decode", 2, 1, 5, 70)))
    bl = I.make_batch(spec, 1, DEV)
    w = I.make_layer_weights(spec, 1, 0, DEV)
    x, r = I.make_activations(spec, bl.num_tokens, 1, DEV)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, 1, 0, DEV)
    kb0, vb0 = bits(kc), bits(vc)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), DEV)
    hid = x.clone()
    res = torch.empty_like(x)
    lb.layer_forward(cfg, w, batch, hid, r, res, kc, vc, ws)
    torch.cuda.synchronize()
    assert lb.get_device_error()[0] == lb.LLAMA_OK
    out, res_ref = O.decoder_layer(oracle_shape(spec), oracle_weights(w), oracle_batch(bl), f32(x),
                                   None if r is None else f32(r), kb0.copy(), vb0.copy())
    assert_close(f32(hid), out, "hidden at max position")
    assert_close(f32(res), res_ref, "residual at max position")


def test_empty_batch_is_a_no_op():
    spec = I.SPECS["tiny"]
    cfg = lb.LayerConfig.from_spec(spec)
    w = I.make_layer_weights(spec, 0, 0, DEV)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    batch = lb.Batch(e, torch.zeros(1, dtype=torch.int32, device=DEV), e,
                     torch.zeros((0, 1), dtype=torch.int32, device=DEV), 1, 1, 1)
    x = torch.empty((0, spec.hidden), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((1, spec.n_kv_heads, 16, spec.head_dim), dtype=torch.bfloat16, device=DEV)
    ws = lb.alloc_workspace(1024, DEV)
    lb.layer_forward(cfg, w, batch, x, None, x, kc, kc.clone(), ws)
    assert lb.get_device_error()[0] == lb.LLAMA_OK
