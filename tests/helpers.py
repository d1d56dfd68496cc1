"""Shared test utilities: tensor conversion, tolerance checks and runners
that feed the same seeded inputs to the CUDA library and to the oracle."""

from __future__ import annotations

import numpy as np
import torch

from oracle import llama_oracle as O

# spec bar: max|gpu - ref| <= 2e-2 * max|ref| per output tensor
TOL = 2e-2


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    return err / scale if scale > 0 else err


def assert_close(gpu, ref, name: str, tol: float = TOL) -> float:
    e = rel_err(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu, dtype=np.float64))), f"{name}: non-finite values"
    assert e <= tol, f"{name}: max|gpu-ref| / max|ref| = {e:.3e} > {tol}"
    return e


def oracle_shape(spec) -> O.LayerShape:
    return O.LayerShape(spec.hidden, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.intermediate, spec.rms_eps,
                        spec.rope_theta, spec.rope_scaling, spec.block_size)


def oracle_weights(w: dict) -> O.LayerWeights:
    return O.LayerWeights(f32(w["ln1"]), f32(w["w_qkv"]), f32(w["w_o"]), f32(w["ln2"]), f32(w["w_gate_up"]),
                          f32(w["w_down"]))


def oracle_batch(bl) -> O.Batch:
    return O.Batch(bl.positions.cpu().numpy().astype(np.int64), bl.query_start_loc.cpu().numpy().astype(np.int64),
                   bl.seq_lens.cpu().numpy().astype(np.int64), bl.block_table.cpu().numpy().astype(np.int64))


def written_slot_mask(bl, num_blocks: int, block_size: int = 16) -> np.ndarray:
    """[num_blocks, block_size] bool: the cache slots this batch writes
    (from the oracle's slot mapping)."""
    ob = oracle_batch(bl)
    slots = O.slot_mapping(ob.positions, ob.query_start_loc, ob.block_table, block_size)
    m = np.zeros((num_blocks, block_size), dtype=bool)
    for s in slots:
        if s >= 0:
            m[s // block_size, s % block_size] = True
    return m


def check_cache(gpu_bits: np.ndarray, ref_bits: np.ndarray, before_bits: np.ndarray, written: np.ndarray, name: str):
    """Slots the batch does not write must be bit-identical to their prior
    contents; written slots must match the oracle within tolerance."""
    untouched = ~written
    assert np.array_equal(gpu_bits[untouched[:, None, :].repeat(gpu_bits.shape[1], 1)],
                          before_bits[untouched[:, None, :].repeat(gpu_bits.shape[1], 1)]), \
        f"{name}: slots outside the batch changed"
    sel = written[:, None, :].repeat(gpu_bits.shape[1], 1)
    g = O.bf16_bits_to_float(gpu_bits[sel])
    r = O.bf16_bits_to_float(ref_bits[sel])
    return assert_close(g, r, f"{name} (written slots)")
