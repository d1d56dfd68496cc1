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


class SubBatch:
    """A subset of the sequences of a batch, re-indexed with a compact cache:
    the oracle runs on it alone (sequences are independent, so the result is
    the same as on the full batch)."""

    def __init__(self, bl, seqs, kc_dev, vc_dev):
        qsl = bl.query_start_loc.cpu().numpy().astype(np.int64)
        bt = bl.block_table.cpu().numpy().astype(np.int64)
        self.seqs = list(seqs)
        self.rows = np.concatenate([np.arange(qsl[b], qsl[b + 1]) for b in self.seqs]).astype(np.int64)
        nblk = [(bl.ctx_lens[b] + bl.q_lens[b] + 15) // 16 for b in self.seqs]
        self.orig_blocks = np.concatenate([bt[b, :n] for b, n in zip(self.seqs, nblk)]).astype(np.int64)
        cbt = -np.ones((len(self.seqs), max(nblk)), np.int64)
        cur = 0
        for i, n in enumerate(nblk):
            cbt[i, :n] = np.arange(cur, cur + n)
            cur += n
        q_lens = [bl.q_lens[b] for b in self.seqs]
        cqsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
        pos = bl.positions.cpu().numpy().astype(np.int64)[self.rows]
        sl = bl.seq_lens.cpu().numpy().astype(np.int64)[self.seqs]
        self.batch = O.Batch(pos, cqsl, sl, cbt)
        idx = torch.as_tensor(self.orig_blocks, device=kc_dev.device)
        self.kc = bits(kc_dev.index_select(0, idx))
        self.vc = bits(vc_dev.index_select(0, idx))

    def gpu_written(self, cache_bits_after: np.ndarray) -> np.ndarray:
        """GPU cache rows [n_rows, nkv, d] at the slots of the subset's tokens."""
        out = []
        for i, p in zip(O.token_sequence(self.batch.query_start_loc), self.batch.positions):
            blk = self.orig_blocks[self.batch.block_table[i, p // 16]]
            out.append(cache_bits_after[blk, :, p % 16, :])
        return np.stack(out)

    def oracle_written(self, compact_bits: np.ndarray) -> np.ndarray:
        out = []
        for i, p in zip(O.token_sequence(self.batch.query_start_loc), self.batch.positions):
            out.append(compact_bits[self.batch.block_table[i, p // 16], :, p % 16, :])
        return np.stack(out)


def untouched_equal(after_bits: np.ndarray, before_bits: np.ndarray, written: np.ndarray) -> bool:
    keep = ~written
    return bool(np.array_equal(after_bits.transpose(0, 2, 1, 3)[keep], before_bits.transpose(0, 2, 1, 3)[keep]))
