"""llama_sample against the oracle's sampler on the same logits, parameters
and uniform draws.

The token is an integer that floating point decides (the GPU computes the
weights in fp32 and sums them in 40-bit fixed point, the oracle in fp64):
tokens must be equal wherever the oracle's margin exceeds 1e-6 (the draw is
that far, relative to the kept mass, from a CDF boundary, and the top-p target
that far from a cumulative boundary; the two sides' weights differ by ~1e-7
of the mass), and elsewhere the GPU's token must still be in the oracle's
kept set.  Greedy rows must match wherever the top-2 gap exceeds
1e-5.  Logprobs (raw log-softmax) within 2e-4.  Two calls are bit-identical."""

import numpy as np
import pytest
import torch

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lbuild.build()
    lb.lib()


def _kept_set(lrow, t, k, p):
    V = lrow.size
    w = np.exp((lrow - lrow.max()) / t)
    keep = np.ones(V, dtype=bool)
    if 0 < k < V:
        keep &= lrow >= np.sort(lrow)[V - k]
    if p < 1.0:
        vals = np.sort(w[keep])[::-1]
        idx = int(np.searchsorted(np.cumsum(vals), p * w[keep].sum(), side="left"))
        keep &= w >= vals[min(idx, vals.size - 1)] * (1 - 1e-6)
    return keep


def _run(logits, t, k, p, u):
    dev = lambda a, dt: torch.tensor(np.asarray(a), dtype=dt, device=DEV)  # noqa: E731
    L = dev(logits, torch.float32)
    rows = L.shape[0]
    tok = torch.empty(rows, dtype=torch.int32, device=DEV)
    lp = torch.empty(rows, dtype=torch.float32, device=DEV)
    args = (L, dev(t, torch.float32), dev(k, torch.int32), dev(p, torch.float32), dev(u, torch.float32))
    lb.sample(*args, tok, lp)
    tok2 = torch.empty_like(tok)
    lb.sample(*args, tok2, None)
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2), "two calls differ"
    return tok.cpu().numpy().astype(np.int64), lp.cpu().numpy()


def _check(logits, t, k, p, u):
    logits32 = np.asarray(logits, dtype=np.float32)
    tok, lp = _run(logits32, t, k, p, u)
    ref_tok, ref_lp, margin = O.sample(logits32.astype(np.float64), t, k, p, u)
    exact = 0
    for b in range(logits32.shape[0]):
        if t[b] < O.GREEDY_TEMPERATURE:
            srt = np.sort(logits32[b].astype(np.float64))
            if srt.size == 1 or srt[-1] - srt[-2] > 1e-5:
                assert tok[b] == ref_tok[b], f"greedy row {b}"
                exact += 1
        elif margin[b] > 1e-6:
            assert tok[b] == ref_tok[b], f"row {b}: {tok[b]} vs {ref_tok[b]} (margin {margin[b]:.2e})"
            exact += 1
        else:
            assert _kept_set(logits32[b].astype(np.float64), t[b], k[b], p[b])[tok[b]], f"row {b} outside the kept set"
    # raw log-softmax at the GPU's own token (where the tokens agree it is the oracle's logprob)
    ref = logits32.astype(np.float64)[np.arange(len(tok)), tok] - _log_z(logits32)
    assert np.max(np.abs(lp.astype(np.float64) - ref)) < 2e-4
    same = tok == ref_tok
    assert np.max(np.abs(lp[same].astype(np.float64) - ref_lp[same]), initial=0.0) < 2e-4
    return exact


def _log_z(logits32):
    x = logits32.astype(np.float64)
    m = x.max(axis=1)
    return m + np.log(np.exp(x - m[:, None]).sum(axis=1))


def test_sampler_full_vocabulary():
    # the stack's head: 34 rows of vocab 128256, every mode
    rng = np.random.default_rng(0)
    B, V = 34, 128256
    logits = rng.normal(size=(B, V)) * 2.5
    t = np.array([0.0, 1e-6] + list(rng.uniform(0.4, 1.6, size=B - 2)))
    k = rng.choice([0, 1, 5, 50, 1000, V, V + 7, -3], size=B)
    p = rng.choice([1.0, 0.95, 0.9, 0.5, 0.1, 0.0, 1.3], size=B)
    u = rng.random(B)
    exact = _check(logits, t, k, p, u)
    assert exact >= B - 3


def test_sampler_full_vocabulary_with_ties_at_the_k_boundary():
    # integer logits over the full vocabulary: at k = 1000 more than 1024 keys
    # tie at or above the k-th value (the general path), at k = 50 they do not
    # (the candidate path); one row per cluster size as well
    rng = np.random.default_rng(5)
    B, V = 12, 128256
    logits = np.round(rng.normal(size=(B, V)) * 2)
    t = np.full(B, 0.9)
    k = np.array([1000, 50] * (B // 2))
    p = rng.choice([1.0, 0.9, 0.5], size=B)
    u = rng.random(B)
    _check(logits, t, k, p, u)
    _check(logits[:1], t[:1], k[:1], p[:1], u[:1])
    _check(logits[1:2], t[1:2], k[1:2], p[1:2], u[1:2])


@pytest.mark.parametrize("V", [1, 7, 37, 1000])
def test_sampler_small_and_ragged_vocabularies_with_ties(V):
    rng = np.random.default_rng(V)
    B = 64
    logits = np.round(rng.normal(size=(B, V)) * 2)  # integer logits: many ties
    t = rng.choice([0.0, 0.5, 1.0, 2.0], size=B)
    k = rng.integers(-1, V + 2, size=B)
    p = rng.choice([1.0, 0.9, 0.6, 0.3, 0.0], size=B)
    u = rng.random(B)
    _check(logits, t, k, p, u)


def test_sampler_frequencies_follow_the_distribution():
    # one row repeated under evenly spaced draws: the GPU's token frequencies are
    # the renormalised probabilities of the kept set, to 1/N
    V, N = 50, 4096
    rng = np.random.default_rng(9)
    row = rng.normal(size=V)
    logits = np.repeat(row[None], N, axis=0)
    u = (np.arange(N) + 0.5) / N
    tok, _ = _run(logits.astype(np.float32), np.full(N, 0.8), np.full(N, 20), np.full(N, 0.9), u)
    keep = _kept_set(row, 0.8, 20, 0.9)
    w = np.where(keep, np.exp((row - row.max()) / 0.8), 0)
    assert np.max(np.abs(np.bincount(tok, minlength=V) / N - w / w.sum())) < 2.5 / N
    # no truncation (top-k off, top-p 1): the whole softmax at temperature 0.8
    tok, _ = _run(logits.astype(np.float32), np.full(N, 0.8), np.zeros(N), np.ones(N), u)
    w = np.exp((row - row.max()) / 0.8)
    assert np.max(np.abs(np.bincount(tok, minlength=V) / N - w / w.sum())) < 2.5 / N


def test_sampler_no_truncation_full_vocabulary_frequencies():
    # one 128256-wide row (a cluster of CTAs) under evenly spaced draws, no
    # truncation: the cumulative frequencies follow the softmax's CDF
    V, N = 128256, 64
    rng = np.random.default_rng(10)
    row = rng.normal(size=V) * 3
    logits = np.repeat(row[None].astype(np.float32), N, axis=0)
    u = (np.arange(N) + 0.5) / N
    tok, _ = _run(logits, np.ones(N), np.zeros(N), np.ones(N), u)
    x = row.astype(np.float32).astype(np.float64)
    cdf = np.cumsum(np.exp(x - x.max()))
    cdf /= cdf[-1]
    # token n is the first where the CDF exceeds u_n; a draw within rounding
    # (fp32 weights, 40-bit fixed point) of a step may take the neighbouring token
    want = np.searchsorted(cdf, u, side="right")
    near = np.minimum(np.abs(cdf[want] - u), np.abs(cdf[np.maximum(want - 1, 0)] - u)) < 1e-5
    assert np.all((tok == want) | near), np.nonzero((tok != want) & ~near)
