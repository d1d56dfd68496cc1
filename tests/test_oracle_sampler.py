"""Pins of the oracle's sampler (oracle.llama_oracle.sample) against what the
mathematics fixes: the greedy and k = 1 limits are the argmax; over a grid of
N evenly spaced draws the inverse CDF picks every kept token with exactly its
renormalised probability (to 1/N); temperature rescales the logits
(closed form); hand-worked top-k / top-p sets, ties included; the logprob is
scipy's log_softmax at the token."""

import numpy as np
import pytest
from scipy.special import log_softmax, softmax

from oracle import llama_oracle as O


def _draw_frequencies(logits, t, k, p, n=8000):
    u = (np.arange(n) + 0.5) / n
    rows = np.repeat(np.asarray(logits, dtype=np.float64)[None], n, axis=0)
    tok, _, _ = O.sample(rows, np.full(n, t), np.full(n, k), np.full(n, p), u)
    return np.bincount(tok, minlength=len(logits)) / n


def test_greedy_rows_take_the_argmax():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(6, 50))
    for t in (0.0, 1e-6, 9.9e-6):
        tok, lp, margin = O.sample(x, np.full(6, t), np.zeros(6), np.ones(6), rng.random(6))
        assert np.array_equal(tok, np.argmax(x, axis=1))
        assert np.all(np.isinf(margin))


def test_top_k_one_is_the_argmax_for_any_draw():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(8, 40))
    tok, _, _ = O.sample(x, np.full(8, 0.7), np.ones(8), np.ones(8), rng.random(8))
    assert np.array_equal(tok, np.argmax(x, axis=1))


def test_inverse_cdf_reproduces_the_softmax():
    rng = np.random.default_rng(2)
    x = rng.normal(size=12) * 2
    f = _draw_frequencies(x, 1.0, 0, 1.0)
    assert np.max(np.abs(f - softmax(x))) < 2e-4


def test_temperature_is_a_rescale_of_the_logits():
    rng = np.random.default_rng(3)
    x = rng.normal(size=10) * 3
    for t in (0.5, 2.0):
        f = _draw_frequencies(x, t, 0, 1.0)
        assert np.max(np.abs(f - softmax(x / t))) < 2e-4


def test_top_k_keeps_ties_at_the_boundary():
    x = np.array([3.0, 1.0, 3.0, 0.0, -1.0])
    f = _draw_frequencies(x, 1.0, 1, 1.0)  # the two maxima tie: both stay
    assert abs(f[0] - 0.5) < 1e-4 and abs(f[2] - 0.5) < 1e-4 and f[[1, 3, 4]].sum() == 0
    f = _draw_frequencies(x, 1.0, 3, 1.0)  # k-th largest is 1.0: tokens 0, 1, 2 stay
    ref = softmax(x[[0, 1, 2]])
    assert np.max(np.abs(f[[0, 1, 2]] - ref)) < 2e-4 and f[[3, 4]].sum() == 0


def test_top_p_hand_worked_sets():
    probs = np.array([0.05, 0.5, 0.15, 0.3])
    x = np.log(probs)
    f = _draw_frequencies(x, 1.0, 0, 0.79)  # 0.5 + 0.3 passes 0.79 (0.5 alone does not): tokens 1 and 3
    assert abs(f[1] - 0.5 / 0.8) < 2e-4 and abs(f[3] - 0.3 / 0.8) < 2e-4 and f[[0, 2]].sum() == 0
    f = _draw_frequencies(x, 1.0, 0, 0.81)  # 0.8 falls short: needs the 0.15 as well
    assert abs(f[2] - 0.15 / 0.95) < 2e-4 and f[0] == 0
    f = _draw_frequencies(x, 1.0, 0, 0.0)  # p -> 0 keeps only the most probable token
    assert f[1] == 1.0
    # top-p measures mass inside the top-k set: k = 2 keeps 0.5 and 0.3, and
    # p = 0.6 of their 0.8 needs both (0.5 < 0.48 is false: 0.5 >= 0.48)
    f = _draw_frequencies(x, 1.0, 2, 0.6)
    assert f[1] == 1.0
    f = _draw_frequencies(x, 1.0, 2, 0.7)  # 0.7 * 0.8 = 0.56 > 0.5: both
    assert abs(f[1] - 0.5 / 0.8) < 2e-4 and abs(f[3] - 0.3 / 0.8) < 2e-4


def test_top_p_keeps_ties_at_the_threshold():
    x = np.log(np.array([0.4, 0.2, 0.2, 0.2]))
    f = _draw_frequencies(x, 1.0, 0, 0.5)  # 0.4 + one 0.2 reaches 0.5; the tie keeps all three 0.2
    assert np.max(np.abs(f - np.array([0.4, 0.2, 0.2, 0.2]))) < 2e-4


def test_disabled_limits_and_logprob():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(5, 30))
    u = rng.random(5)
    a, lpa, _ = O.sample(x, np.full(5, 0.9), np.zeros(5), np.ones(5), u)
    b, lpb, _ = O.sample(x, np.full(5, 0.9), np.full(5, 30), np.full(5, 1.5), u)
    assert np.array_equal(a, b)
    ref = log_softmax(x, axis=1)[np.arange(5), a]
    assert np.max(np.abs(lpa - ref)) < 1e-12  # raw logprob: the temperature does not enter


@pytest.mark.parametrize("seed", range(3))
def test_token_is_always_kept(seed):
    rng = np.random.default_rng(10 + seed)
    x = rng.normal(size=(40, 64))
    t = rng.uniform(0.3, 2.0, size=40)
    k = rng.integers(0, 70, size=40)
    p = rng.uniform(0.05, 1.2, size=40)
    tok, _, margin = O.sample(x, t, k, p, rng.random(40))
    for b in range(40):
        if 0 < k[b] < 64:
            assert x[b, tok[b]] >= np.sort(x[b])[64 - k[b]]
    assert np.all(margin >= 0)


# ----------------------------------------------------------- planted mistakes
# Each mutant is the sampler with one plausible mistake; at least one pin above
# must fail on it.

def _mutant(kind):
    def sample(logits, temperature, top_k, top_p, uniform, dtype=np.float64):
        logits = np.asarray(logits, dtype=dtype)
        B, V = logits.shape
        tokens = np.empty(B, dtype=np.int64)
        logprobs = np.empty(B, dtype=dtype)
        margins = np.zeros(B, dtype=dtype)
        for b in range(B):
            lrow = logits[b]
            t = float(temperature[b])
            lmax = lrow.max()
            if t < O.GREEDY_TEMPERATURE:
                tok = int(np.argmax(lrow))
            else:
                w = np.exp((lrow - lmax) / (1.0 if kind == "no_temperature" else t))
                keep = np.ones(V, dtype=bool)
                k = int(top_k[b])
                if 0 < k < V:
                    if kind == "top_k_drops_ties":
                        keep[:] = False
                        keep[np.argsort(-lrow, kind="stable")[:k]] = True
                    else:
                        keep &= lrow >= np.sort(lrow)[V - k]
                p = float(top_p[b])
                if p < 1.0:
                    base = np.ones(V, dtype=bool) if kind == "top_p_over_all_tokens" else keep
                    mass = np.sum(w[base])
                    vals = np.sort(w[keep])[::-1]
                    idx = int(np.searchsorted(np.cumsum(vals), p * mass, side="left"))
                    tau = vals[min(idx, vals.size - 1)]
                    keep &= (w > tau) if kind == "top_p_drops_ties" else (w >= tau)
                c = np.cumsum(np.where(keep, w, 0.0))
                side = "left" if kind == "cdf_side" else "right"
                tok = min(int(np.searchsorted(c, float(uniform[b]) * c[-1], side=side)), V - 1)
            z = lrow / t if (kind == "tempered_logprob" and t >= O.GREEDY_TEMPERATURE) else lrow
            tokens[b] = tok
            logprobs[b] = log_softmax(z)[tok]
        return tokens, logprobs, margins
    return sample


PINS = [test_greedy_rows_take_the_argmax, test_top_k_one_is_the_argmax_for_any_draw,
        test_inverse_cdf_reproduces_the_softmax, test_temperature_is_a_rescale_of_the_logits,
        test_top_k_keeps_ties_at_the_boundary, test_top_p_hand_worked_sets, test_top_p_keeps_ties_at_the_threshold,
        test_disabled_limits_and_logprob]


@pytest.mark.parametrize("kind", ["no_temperature", "top_k_drops_ties", "top_p_over_all_tokens", "top_p_drops_ties",
                                  "tempered_logprob", "cdf_side"])
def test_planted_sampler_mistake_is_caught(monkeypatch, kind):
    monkeypatch.setattr(O, "sample", _mutant(kind))
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught the mutant {kind}"
