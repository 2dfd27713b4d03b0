"""Pins of the oracle's acceptance rule against what the pages fix.

* Worked example and quiz of "Speculative Decoding 101" (gu-log, English),
  Floor 5 / 推測解碼入門 (gu-log, zh-tw), 第 5 層 (fixture worked_example.json).
* Exactness ("Speculative Decoding 101", Floor 5: the output distribution is
  the target's; "Speculative decoding internals", 演算法核心, 關鍵性質 1):
  exhaustive enumeration over every draft sequence and every accept/resample
  branch on tiny vocabularies, compared with the target's own autoregressive
  distribution computed by torch.softmax (a library routine, not the oracle).
* Greedy traces (fixture greedy_traces.json).
* Per-step bounds: at least 1 and at most K+1 tokens (Floor 4).
* A draft equal to the target accepts everything (ratio 1, r < 1).
* Mean tokens per step: the Floor 6 closed form and its printed values.

Every random draw in the enumeration goes through the oracle's own samplers;
the test only chooses representative uniforms (the midpoint of each bin) and
weights each branch by the bin's width.
"""
import json
import os
import zlib
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import accept as acc
from oracle import generate as gen


def _frac(s):
    return Fraction(s)


def _reps(weights):
    """(u, prob) for every non-empty inverse-CDF bin: bin midpoints."""
    w = np.asarray(weights, dtype=np.float64)
    c = np.cumsum(w)
    z = c[-1]
    out = []
    lo = 0.0
    for j in range(w.size):
        if w[j] > 0:
            out.append(((lo + c[j]) / (2 * z), w[j] / z))
        lo = c[j]
    return out


# ---------------------------------------------------------------- worked example
def test_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example.json")))
    p = np.array([float(_frac(x)) for x in g["p"]])
    q = np.array([float(_frac(x)) for x in g["q"]])
    for d, want in enumerate(g["accept_prob"]):
        assert acc.accept_prob(p, q, d) == pytest.approx(float(_frac(want)), abs=1e-15)
    res = acc.residual(p, q)
    assert np.allclose(res, [float(_frac(x)) for x in g["residual_unnormalized"]], atol=1e-15)
    assert np.allclose(res / res.sum(), [float(_frac(x)) for x in g["residual_normalized"]], atol=1e-15)
    # kept mass q(d) * min(1, p/q), total rejected mass == residual mass
    kept = q * np.array([acc.accept_prob(p, q, d) for d in range(3)])
    assert np.allclose(kept, [float(_frac(x)) for x in g["kept_mass"]], atol=1e-15)
    assert 1 - kept.sum() == pytest.approx(float(_frac(g["rejected_mass"])), abs=1e-15)
    assert res.sum() == pytest.approx(float(_frac(g["rejected_mass"])), abs=1e-15)

    # First emitted token through accept_step with K = 1, all branches.
    p_logits = np.log(np.stack([p, p]))
    q_logits = np.log(q)[None, :]
    dist = np.zeros(3)
    for u_d, w_d in _reps(acc.softmax_t(q_logits[0], 1.0)):
        d, _ = acc.draft_sample(q_logits[0], 1.0, u_d)
        a = acc.accept_prob(acc.softmax_t(p_logits[0], 1.0), acc.softmax_t(q_logits[0], 1.0), d)
        branches = [(a / 2, a)] + ([((1 + a) / 2, 1 - a)] if a < 1 else [])
        for r, w_r in branches:
            sub = _reps(acc.residual(acc.softmax_t(p_logits[0], 1.0), acc.softmax_t(q_logits[0], 1.0))) \
                if r >= a else [(0.5, 1.0)]
            for u_res, w_u in sub:
                em, _, _ = acc.accept_step(p_logits, q_logits, [d], 1.0, [r], [u_res], 0.5)
                dist[em[0]] += w_d * w_r * w_u
    assert np.allclose(dist, [float(_frac(x)) for x in g["final"]], atol=1e-14)

    quiz = g["quiz"]
    assert acc.accept_prob(p, q, g["tokens"].index(quiz["token"])) == float(_frac(quiz["accept_prob"]))


# ---------------------------------------------------------------- exactness
class TableModel:
    """Logits as a fixed pseudo-random function of the context tuple."""

    def __init__(self, vocab, salt, scale=1.5, zero_prob=0.0):
        self.vocab, self.salt, self.scale, self.zero_prob = vocab, salt, scale, zero_prob

    def logits(self, ctx):
        h = zlib.crc32(np.asarray([self.salt] + list(ctx), dtype=np.int64).tobytes())
        rng = np.random.default_rng(h)
        z = rng.normal(0.0, self.scale, self.vocab)
        if self.zero_prob:
            dead = rng.random(self.vocab) < self.zero_prob
            dead[rng.integers(self.vocab)] = False       # keep at least one token
            z[dead] = -np.inf
        return z


def _step_outcomes(tm, dm, ctx, k, temp):
    """{emitted tuple: probability} of one oracle step, all branches."""
    out = {}

    def rec(drafts, q_rows, weight):
        i = len(drafts)
        if i == k:
            p_logits = np.stack([tm.logits(ctx + drafts[:j]) for j in range(k + 1)])
            p = acc.softmax_t(p_logits, temp)
            q = acc.softmax_t(np.stack(q_rows), temp)

            def walk(j, r_vec, u_vec, wgt):
                if j == k:
                    for u_b, w_b in _reps(p[k]):
                        em, n, _ = acc.accept_step(p_logits, np.stack(q_rows), drafts, temp,
                                                   r_vec, u_vec, u_b)
                        out[tuple(em)] = out.get(tuple(em), 0.0) + wgt * w_b
                    return
                a = acc.accept_prob(p[j], q[j], drafts[j])
                walk(j + 1, r_vec[:j] + [a / 2] + r_vec[j + 1:], u_vec, wgt * a)
                if a < 1:
                    for u_r, w_u in _reps(acc.residual(p[j], q[j])):
                        r2 = r_vec[:j] + [(1 + a) / 2] + r_vec[j + 1:]
                        u2 = u_vec[:j] + [u_r] + u_vec[j + 1:]
                        em, n, _ = acc.accept_step(p_logits, np.stack(q_rows), drafts, temp, r2, u2, 0.5)
                        out[tuple(em)] = out.get(tuple(em), 0.0) + wgt * (1 - a) * w_u

            walk(0, [0.5] * k, [0.5] * k, weight)
            return
        lq = dm.logits(ctx + drafts)
        for u, w in _reps(acc.softmax_t(lq, temp)):
            d, _ = acc.draft_sample(lq, temp, u)
            rec(drafts + [d], q_rows + [lq], weight * w)

    rec([], [], 1.0)
    return out


def _spec_dist(tm, dm, ctx, need, k, temp, memo):
    key = (tuple(ctx), need)
    if key in memo:
        return memo[key]
    res = {}
    for em, pr in _step_outcomes(tm, dm, list(ctx), k, temp).items():
        if len(em) >= need:
            res[em[:need]] = res.get(em[:need], 0.0) + pr
        else:
            for tail, pt in _spec_dist(tm, dm, list(ctx) + list(em), need - len(em), k, temp, memo).items():
                key2 = em + tail
                res[key2] = res.get(key2, 0.0) + pr * pt
    memo[key] = res
    return res


def _target_dist(tm, ctx, need, temp):
    """Target's own autoregressive distribution of the next `need` tokens,
    from torch.softmax (library routine)."""
    res = {(): 1.0}
    for _ in range(need):
        nxt = {}
        for seq, pr in res.items():
            p = torch.softmax(torch.tensor(tm.logits(list(ctx) + list(seq)), dtype=torch.float64) / temp, 0)
            for y in range(tm.vocab):
                if p[y] > 0:
                    nxt[seq + (y,)] = nxt.get(seq + (y,), 0.0) + pr * float(p[y])
        res = nxt
    return res


@pytest.mark.parametrize("vocab,k,need,temp,zero", [
    (2, 1, 3, 1.0, 0.0),
    (3, 2, 3, 1.0, 0.0),
    (4, 3, 2, 1.0, 0.0),
    (3, 3, 4, 0.7, 0.0),
    (5, 2, 3, 1.3, 0.3),
    (8, 1, 2, 1.0, 0.25),
])
def test_enumeration_exactness(vocab, k, need, temp, zero):
    tm = TableModel(vocab, salt=11, zero_prob=zero)
    dm = TableModel(vocab, salt=97, scale=2.5, zero_prob=zero)
    ctx = [1 % vocab, 0]
    spec = _spec_dist(tm, dm, ctx, need, k, temp, {})
    target = _target_dist(tm, ctx, need, temp)
    assert sum(spec.values()) == pytest.approx(1.0, abs=1e-12)
    keys = set(spec) | set(target)
    err = max(abs(spec.get(s, 0.0) - target.get(s, 0.0)) for s in keys)
    assert err < 1e-12, err


def test_enumeration_detects_planted_mistake():
    """A plausible mistake planted in the oracle (residual (q - p)+ instead of
    (p - q)+) must break the exactness check, so the check has teeth."""
    tm, dm = TableModel(3, salt=5), TableModel(3, salt=6, scale=2.0)
    good = acc.residual
    try:
        acc.residual = lambda p, q: np.maximum(np.asarray(q) - np.asarray(p), 0.0)
        spec = _spec_dist(tm, dm, [0], 2, 2, 1.0, {})
    finally:
        acc.residual = good
    target = _target_dist(tm, [0], 2, 1.0)
    keys = set(spec) | set(target)
    assert max(abs(spec.get(s, 0.0) - target.get(s, 0.0)) for s in keys) > 1e-3


# ---------------------------------------------------------------- greedy traces
def test_greedy_traces(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "greedy_traces.json")))
    total_words = 0
    for tr in g["traces"]:
        words = sorted(set(tr["draft"]) | set(tr["target"]) | {"<unspecified>"})
        ids = {w: i for i, w in enumerate(words)}
        V, K = len(words), len(tr["draft"])
        p_logits = np.full((K + 1, V), -1.0)
        for j, w in enumerate(tr["target"]):
            p_logits[j, ids[w]] = 5.0
        q_logits = np.full((K, V), -1.0)
        drafts = [ids[w] for w in tr["draft"]]
        for j, d in enumerate(drafts):
            q_logits[j, d] = 5.0
        em, n, _ = acc.accept_step(p_logits, q_logits, drafts, 0, None, None, None)
        assert [words[t] for t in em] == tr["emitted"], tr["source"]
        assert n == len(tr["emitted"]) - 1
        if "English" in tr["source"]:
            total_words += len(em)
    assert total_words == g["boss_total"]["words"]


# ---------------------------------------------------------------- bounds / identity
@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_bounds_and_identity(temp):
    rng = np.random.default_rng(3)
    for s in range(300):
        k = int(rng.integers(1, 9))
        V = int(rng.integers(2, 50))
        p = rng.normal(0, 2, (k + 1, V))
        q = rng.normal(0, 2, (k, V))
        if temp == 0:
            drafts = [acc.argmax_lowest(q[i]) for i in range(k)]
        else:
            drafts = [gen.draft_token(q[i], temp, 0, s, i + 1)[0] for i in range(k)]
        em, n, _ = gen.verify(p, q, drafts, temp, 0, s)
        assert 1 <= len(em) <= k + 1 and len(em) == n + 1
        assert em[:n] == drafts[:n]
        # draft == target: everything accepted
        q_same = p[:k]
        d_same = [acc.argmax_lowest(q_same[i]) if temp == 0 else
                  gen.draft_token(q_same[i], temp, 0, s, i + 1)[0] for i in range(k)]
        em2, n2, _ = gen.verify(p, q_same, d_same, temp, 0, s)
        assert n2 == k and len(em2) == k + 1


def test_first_reject_yields_one_token():
    """推測解碼入門, 魔王關 quiz: a rejected first slip still yields exactly one token."""
    p = np.log(np.array([[0.0001, 0.9999], [0.5, 0.5], [0.5, 0.5]]))
    q = np.log(np.array([[0.9999, 0.0001], [0.5, 0.5]]))
    em, n, _ = acc.accept_step(p, q, [0, 0], 1.0, [0.9, 0.0], [0.3, 0.3], 0.3)
    assert n == 0 and em == [1]


# ---------------------------------------------------------------- E[tokens]
def test_expected_tokens_closed_form(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "expected_tokens.json")))
    for row in g["rows"]:
        a, k = row["alpha"], row["k"]
        assert a ** (k + 1) == pytest.approx(row["alpha_pow"], abs=5e-4)
        assert round(acc.expected_tokens_per_step(a, k), 2) == row["printed"]


@pytest.mark.parametrize("alpha,k", [(0.8, 4), (0.5, 4), (0.8, 8)])
def test_expected_tokens_enumeration_and_monte_carlo(alpha, k):
    # q is one-hot on token 0, so every draft is token 0 and its acceptance
    # probability is exactly p(0) = alpha, independently per position.
    p = np.log(np.tile([alpha, 1 - alpha], (k + 1, 1)))
    with np.errstate(divide="ignore"):
        q = np.log(np.tile([1.0, 0.0], (k, 1)))
    drafts = [0] * k
    # exact: enumerate the first-rejection position through accept_step
    mean = 0.0
    for stop in range(k + 1):
        r = [alpha / 2] * stop + [(1 + alpha) / 2] * (k - stop)
        em, n, _ = acc.accept_step(p, q, drafts, 1.0, r, [0.5] * k, 0.5)
        assert n == stop
        mean += len(em) * (alpha ** stop) * ((1 - alpha) if stop < k else 1.0)
    assert mean == pytest.approx(acc.expected_tokens_per_step(alpha, k), rel=1e-12)
    # Monte Carlo through the Philox draw layout
    n_steps = 20000
    counts = np.array([len(gen.verify(p, q, drafts, 1.0, 1, s)[0]) for s in range(n_steps)])
    sem = counts.std() / np.sqrt(n_steps)
    assert abs(counts.mean() - acc.expected_tokens_per_step(alpha, k)) < 4 * sem
