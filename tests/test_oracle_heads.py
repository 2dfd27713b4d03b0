"""Pins of the self-draft heads in the oracle (oracle/heads.py).

"Speculative Decoding 101", Floor 6 and "Speculative decoding internals",
三條主流變體 (MTP): extra prediction heads on the target draft the next
positions and the target verifies them by the unchanged rule.  Pins:

* Closed form: two heads on a 2-wide input, each logit worked out by hand
  from silu(x) = x / (1 + e^-x) (values of the logistic function at 1 and 2).
* Zero heads are the target's own LM head: every row equals the target's
  logits for the pending token (the position the heads read), from the
  forward pass pinned in test_oracle_model.py -- a head reading any other
  position, or a dropped or doubled norm, fails this.
* The bf16 dataflow with its rounding replaced by the identity is the
  definition.
* Exactness, exhaustively: on a 1-layer model, the distribution of the
  emitted tokens over every draft and accept / resample branch (drafts drawn
  independently from the head rows) equals the target's own autoregressive
  distribution from torch.softmax.
* Exactness of spec_step as wired (the draft of position i from head row i,
  the streams of its uniforms): the first emitted token over many seeds
  follows the target's next-token distribution (chi-square), and drawing
  each draft from the next head's row instead breaks it.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import accept as acc
from oracle import generate as gen
from oracle import heads as hd
from oracle import model
from test_oracle_accept import _reps

SHAPE = workloads.ModelShape("headtiny", 1, 16, 2, 1, 8, 32, 3, 10000.0, dtype="f32")


def _tiny(seed=5, std=0.5, k=2, head_std=0.6):
    w = workloads.make_weights(SHAPE, seed=seed, std=std)
    g = torch.Generator().manual_seed(seed + 100)
    heads = torch.randn(k, SHAPE.d_model, SHAPE.d_model, generator=g, dtype=torch.float64) * head_std
    return gen.Model(SHAPE, w), heads


def test_heads_closed_form():
    # u = (1, -1) (a = u, s = 1).  Head 1 = I: W u = (1, -1), silu -> (0.7310585786300049,
    # -0.2689414213699951) (logistic(1) = 0.7310585786300049), z = (1.7310585786300049,
    # -1.2689414213699951).  Head 2 = [[0, 2], [0, 0]]: W u = (-2, 0), silu(-2) = -2 / (1 + e^2)
    # = -0.2384058440442351, z = (0.7615941559557649, -1).  LM head rows (1, 0), (0, 1), (1, 1).
    lm = torch.tensor([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]], dtype=torch.float64)
    heads = torch.tensor([[[1.0, 0.0], [0.0, 1.0]], [[0.0, 2.0], [0.0, 0.0]]], dtype=torch.float64)
    want = np.array([[1.7310585786300049, -1.2689414213699951, 0.4621171572600098],
                     [0.7615941559557649, -1.0, -0.2384058440442351]])
    a = torch.tensor([[1.0, -1.0]], dtype=torch.float64)
    got = hd.heads_from_input(a, 1.0, heads, lm).numpy()
    assert np.allclose(got, want, atol=1e-15, rtol=0)
    # the same input as a = 2u scaled by s = 1/2 (the bf16 dataflow's split)
    got2 = hd.heads_from_input(2 * a, 0.5, heads, lm).numpy()
    assert np.allclose(got2, want, atol=1e-15, rtol=0)


@pytest.mark.parametrize("shape", [SHAPE, workloads.small_shape(n_layers=1, vocab=64, dtype="f32")])
def test_zero_heads_are_the_target_head(shape):
    w = workloads.make_weights(shape, seed=3, std=0.3)
    T = gen.Model(shape, w)
    zero = torch.zeros(3, shape.d_model, shape.d_model, dtype=torch.float64)
    ctx = workloads.make_prompt(shape.vocab, 9, seed=4)[0].tolist()
    rows = hd.head_logits(T, zero, ctx)
    base = T.logits(ctx[:-1], last=1)[0]       # the pending token's distribution
    assert np.allclose(rows, base[None, :], atol=1e-12, rtol=0)
    wrong = T.logits(ctx, last=1)[0]            # one position later
    assert np.abs(rows[0] - wrong).max() > 1e-3


def test_identity_rounding_is_the_definition():
    T, heads = _tiny()
    ctx = [0, 2, 1, 1, 2]
    want = hd.head_logits(T, heads, ctx)
    a, s = hd.head_input(gen.Model(SHAPE, T.weights, act="bf16"), ctx)   # bf16 split, rounded
    ident = lambda t: t
    h = model.hidden(SHAPE, T.weights, ctx[:-1], ident)[-1:]
    a, s = model.final_input(SHAPE, T.weights, h, ident)
    got = hd.heads_from_input(a, s, heads, T.weights["lm_head"], ident).numpy()
    assert np.allclose(got, want, atol=1e-12, rtol=0)


def _heads_step_outcomes(T, heads, ctx, k, temp, memo):
    """{emitted tuple: probability} of one heads-drafted step, all branches."""
    q_logits = hd.head_logits(T, heads, ctx)[:k]
    q = acc.softmax_t(q_logits, temp)
    V = SHAPE.vocab
    out = {}
    for flat in range(V ** k):
        drafts = [(flat // V ** i) % V for i in range(k)]
        w = float(np.prod([q[i][drafts[i]] for i in range(k)]))
        if w == 0:
            continue
        key = tuple(ctx + drafts)
        if key not in memo:
            memo[key] = T.logits(ctx + drafts, last=k + 1)
        p_logits = memo[key]
        p = acc.softmax_t(p_logits, temp)

        def walk(j, r_vec, u_vec, wgt):
            if j == k:
                for u_b, w_b in _reps(p[k]):
                    em, _, _ = acc.accept_step(p_logits, q_logits, drafts, temp, r_vec, u_vec, u_b)
                    out[tuple(em)] = out.get(tuple(em), 0.0) + wgt * w_b
                return
            a = acc.accept_prob(p[j], q[j], drafts[j])
            if a > 0:
                walk(j + 1, r_vec[:j] + [a / 2] + r_vec[j + 1:], u_vec, wgt * a)
            if a < 1:
                for u_r, w_u in _reps(acc.residual(p[j], q[j])):
                    r2 = r_vec[:j] + [(1 + a) / 2] + r_vec[j + 1:]
                    u2 = u_vec[:j] + [u_r] + u_vec[j + 1:]
                    em, _, _ = acc.accept_step(p_logits, q_logits, drafts, temp, r2, u2, 0.5)
                    out[tuple(em)] = out.get(tuple(em), 0.0) + wgt * (1 - a) * w_u

        walk(0, [0.5] * k, [0.5] * k, w)
    return out


def _heads_dist(T, heads, ctx, need, k, temp, memo):
    res = {}
    for em, pr in _heads_step_outcomes(T, heads, list(ctx), k, temp, memo).items():
        if len(em) >= need:
            res[em[:need]] = res.get(em[:need], 0.0) + pr
        else:
            for tail, pt in _heads_dist(T, heads, list(ctx) + list(em), need - len(em), k, temp, memo).items():
                res[em + tail] = res.get(em + tail, 0.0) + pr * pt
    return res


def _target_dist(T, ctx, need, temp):
    res = {(): 1.0}
    for _ in range(need):
        nxt = {}
        for seq, pr in res.items():
            z = torch.tensor(T.logits(list(ctx) + list(seq), last=1)[0], dtype=torch.float64)
            p = torch.softmax(z / temp, 0)
            for y in range(SHAPE.vocab):
                nxt[seq + (y,)] = nxt.get(seq + (y,), 0.0) + pr * float(p[y])
        res = nxt
    return res


@pytest.mark.parametrize("k,need,temp", [(1, 2, 1.0), (2, 2, 1.0), (2, 3, 0.7)])
def test_heads_enumeration_exactness(k, need, temp):
    T, heads = _tiny(k=k)
    ctx = [2, 0, 1]
    spec = _heads_dist(T, heads, ctx, need, k, temp, {})
    target = _target_dist(T, ctx, need, temp)
    assert sum(spec.values()) == pytest.approx(1.0, abs=1e-12)
    err = max(abs(spec.get(s, 0.0) - target.get(s, 0.0)) for s in set(spec) | set(target))
    assert err < 1e-12, err
    # the heads' proposal really differs from the target (the check is not vacuous)
    q = acc.softmax_t(hd.head_logits(T, heads, ctx)[:k], temp)
    p1 = acc.softmax_t(T.logits(ctx, last=1)[0], temp)
    assert np.abs(q[0] - p1).max() > 0.1


def _first_token_counts(T, heads, ctx, k, n):
    """Counts of the first emitted token of heads.spec_step over steps 0..n-1
    (every step on the same context: independent uniforms per step)."""
    memo_q, memo_p = {}, {}
    real_q, real_p = hd.head_logits, T.logits

    def q_cached(t, h, c):
        key = tuple(c)
        if key not in memo_q:
            memo_q[key] = real_q(t, h, c)
        return memo_q[key]

    def p_cached(toks, last):
        key = (tuple(toks), last)
        if key not in memo_p:
            memo_p[key] = real_p(toks, last)
        return memo_p[key]

    counts = np.zeros(SHAPE.vocab)
    hd.head_logits, T.logits = q_cached, p_cached
    try:
        for s in range(n):
            res = hd.spec_step(T, heads, ctx, k, 1.0, seed=77, step=s)
            counts[res.emitted[0]] += 1
    finally:
        hd.head_logits = real_q
        del T.logits
    return counts


def _chi2(counts, p):
    e = counts.sum() * p
    return float(((counts - e) ** 2 / e).sum())


def test_spec_step_first_token_follows_target():
    T, heads = _tiny(seed=34, std=0.2, k=2, head_std=1.0)
    ctx = [1, 2, 0, 2]
    p1 = acc.softmax_t(T.logits(ctx, last=1)[0], 1.0)
    q = acc.softmax_t(hd.head_logits(T, heads, ctx)[:2], 1.0)
    assert np.abs(q[0] - q[1]).max() > 0.3 and np.abs(q[0] - p1).max() > 0.2
    n = 6000
    chi = _chi2(_first_token_counts(T, heads, ctx, 2, n), p1)
    assert chi < 13.8, chi   # 2 degrees of freedom: P(chi2 > 13.8) = 0.001

    # planted mistake: each draft drawn from the next head's row (the ratio
    # still uses its own row) -- no longer the target's distribution
    real = gen.draft_token
    rows = {}
    real_q = hd.head_logits

    def stash(t, h, c):
        rows["q"] = real_q(t, h, c)
        return rows["q"]

    def shifted(q_row, temperature, seed, step, i, row=0, tie_eps=acc.TIE_EPS):
        return real(rows["q"][i % 2], temperature, seed, step, i, row, tie_eps)

    hd.head_logits, gen.draft_token = stash, shifted
    try:
        counts = np.zeros(SHAPE.vocab)
        for s in range(1500):
            counts[hd.spec_step(T, heads, ctx, 2, 1.0, seed=77, step=s).emitted[0]] += 1
    finally:
        hd.head_logits, gen.draft_token = real_q, real
    chi_bad = _chi2(counts, p1)
    print(f"chi2 {chi:.2f} (as wired), {chi_bad:.1f} (planted)")
    assert chi_bad > 30.0
