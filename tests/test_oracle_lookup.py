"""Pins of the prompt-lookup drafter in the oracle (oracle/lookup.py).

"Speculative Decoding 101", Floor 6: n-gram drafting searches the preceding
text for a chunk likely to repeat and drafts what followed it; verification
keeps the same rules.  Pins:

* Match and drafts on hand-worked contexts (the reading stated in
  oracle/lookup.py: longest suffix match up to n_max, most recent on ties,
  self-extending copy, pending token repeated without a match), each expected
  list worked out by hand in the comments.
* Exactness: with the deterministic drafter (q one-hot at each draft) the
  distribution of the emitted tokens, enumerated over every accept/resample
  branch, equals the target's own autoregressive distribution computed by
  torch.softmax -- the theorem the pages rest on, for this proposal.
* A planted mistake (keeping the draft in the residual) breaks that check.
"""
import numpy as np
import pytest
import torch

from oracle import accept as acc
from oracle import lookup as lk
from test_oracle_accept import TableModel, _reps, _target_dist


def test_match_and_drafts_hand_worked():
    # ctx = 5 6 7 8 5 6 (pending 6 at index 5).  j = 1: 6 = 6, 5 = 5, then the
    # context starts -> m = 2; j = 0, 2, 3, 4 mismatch at once.  Drafts follow
    # index 1: 7 8 5 6, then the copy reaches the first draft: 7.
    assert lk.best_match([5, 6, 7, 8, 5, 6], 3) == (1, 2)
    assert lk.lookup_drafts([5, 6, 7, 8, 5, 6], 5, 3) == [7, 8, 5, 6, 7]
    # ctx = 1 2 3 0 2 3 5 1 2 3: j = 2 matches 3 tokens (1 2 3), j = 5 only 2
    # (2 3, then 0 != 1): the longest wins -> drafts 0 2 3 5 1.
    ctx = [1, 2, 3, 0, 2, 3, 5, 1, 2, 3]
    assert lk.best_match(ctx, 3) == (2, 3)
    assert lk.lookup_drafts(ctx, 5, 3) == [0, 2, 3, 5, 1]
    # n_max = 2: j = 2 and j = 5 both reach 2, the most recent (5) wins ->
    # 5 1 2 3, then the first draft again: 5.
    assert lk.best_match(ctx, 2) == (5, 2)
    assert lk.lookup_drafts(ctx, 5, 2) == [5, 1, 2, 3, 5]
    # n_max = 1: the most recent earlier 3 is at index 5 -> 5 1 2 3 5.
    assert lk.best_match(ctx, 1) == (5, 1)
    # no earlier occurrence of the pending token: K copies of it
    assert lk.best_match([1, 2, 3, 4], 3) == (-1, 0)
    assert lk.lookup_drafts([1, 2, 3, 4], 4, 3) == [4, 4, 4, 4]
    # a run: 7 7 7 (pending 7): j = 1 matches 2 (7 7), j = 0 one -> drafts
    # copy index 2 onwards: 7, then the drafts themselves: 7 7.
    assert lk.lookup_drafts([7, 7, 7], 3, 3) == [7, 7, 7]


def test_onehot_logits():
    q = lk.onehot_logits([2, 0], 4)
    assert q.shape == (2, 4)
    for T in (0.5, 1.0, 2.0):
        p = acc.softmax_t(q, T)
        assert np.array_equal(p, np.array([[0, 0, 1, 0], [1, 0, 0, 0]], dtype=np.float64))
    # acceptance probability is p(d); the residual is p without d
    p = np.array([0.1, 0.2, 0.3, 0.4])
    qq = acc.softmax_t(q[0], 1.0)
    assert acc.accept_prob(p, qq, 2) == pytest.approx(0.3, abs=1e-15)
    assert np.allclose(acc.residual(p, qq), [0.1, 0.2, 0.0, 0.4], atol=1e-15)


def _lookup_step_outcomes(tm, ctx, k, n_max, temp):
    """{emitted tuple: probability} of one prompt-lookup step, all branches."""
    drafts = lk.lookup_drafts(ctx, k, n_max)
    p_logits = np.stack([tm.logits(ctx + drafts[:j]) for j in range(k + 1)])
    q_logits = lk.onehot_logits(drafts, tm.vocab)
    p = acc.softmax_t(p_logits, temp)
    q = acc.softmax_t(q_logits, temp)
    out = {}

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

    walk(0, [0.5] * k, [0.5] * k, 1.0)
    return out


def _lookup_dist(tm, ctx, need, k, n_max, temp, memo):
    key = (tuple(ctx), need)
    if key in memo:
        return memo[key]
    res = {}
    for em, pr in _lookup_step_outcomes(tm, list(ctx), k, n_max, temp).items():
        if len(em) >= need:
            res[em[:need]] = res.get(em[:need], 0.0) + pr
        else:
            for tail, pt in _lookup_dist(tm, list(ctx) + list(em), need - len(em), k, n_max, temp, memo).items():
                res[em + tail] = res.get(em + tail, 0.0) + pr * pt
    memo[key] = res
    return res


@pytest.mark.parametrize("vocab,k,n_max,need,ctx,temp", [
    (2, 2, 2, 3, [0, 1, 0], 1.0),
    (3, 3, 3, 3, [1, 2, 1, 2], 1.0),
    (4, 2, 1, 3, [3, 0, 3], 0.8),
    (3, 4, 2, 4, [0, 0, 1], 1.3),
])
def test_lookup_enumeration_exactness(vocab, k, n_max, need, ctx, temp):
    tm = TableModel(vocab, salt=23)
    spec = _lookup_dist(tm, ctx, need, k, n_max, temp, {})
    target = _target_dist(tm, ctx, need, temp)
    assert sum(spec.values()) == pytest.approx(1.0, abs=1e-12)
    keys = set(spec) | set(target)
    err = max(abs(spec.get(s, 0.0) - target.get(s, 0.0)) for s in keys)
    assert err < 1e-12, err


def test_lookup_enumeration_detects_planted_mistake():
    """Keeping the rejected draft in the residual (drawing from p instead of
    normalize((p - q)+)) must break exactness."""
    tm = TableModel(3, salt=29)
    good = acc.residual
    try:
        acc.residual = lambda p, q: np.asarray(p, dtype=np.float64)
        spec = _lookup_dist(tm, [1, 2, 1], 2, 2, 2, 1.0, {})
    finally:
        acc.residual = good
    target = _target_dist(tm, [1, 2, 1], 2, 1.0)
    err = max(abs(spec.get(s, 0.0) - target.get(s, 0.0)) for s in set(spec) | set(target))
    assert err > 1e-3
