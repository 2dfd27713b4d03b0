"""Pins of the oracle's generation loop on the tiny speculative-generation
workload (2 layers, d=128, vocab 256, fp32; draft = layer 0 + noise).

* Greedy speculative output is identical to plain greedy autoregressive
  output ("Speculative Decoding 101", Floor 4 and Boss Level: every emitted
  word is one the oracle itself would have produced).
* Every step emits between 1 and K+1 tokens; drafts before the first
  rejection are emitted unchanged.
* A draft identical to the target accepts all K drafts every step.
* generate(n) returns exactly n tokens (overshoot truncated).
* The mixed draft's previous-step rows, worked by hand on table models:
  before the first step they are the target rows at positions L-1-K .. L-1
  (L = the pending token's position), and draft i mixes with row i-1.
* Plain decoding's draw: greedy by hand (lowest id on ties, the tie flag),
  and at T > 0 a chi-square test of 6000 draws against softmax(logits / T)
  that a draw at the wrong temperature fails; the top-2 gap by hand; the
  step's uniforms on their streams and positions.
"""
import numpy as np
import pytest

import workloads
from oracle import generate as gen


@pytest.fixture(scope="module")
def tiny():
    shape = workloads.TINY
    w = workloads.make_weights(shape, seed=0)
    dshape, dw = workloads.noisy_layer0_draft(shape, w, seed=1)
    prompt = workloads.make_prompt(shape.vocab, 16, seed=0)[0].tolist()
    return gen.Model(shape, w), gen.Model(dshape, dw), prompt


def test_greedy_spec_equals_greedy_ar(tiny):
    target, draft, prompt = tiny
    spec, steps = gen.generate(target, draft, prompt, 40, 4, 0.0, seed=0)
    ar = gen.ar_generate(target, prompt, 40, 0.0, seed=0)
    assert spec == ar
    assert all(1 <= len(s.emitted) <= 5 for s in steps)


@pytest.mark.parametrize("mix", [0.0, 0.5])
def test_sampled_generation_invariants(tiny, mix):
    target, draft, prompt = tiny
    out, steps = gen.generate(target, draft, prompt, 24, 4, 1.0, seed=0, mix_lambda=mix)
    assert len(out) == 24
    for s in steps:
        assert 1 <= len(s.emitted) <= 5
        assert s.emitted[:s.n_accepted] == s.drafts[:s.n_accepted]
        assert s.p_logits.shape == (5, 256) and s.q_logits.shape == (4, 256)


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_draft_equal_target_accepts_all(tiny, temp):
    target, _, prompt = tiny
    out, steps = gen.generate(target, target, prompt, 15, 4, temp, seed=3)
    assert all(s.n_accepted == 4 and len(s.emitted) == 5 for s in steps)


def test_sampled_first_token_uses_target_distribution(tiny):
    """With the same seed, step 0's emitted tokens do not depend on whether the
    draft is the target or the noisy draft when the first draft is rejected:
    the replacement comes from (p - q)+, which the draft changes -- so only
    check the weaker fact that both runs emit valid tokens and that the
    draft-equals-target run reproduces plain sampling of its drafts."""
    target, draft, prompt = tiny
    res = gen.spec_step(target, target, prompt, 4, 1.0, 0, 0)
    assert res.emitted[:4] == res.drafts
    assert np.allclose(res.q_logits, res.p_logits[:4], atol=1e-10)


class _Table:
    """Table model: the logit row for position j of `tokens` is
    [j, tokens[j], 0, ...] (target), or a fixed row (draft)."""

    def __init__(self, vocab, fixed=None):
        self.vocab, self.fixed = vocab, fixed

    def logits(self, tokens, last):
        n = len(tokens)
        rows = np.zeros((last, self.vocab))
        for r, j in enumerate(range(n - last, n)):
            if self.fixed is not None:
                rows[r] = self.fixed
            else:
                rows[r, 0], rows[r, 1] = j, tokens[j]
        return rows


def test_prefill_prev_rows_by_hand():
    """Prompt 10..19: the pending token 19 sits at position L = 9; with K = 3
    the previous-step rows are the target rows at positions 5, 6, 7, 8
    (tokens 15..18).  A one-position shift either way fails."""
    target = _Table(32)
    prev = gen.prefill_prev_logits(target, list(range(10, 20)), 3)
    assert prev.shape == (4, 32)
    assert prev[:, :2].tolist() == [[5, 15], [6, 16], [7, 17], [8, 18]]
    assert not prev[:, 2:].any()


def test_mixed_draft_rows_by_hand():
    """lambda = 0.5, K = 2, V = 4, draft row [2, 0, 0, 0] at every position,
    previous rows [[0,0,4,0], [0,0,0,8], [1,1,1,1]]: q_1 = [1,0,2,0] (row 0),
    q_2 = [1,0,0,4] (row 1), so the greedy drafts are 2 then 3.  Mixing with
    row i instead of row i-1 would propose 3 first."""
    draft = _Table(4, fixed=np.array([2.0, 0, 0, 0]))
    target = _Table(4, fixed=np.array([0.0, 0, 0, 1]))
    prev = np.array([[0.0, 0, 4, 0], [0, 0, 0, 8], [1, 1, 1, 1]])
    res = gen.spec_step(target, draft, [1, 2, 3], 2, 0.0, 0, 0, prev, 0.5)
    assert res.q_logits.tolist() == [[1, 0, 2, 0], [1, 0, 0, 4]]
    assert res.drafts == [2, 3]
    # the target's argmax is 3 everywhere: draft 2 is rejected and replaced by 3
    assert res.emitted == [3] and res.n_accepted == 0


def test_top2_gap_by_hand():
    from oracle import accept as acc
    assert acc.top2_gap([3.0, 1.0, 2.0]) == 1.0
    assert acc.top2_gap([2.0, 2.0, 0.0]) == 0.0          # a tie at the top
    assert acc.top2_gap([-1.0, -4.0]) == 3.0
    assert acc.top2_gap([5.0]) == np.inf                 # one token: no runner-up


def test_ar_greedy_draw_and_tie_flag():
    """Plain decoding at T = 0 is the argmax, lowest id on ties, flagged when
    the top-2 gap is under the tie window ([101] Floor 4's greedy rule)."""
    from oracle import accept as acc
    tok, fl = gen.ar_token_flagged([1.0, 5.0, 5.0, 2.0], 0.0, 0, 0)
    assert tok == 1 and fl & acc.FLAG_NEAR_TIE
    tok, fl = gen.ar_token_flagged([1.0, 5.0, 4.9], 0.0, 0, 0, tie_eps=0.2)
    assert tok == 1 and fl & acc.FLAG_NEAR_TIE
    tok, fl = gen.ar_token_flagged([1.0, 5.0, 4.9], 0.0, 0, 0, tie_eps=0.05)
    assert tok == 1 and fl == 0


def test_ar_sampled_draw_follows_softmax():
    """Plain decoding at T > 0 draws from softmax(logits / T): over 6000
    steps (each its own stream-4 uniform) the token counts pass a chi-square
    test against the closed-form probabilities, and a draw at the wrong
    temperature (a planted mistake, checked the same way) fails it."""
    from scipy.stats import chisquare
    logits = np.array([0.0, 1.0, -0.5, 2.0, 0.3])
    temp, n = 0.7, 6000
    e = np.exp((logits - logits.max()) / temp)
    probs = e / e.sum()
    counts = np.bincount([gen.ar_token(logits, temp, 11, s) for s in range(n)], minlength=logits.size)
    assert chisquare(counts, probs * n).pvalue > 1e-3
    wrong = np.bincount([gen.ar_token(logits, 1.0, 11, s) for s in range(n)], minlength=logits.size)
    assert chisquare(wrong, probs * n).pvalue < 1e-6


def test_step_uniforms_layout():
    """The uniforms of one speculative step follow reading 7's layout: the
    ratio tests r_i and the residual draws on streams 1 and 2 at positions
    1..K, the bonus draw on stream 3 at position K+1, sequence b in the row
    word -- so no two of them coincide and the rows are independent."""
    from oracle import philox
    k, seed, step = 4, 7, 3
    r, u_res, u_bonus = gen.step_uniforms(seed, step, k)
    for i in range(1, k + 1):
        assert r[i - 1] == philox.uniform(seed, step, i, 1)
        assert u_res[i - 1] == philox.uniform(seed, step, i, 2)
    assert u_bonus == philox.uniform(seed, step, k + 1, 3)
    allu = np.concatenate([r, u_res, [u_bonus]])
    assert len(set(allu.tolist())) == allu.size and ((allu >= 0) & (allu < 1)).all()
    r1, _, _ = gen.step_uniforms(seed, step, k, row=1)
    assert not np.array_equal(r, r1)
