"""One speculative step, the generation loop and plain decoding, in fp64.

Test infrastructure: see the package docstring.

Step layout ("Speculative decoding internals", 演算法核心, Steps 1-4; "Speculative
Decoding 101", Floors 4-5 and the Boss Level replay):

* The committed sequence ``seq`` ends with the pending token t (position L);
  the target has not yet scored position L.
* Draft loop, i = 1..K: draft logits at the last position of seq + d_<i,
  optionally mixed with the target's previous-step logits row i-1 at weight
  lambda, then d_i ~ softmax(. / T) (argmax when T == 0).
* Verify: target logits at positions L..L+K of seq + d_1..d_K (K+1 rows).
* Accept (see ``accept.accept_step``); the emitted tokens are appended to
  seq, the last of them becomes the new pending token; everything after the
  first rejection is discarded (the cache is simply rebuilt from seq here).
* The target's K+1 logit rows of this step are the "previous-step logits"
  of the next.  Before the first step they are the target logits at prompt
  positions L-1-K .. L-1: the last K+1 positions scored by a prefill of
  everything before the pending token.
* ``generate(n)`` steps until at least n tokens are emitted and truncates to n.

Random draws follow the layout in ``philox`` (step s counts speculative steps
from 0; autoregressive decoding counts its own steps from 0 on stream 4).
"""
from dataclasses import dataclass, field

import numpy as np

from . import accept as acc
from . import model
from .philox import (STREAM_ACCEPT, STREAM_AR, STREAM_BONUS, STREAM_DRAFT,
                     STREAM_RESIDUAL, uniform)


@dataclass
class Model:
    shape: object
    weights: dict
    act: str = "f64"     # "bf16": a bf16 model's dataflow (see oracle.model)

    def logits(self, tokens, last):
        return model.forward(self.shape, self.weights, tokens, last=last, act=self.act).numpy()


@dataclass
class StepResult:
    emitted: list
    n_accepted: int
    flags: int
    drafts: list = field(default_factory=list)
    q_logits: np.ndarray = None      # [K, V] (after mixing)
    p_logits: np.ndarray = None      # [K+1, V]


def step_uniforms(seed, step, k, row=0):
    """(r[K], u_res[K], u_bonus) of speculative step ``step``."""
    i = np.arange(1, k + 1)
    r = uniform(seed, step, i, STREAM_ACCEPT, row)
    u_res = uniform(seed, step, i, STREAM_RESIDUAL, row)
    u_bonus = uniform(seed, step, k + 1, STREAM_BONUS, row)
    return np.atleast_1d(r), np.atleast_1d(u_res), u_bonus


def draft_token(q_logits_row, temperature, seed, step, i, row=0, tie_eps=acc.TIE_EPS):
    """d_i from a draft logit row, with the step's stream-0 uniform."""
    return acc.draft_sample(q_logits_row, temperature,
                            uniform(seed, step, i, STREAM_DRAFT, row), tie_eps)


def verify(p_logits, q_logits, drafts, temperature, seed, step, row=0, tie_eps=acc.TIE_EPS):
    """Acceptance of one step on given logits (target [K+1, V], draft [K, V])."""
    k = len(drafts)
    r, u_res, u_bonus = step_uniforms(seed, step, k, row)
    return acc.accept_step(p_logits, q_logits, drafts, temperature, r, u_res, u_bonus, tie_eps)


def prefill_prev_logits(target: Model, prompt, k):
    """Target logits at prompt positions L-1-K .. L-1 ([K+1, V])."""
    seq = [int(t) for t in prompt]
    L = len(seq) - 1
    if L - 1 - k < 0:
        raise ValueError("prompt too short for the previous-logit rows")
    return target.logits(seq[:L], last=k + 1)


def spec_step(target: Model, draft: Model, seq, k, temperature, seed, step,
              prev=None, mix_lambda=0.0, row=0, tie_eps=acc.TIE_EPS):
    ctx = [int(t) for t in seq]
    drafts, q_rows, flags = [], [], 0
    for i in range(1, k + 1):
        lq = draft.logits(ctx + drafts, last=1)[0]
        if mix_lambda:
            lq = (1.0 - mix_lambda) * lq + mix_lambda * np.asarray(prev[i - 1], dtype=np.float64)
        d, f = draft_token(lq, temperature, seed, step, i, row, tie_eps)
        drafts.append(d)
        q_rows.append(lq)
        flags |= f
    p_rows = target.logits(ctx + drafts, last=k + 1)
    q_rows = np.stack(q_rows)
    emitted, n, f = verify(p_rows, q_rows, drafts, temperature, seed, step, row, tie_eps)
    return StepResult(emitted, n, flags | f, drafts, q_rows, p_rows)


def generate(target: Model, draft: Model, prompt, n_new, k, temperature, seed,
             mix_lambda=0.0, row=0):
    """Speculative generation of n_new tokens; returns (tokens, steps)."""
    seq = [int(t) for t in prompt]
    prev = prefill_prev_logits(target, seq, k) if mix_lambda else None
    out, steps = [], []
    s = 0
    while len(out) < n_new:
        res = spec_step(target, draft, seq, k, temperature, seed, s, prev, mix_lambda, row)
        seq += res.emitted
        out += res.emitted
        prev = res.p_logits
        steps.append(res)
        s += 1
    return out[:n_new], steps


def ar_token_flagged(logits_row, temperature, seed, step, row=0, tie_eps=acc.TIE_EPS):
    """Plain decoding's draw at step ``step``: argmax at T = 0, else the
    inverse CDF of softmax(logits / T) with the stream-4 uniform at position
    0.  Returns (token, flags): FLAG_NEAR_TIE when the top-2 logit gap is
    below tie_eps (T = 0), FLAG_NEAR_EDGE when the target lands within
    EDGE_EPS of a bin edge (T > 0)."""
    if temperature == 0:
        flags = acc.FLAG_NEAR_TIE if acc.top2_gap(logits_row) < tie_eps else 0
        return acc.argmax_lowest(logits_row), flags
    p = acc.softmax_t(logits_row, temperature)
    j, margin = acc.inverse_cdf(p, uniform(seed, step, 0, STREAM_AR, row))
    return j, (acc.FLAG_NEAR_EDGE if margin < acc.EDGE_EPS else 0)


def ar_token(logits_row, temperature, seed, step, row=0):
    return ar_token_flagged(logits_row, temperature, seed, step, row)[0]


def ar_generate(target: Model, prompt, n_new, temperature, seed, row=0):
    """Plain autoregressive decoding with the target alone."""
    seq = [int(t) for t in prompt]
    out = []
    for s in range(n_new):
        tok = ar_token(target.logits(seq, last=1)[0], temperature, seed, s, row)
        seq.append(tok)
        out.append(tok)
    return out
