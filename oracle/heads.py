"""Self-draft heads on the target (extra prediction heads, "MTP"), plainly.

Test infrastructure: see the package docstring.

"Speculative Decoding 101", Floor 6: later variants need no second model --
extra prediction heads on the big model guess the next few positions, and
the big model verifies the guesses by the same rule.  "Speculative decoding
internals", section 三條主流變體 (MTP): the target carries K extra heads at its
output end, head i predicting position N + i.  The pages fix no head
architecture; the readings used here:

* Input.  With the committed context x_0 .. x_L (x_L the pending token, not
  yet scored), the target has scored positions 0 .. L-1; the heads read its
  final hidden state at position L-1 through the LM head's input
  u = RMSNorm_final(h_{L-1}) (where the target's own LM head predicts x_L).
* Head i (1..K) predicts position L + i -- the position of draft d_i in the
  verify pass [x_L, d_1 .. d_K]:  z_i = u + silu(W_i u) with one d x d matrix
  W_i per head, and logits_i = W_head z_i through the target's own LM head.
* Drafts.  q_i = softmax(logits_i / T); d_i is drawn from q_i with the
  stream-0 uniform of position i, exactly as a draft model's d_i (argmax at
  T = 0).  The heads see only the context, so every q_i is fixed before any
  draft: the acceptance rule ("Speculative decoding internals", 演算法核心
  Steps 3-4) holds for any proposal fixed before the target's rows are read,
  and the output stays the target's distribution.
* bf16 dataflow (act "bf16", see oracle.model): the head GEMMs read
  a = bf16(h * g) and scale their sums by s = 1/rms(h) (u = a * s), and z_i is
  rounded to bf16 where it is stored as the LM head's input.

Random heads have no trained acceptance; only the structure and the cost of
drafting from the target's own hidden state are exercised.
"""
import numpy as np
import torch

from . import generate as gen
from . import model


def head_input(target: gen.Model, ctx):
    """(a, s) of the LM-head input at the last scored position of ctx
    (ctx ends with the pending token): u = a * s, shape [1, d]."""
    rnd = model.ACT_ROUNDING[target.act]
    toks = [int(t) for t in ctx[:-1]]
    h = model.hidden(target.shape, target.weights, toks, rnd)[-1:]
    return model.final_input(target.shape, target.weights, h, rnd)


def heads_from_input(a, s, heads, lm_head, rnd=None):
    """Logit rows [K, V] of heads [K][d][d] (any float dtype) on the LM-head
    input (a, s) (u = a * s), with the LM head lm_head [V][d]."""
    u = a * s
    w_head = model._w(lm_head)
    rows = []
    for i in range(heads.shape[0]):
        y = model.silu((a @ model._w(heads[i]).T) * s)
        z = u + y
        if rnd is not None:
            z = rnd(z)
        rows.append((z @ w_head.T)[0])
    return torch.stack(rows)


def head_logits(target: gen.Model, heads, ctx):
    """q logit rows [K, V] (numpy fp64) of the heads after context ctx."""
    rnd = model.ACT_ROUNDING[target.act]
    a, s = head_input(target, ctx)
    return heads_from_input(a, s, heads, target.weights["lm_head"], rnd).numpy()


def spec_step(target: gen.Model, heads, seq, k, temperature, seed, step, row=0,
              tie_eps=gen.acc.TIE_EPS):
    """One speculative step drafted by the heads on the committed sequence
    seq; returns a generate.StepResult."""
    ctx = [int(t) for t in seq]
    q_rows = head_logits(target, heads, ctx)[:k]
    drafts, flags = [], 0
    for i in range(1, k + 1):
        d, f = gen.draft_token(q_rows[i - 1], temperature, seed, step, i, row, tie_eps)
        drafts.append(d)
        flags |= f
    p_rows = target.logits(ctx + drafts, last=k + 1)
    emitted, n, f = gen.verify(p_rows, q_rows, drafts, temperature, seed, step, row, tie_eps)
    return gen.StepResult(emitted, n, flags | f, drafts, np.asarray(q_rows), p_rows)


def generate(target: gen.Model, heads, prompt, n_new, k, temperature, seed, row=0):
    """Speculative generation of n_new tokens drafted by the heads."""
    seq = [int(t) for t in prompt]
    out, steps, s = [], [], 0
    while len(out) < n_new:
        res = spec_step(target, heads, seq, k, temperature, seed, s, row)
        seq += res.emitted
        out += res.emitted
        steps.append(res)
        s += 1
    return out[:n_new], steps
