"""Prompt-lookup (n-gram) drafting and its speculative step, plainly.

Test infrastructure: see the package docstring.

"Speculative Decoding 101", Floor 6 (The Days It's All for Nothing): n-gram
approaches such as prompt lookup draft without a model -- they search the
preceding text for a chunk that is likely to repeat and use what followed it
as the draft, and the verification follows the same rules as with a draft
model (the Boss Level's closing names the variant that drafts from the prompt
itself).  The pages fix no further detail; the readings used here:

* Match: the earlier position j (0 <= j < L, L = index of the pending token
  t) whose tokens ending at j agree with the context's last tokens ending at
  L for the most steps, m(j) = max{m <= n_max : ctx[j-i] == ctx[L-i] for all
  i < m}; the longest m wins, ties go to the largest (most recent) j; m = 0
  everywhere means no match.
* Drafts: what followed the match, d_i = ext[j + i] for i = 1..K, where ext is
  the context followed by the drafts themselves (a continuation that runs
  into the pending token keeps copying what it has drafted).  No match: K
  copies of the pending token.
* The drafter is deterministic, so its distribution q_i is one-hot at d_i
  (logit 0 at d_i, -inf elsewhere, for any temperature).  The acceptance rule
  is unchanged ("Speculative decoding internals", 演算法核心 Steps 3-4): accept
  d_i with probability min(1, p_i(d_i) / 1) = p_i(d_i); on rejection draw from
  normalize((p_i - q_i)+), i.e. p_i without d_i; greedy: accept iff d_i is
  the target's argmax.
"""
import numpy as np

from . import generate as gen


def best_match(ctx, n_max):
    """(j, m): the most recent longest match of the suffix of ctx (the last
    element is the pending token), m = 0 when none."""
    L = len(ctx) - 1
    best_j, best_m = -1, 0
    for j in range(L - 1, -1, -1):
        m = 0
        while m < n_max and j - m >= 0 and ctx[j - m] == ctx[L - m]:
            m += 1
        if m > best_m:   # scanning from the end: the first j of a length is the most recent
            best_j, best_m = j, m
    return best_j, best_m


def lookup_drafts(ctx, k, n_max):
    """The K drafts of prompt lookup for context ctx (ending with the pending token)."""
    ctx = [int(t) for t in ctx]
    j, m = best_match(ctx, n_max)
    if m == 0:
        return [ctx[-1]] * k
    ext = list(ctx)
    for i in range(1, k + 1):
        ext.append(ext[j + i])
    return ext[len(ctx):]


def onehot_logits(drafts, vocab):
    """q logit rows of a deterministic drafter: 0 at d_i, -inf elsewhere."""
    q = np.full((len(drafts), vocab), -np.inf)
    for i, d in enumerate(drafts):
        q[i, int(d)] = 0.0
    return q


def spec_step(target, seq, k, n_max, temperature, seed, step, row=0, tie_eps=gen.acc.TIE_EPS):
    """One prompt-lookup speculative step on the committed sequence seq."""
    ctx = [int(t) for t in seq]
    drafts = lookup_drafts(ctx, k, n_max)
    p = target.logits(ctx + drafts, last=k + 1)
    q = onehot_logits(drafts, target.shape.vocab)
    emitted, n, flags = gen.verify(p, q, drafts, temperature, seed, step, row, tie_eps)
    return drafts, p, q, emitted, n, flags
