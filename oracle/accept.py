"""Acceptance, residual resampling and bonus draw, in fp64 (host side).

Test infrastructure: see the package docstring.

Sources (restated, not copied):

* "Speculative decoding internals" (tarrragon LLM notes), section
  "演算法核心：sampling 階段的接受邏輯": Step 1 (the drafter proposes d_1..d_K
  and keeps D(d_i)), Step 2 (one target pass gives T_1..T_{K+1}), Step 3
  (left to right: accept d_i when r < min(1, T_i(d_i)/D(d_i)), else draw a
  replacement from normalize((T_i - D)+) and stop), Step 4 (bonus draw from
  T_{K+1} when all K are accepted).
* "Speculative Decoding 101" (gu-log, English), Floor 5: the same rule with
  the worked example p = (.5, .3, .2), q = (.8, .1, .1); Floor 4: the greedy
  rule (accept on match, emit the target's token at the first mismatch and
  discard everything after it, bonus token when all match).

Readings where the pages leave a step open:

* r in [0, 1) and the comparison is strict, so P(accept) = min(1, p/q).
* q(d) == 0 cannot happen when d ~ q; if it does, the ratio is +inf (accept).
* Residual mass 0 after a rejection (only through rounding): draw from p
  instead and raise FLAG_RESID_ZERO.
* Inverse CDF over unnormalised weights w: target t = u * sum(w); pick the
  smallest j whose running sum exceeds t, scanning token ids upward; if
  rounding leaves t at or above the final sum, take the largest j with w_j > 0.
* Argmax ties go to the lowest token id.
* The temperature T scales both target and draft logits; T == 0 is greedy.
"""
import numpy as np

FLAG_RESID_ZERO = 1 << 0     # rejection with zero residual mass (fallback to p)
FLAG_NEAR_RATIO = 1 << 1     # |r - min(1, ratio)| < RATIO_EPS
FLAG_NEAR_EDGE = 1 << 2      # an inverse-CDF target within EDGE_EPS of a bin edge
FLAG_NEAR_TIE = 1 << 3       # greedy: top-2 logit gap below TIE_EPS

RATIO_EPS = 1e-5
EDGE_EPS = 1e-6
TIE_EPS = 4e-2


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def softmax_t(logits, temperature):
    """softmax(logits / T) along the last axis, in fp64 (T > 0)."""
    z = _f64(logits) / float(temperature)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def argmax_lowest(logits):
    """Index of the largest logit, lowest index on ties."""
    row = _f64(logits)
    return int(np.flatnonzero(row == row.max())[0])


def top2_gap(logits):
    row = np.sort(_f64(logits))
    return float(row[-1] - row[-2]) if row.size > 1 else np.inf


def inverse_cdf(weights, u):
    """Inverse-CDF draw from unnormalised non-negative weights.

    Returns (index, edge_margin) where edge_margin is the distance of the
    target u * Z to the nearest edge of the chosen bin, relative to Z.
    """
    w = _f64(weights)
    c = np.cumsum(w)
    z = c[-1]
    t = float(u) * z
    above = np.flatnonzero(c > t)
    if above.size:
        j = int(above[0])
    else:
        j = int(np.flatnonzero(w > 0)[-1])
    lo = c[j - 1] if j > 0 else 0.0
    margin = min(t - lo, c[j] - t) / z if z > 0 else 0.0
    return j, float(margin)


def accept_prob(p, q, d):
    """min(1, p(d) / q(d)) with q(d) == 0 read as an infinite ratio."""
    pd, qd = float(p[d]), float(q[d])
    if qd <= 0.0:
        return 1.0
    return min(1.0, pd / qd)


def residual(p, q):
    """Unnormalised residual weights max(0, p - q) (the "difference wheel")."""
    return np.maximum(_f64(p) - _f64(q), 0.0)


def draft_sample(q_logits, temperature, u, tie_eps=TIE_EPS):
    """Draw d ~ softmax(q_logits / T) by inverse CDF; argmax when T == 0.

    Returns (token, flags).  ``tie_eps``: greedy near-tie window (twice the
    logit tolerance of the precision being compared).
    """
    if temperature == 0:
        flags = FLAG_NEAR_TIE if top2_gap(q_logits) < tie_eps else 0
        return argmax_lowest(q_logits), flags
    z = _f64(q_logits) / float(temperature)
    w = np.exp(z - z.max())
    j, margin = inverse_cdf(w, u)
    return j, (FLAG_NEAR_EDGE if margin < EDGE_EPS else 0)


def accept_step(p_logits, q_logits, drafts, temperature, r, u_res, u_bonus, tie_eps=TIE_EPS):
    """One verification: returns (emitted tokens, n_accepted, flags).

    p_logits: [K+1, V] target logits at the K+1 verified positions.
    q_logits: [K, V] draft logits (after any mixing) that proposed d_1..d_K.
    drafts:   [K] draft tokens.
    r, u_res: [K] uniforms of the ratio test and of the residual draws.
    u_bonus:  uniform of the bonus draw.
    """
    p_logits = _f64(p_logits)
    q_logits = _f64(q_logits)
    k = len(drafts)
    emitted = []
    flags = 0
    if temperature == 0:
        for i in range(k):
            t_i = argmax_lowest(p_logits[i])
            if top2_gap(p_logits[i]) < tie_eps:
                flags |= FLAG_NEAR_TIE
            if int(drafts[i]) == t_i:
                emitted.append(t_i)
                continue
            emitted.append(t_i)           # first mismatch: the target's own token
            return emitted, i, flags
        if top2_gap(p_logits[k]) < tie_eps:
            flags |= FLAG_NEAR_TIE
        emitted.append(argmax_lowest(p_logits[k]))   # bonus
        return emitted, k, flags

    p = softmax_t(p_logits, temperature)
    q = softmax_t(q_logits, temperature)
    for i in range(k):
        d = int(drafts[i])
        a = accept_prob(p[i], q[i], d)
        if abs(float(r[i]) - a) < RATIO_EPS:
            flags |= FLAG_NEAR_RATIO
        if float(r[i]) < a:
            emitted.append(d)
            continue
        w = residual(p[i], q[i])
        if w.sum() <= 0.0:
            flags |= FLAG_RESID_ZERO
            w = p[i]
        j, margin = inverse_cdf(w, u_res[i])
        if margin < EDGE_EPS:
            flags |= FLAG_NEAR_EDGE
        emitted.append(j)
        return emitted, i, flags
    j, margin = inverse_cdf(p[k], u_bonus)
    if margin < EDGE_EPS:
        flags |= FLAG_NEAR_EDGE
    emitted.append(j)
    return emitted, k, flags


def expected_tokens_per_step(alpha, k):
    """(1 - alpha^(k+1)) / (1 - alpha): mean tokens per target pass for i.i.d.
    acceptance alpha ("Speculative Decoding 101", Floor 6)."""
    if alpha == 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)
