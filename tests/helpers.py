"""Shared helpers of the GPU tests (not collected as tests)."""
import numpy as np
import torch

import speculative_decoding_verification_step_gb300 as sv
from oracle import accept as acc
from oracle import generate as gen
from oracle import heads as hd

SKIP_FLAGS = acc.FLAG_NEAR_EDGE | acc.FLAG_NEAR_RATIO | acc.FLAG_NEAR_TIE | acc.FLAG_RESID_ZERO


def to_device(w, device="cuda"):
    out = {}
    for k, v in w.items():
        out[k] = [{kk: vv.to(device) for kk, vv in l.items()} for l in v] if k == "layers" else v.to(device)
    return out


def decoder(shape, w, dshape, dw, k, max_ctx, temperature=0.0, seed=0, mix=0.0, flags=0):
    sv.build()
    return sv.SpecDecoder(shape, w, dshape, dw, k, max_ctx, temperature=temperature, seed=seed,
                          mix_lambda=mix, flags=flags)


def logit_tol(shape):
    """Forward-pass tolerance on logits: 2e-2 absolute for bf16 models (fp32
    accumulation), 5e-5 for fp32 models."""
    return 2e-2 if shape.dtype == "bf16" else 5e-5


def tie_eps(shape):
    return 2 * logit_tol(shape)


def equal_mass_bins(p, nbins):
    """Assign tokens (sorted by probability, descending) to nbins bins of
    about equal target mass.  Returns bin id per token."""
    order = np.argsort(-p, kind="stable")
    cum = np.cumsum(p[order])
    ids = np.minimum((cum - p[order] / 2) * nbins, nbins - 1).astype(int)
    # a single heavy token can span several nominal bins: keep non-empty ones
    _, ids = np.unique(ids, return_inverse=True)
    out = np.empty_like(ids)
    out[order] = ids
    return out


def teacher_forced(dec, T, D, prompt, k, temp, n_new, tol, mix=0.0, seed=0, max_ctx=256, tie=None,
                   extra=None, alt=None, heads=None, prefilled=False):
    """Run speculative steps on the GPU decoder `dec` (already built, not yet
    prefilled) and check each one against the oracle models T (target) and D
    (draft), starting every oracle step from the GPU's committed context:

    * stage (i): the draft rows up to the first draft that differs from the
      oracle's own, and the K+1 target rows when every draft agrees, within
      `tol` of the oracle's forward;
    * drafts: each is the oracle's inverse-CDF draw (argmax at T = 0) on the
      GPU's own draft row with the step's Philox uniform -- exact except
      flagged near-edge / near-tie draws;
    * stage (ii): the oracle's acceptance on the GPU's logits and drafts gives
      the GPU's emitted tokens, exactly, except flagged draws;
    * the committed context grows by exactly the emitted tokens.

    alt = (T_alt, D_alt), if given: the same models in another precision of
    the oracle (its bf16 dataflow); each compared row set is then held to tol
    plus the largest difference between the two oracle precisions on those
    rows.  extra(step, ctx, p, q, drafts, ref), if given, runs further checks
    on each step's GPU logits.  heads, if given: the drafts come from these
    self-draft heads on T (oracle.heads; D and alt's draft are unused), and
    every head row is compared (they do not depend on the drafts).
    prefilled: dec already holds the committed context `prompt` (no prefill
    here).  Returns (tokens, steps, skipped, worst) with worst = the largest
    (error, allowed) seen."""
    tie = 2 * tol if tie is None else tie
    if not prefilled:
        dec.prefill(prompt)
    ctx = [int(t) for t in prompt]
    prev = gen.prefill_prev_logits(T, ctx, k) if mix else None
    out, step, skipped, tokens = 0, 0, 0, []
    worst = (0.0, tol)
    while out < n_new:
        toks, _ = dec.step()
        p, q, d, context = dec.last_step_debug(max_ctx)
        assert 1 <= len(toks) <= k + 1
        if heads is not None:
            ref = hd.spec_step(T, heads, ctx, k, temp, seed, step, tie_eps=tie)
        else:
            ref = gen.spec_step(T, D, ctx, k, temp, seed, step, prev, mix, tie_eps=tie)
        same = 0
        while same < k and ref.drafts[same] == int(d[same]):
            same += 1
        upto = k if heads is not None else min(k, same + 1)
        allow_q = tol
        if alt is not None:
            T_alt, D_alt = alt
            alt_heads = hd.head_logits(T_alt, heads, ctx) if heads is not None else None
            for i in range(upto):
                lq = alt_heads[i] if heads is not None else D_alt.logits(ctx + ref.drafts[:i], last=1)[0]
                if mix:
                    lq = (1.0 - mix) * lq + mix * np.asarray(prev[i], dtype=np.float64)
                allow_q = max(allow_q, tol + np.abs(lq - ref.q_logits[i]).max())
        err_q = np.abs(q[:upto] - ref.q_logits[:upto]).max()
        worst = max(worst, (err_q, allow_q))
        assert err_q < allow_q, (step, err_q, allow_q)
        if same == k:
            allow_p = tol
            if alt is not None:
                allow_p = tol + np.abs(alt[0].logits(ctx + ref.drafts, last=k + 1) - ref.p_logits).max()
            err_p = np.abs(p - ref.p_logits).max()
            worst = max(worst, (err_p, allow_p))
            assert err_p < allow_p, (step, err_p, allow_p)
        for i in range(k):
            dg, fl = gen.draft_token(q[i], temp, seed, step, i + 1, tie_eps=0.0)
            if not fl & SKIP_FLAGS:
                assert dg == int(d[i]), (step, i, dg, int(d[i]))
        if extra is not None:
            extra(step, ctx, p, q, d, ref)
        em, n, fl = gen.verify(p, q, list(d), temp, seed, step, tie_eps=0.0)
        if fl & SKIP_FLAGS:
            skipped += 1
        else:
            assert em == toks, (step, em, toks)
        assert [int(t) for t in context[len(ctx):]] == toks
        ctx = [int(t) for t in context]
        prev = p.astype(np.float64)
        tokens += toks
        out += len(toks)
        step += 1
    return tokens, step, skipped, worst
