"""Shared helpers of the GPU tests (not collected as tests)."""
import numpy as np
import torch

import speculative_decoding_verification_step_gb300 as sv
from oracle import accept as acc

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
