"""Pins of the oracle's forward pass (component-wise).

The pages give no worked transformer example, so the forward is pinned to
library routines and closed forms instead of to itself:

* RMSNorm against torch.nn.functional.rms_norm;
* RoPE against its complex-number form (x_i + j x_{i+hd/2}) * e^{j pos w_i},
  identity at position 0, norm preservation, and the relative-position
  property <R(m) q, R(n) k> = <R(m+s) q, R(n+s) k>;
* causal GQA attention against torch.nn.functional.scaled_dot_product_attention
  with the KV heads repeated;
* SiLU against torch.nn.functional.silu;
* the whole decoder against a composition of torch.nn.functional routines
  (linear, rms_norm, scaled_dot_product_attention, silu) -- catches a
  transposed weight, a missing residual or a misplaced norm;
* causality: appending tokens never changes earlier positions' logits.
"""
import math

import pytest
import torch
import torch.nn.functional as F

import workloads
from oracle import model

F64 = torch.float64


def test_rms_norm_library():
    x = torch.randn(7, 64, dtype=F64)
    g = torch.rand(64, dtype=torch.float32) + 0.5
    want = F.rms_norm(x, (64,), weight=g.to(F64), eps=1e-5)
    assert torch.allclose(model.rms_norm(x, g, 1e-5), want, atol=1e-14)


def _rope_complex(x, positions, theta):
    hd = x.shape[-1]
    i = torch.arange(hd // 2, dtype=F64)
    w = float(theta) ** (-2.0 * i / hd)
    ang = torch.as_tensor(positions, dtype=F64)[:, None] * w[None, :]
    z = torch.complex(x[..., : hd // 2], x[..., hd // 2:]) * torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


@pytest.mark.parametrize("hd,theta", [(32, 10000.0), (64, 500000.0), (128, 500000.0)])
def test_rope(hd, theta):
    x = torch.randn(9, 3, hd, dtype=F64)
    pos = torch.arange(100, 109)
    y = model.apply_rope(x, pos, theta)
    assert torch.allclose(y, _rope_complex(x, pos, theta), atol=1e-12)
    assert torch.allclose(model.apply_rope(x, torch.zeros(9, dtype=torch.long), theta), x, atol=0)
    assert torch.allclose(y.norm(dim=-1), x.norm(dim=-1), atol=1e-12)
    q, k = torch.randn(1, 1, hd, dtype=F64), torch.randn(1, 1, hd, dtype=F64)
    dots = [(model.apply_rope(q, [m + s], theta) * model.apply_rope(k, [n + s], theta)).sum()
            for (m, n, s) in [(5, 2, 0), (5, 2, 37), (5, 2, 4000)]]
    assert float(dots[0]) == pytest.approx(float(dots[1]), abs=1e-10)
    assert float(dots[0]) == pytest.approx(float(dots[2]), abs=1e-9)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8)])
def test_attention_library(hq, hkv):
    n, hd = 11, 16
    q = torch.randn(n, hq, hd, dtype=F64)
    k = torch.randn(n, hkv, hd, dtype=F64)
    v = torch.randn(n, hkv, hd, dtype=F64)
    got = model.causal_attention(q, k, v)
    rep = hq // hkv
    want = F.scaled_dot_product_attention(
        q.transpose(0, 1), k.repeat_interleave(rep, dim=1).transpose(0, 1),
        v.repeat_interleave(rep, dim=1).transpose(0, 1), is_causal=True).transpose(0, 1)
    assert torch.allclose(got, want, atol=1e-12)
    # the first position attends to itself only
    assert torch.allclose(got[0], v[0].repeat_interleave(rep, dim=0), atol=1e-14)


def test_silu_library():
    x = torch.linspace(-30, 30, 1001, dtype=F64)
    assert torch.allclose(model.silu(x), F.silu(x), atol=1e-13)


def _library_forward(shape, w, tokens):
    """The decoder written with torch.nn.functional routines."""
    cast = lambda t: t.to(F64)
    tok = torch.as_tensor(tokens, dtype=torch.long)
    n = tok.numel()
    hq, hkv, hd = shape.n_heads, shape.n_kv_heads, shape.head_dim
    x = cast(w["embed"])[tok]
    pos = torch.arange(n)
    for lw in w["layers"]:
        a = F.rms_norm(x, (shape.d_model,), weight=cast(lw["attn_norm"]), eps=shape.rms_eps)
        q = _rope_complex(F.linear(a, cast(lw["wq"])).view(n, hq, hd), pos, shape.rope_theta)
        k = _rope_complex(F.linear(a, cast(lw["wk"])).view(n, hkv, hd), pos, shape.rope_theta)
        v = F.linear(a, cast(lw["wv"])).view(n, hkv, hd)
        rep = hq // hkv
        o = F.scaled_dot_product_attention(
            q.transpose(0, 1), k.repeat_interleave(rep, 1).transpose(0, 1),
            v.repeat_interleave(rep, 1).transpose(0, 1), is_causal=True).transpose(0, 1)
        x = x + F.linear(o.reshape(n, hq * hd), cast(lw["wo"]))
        b = F.rms_norm(x, (shape.d_model,), weight=cast(lw["ffn_norm"]), eps=shape.rms_eps)
        x = x + F.linear(F.silu(F.linear(b, cast(lw["w_gate"]))) * F.linear(b, cast(lw["w_up"])),
                         cast(lw["w_down"]))
    x = F.rms_norm(x, (shape.d_model,), weight=cast(w["final_norm"]), eps=shape.rms_eps)
    return F.linear(x, cast(w["lm_head"]))


@pytest.mark.parametrize("shape", [workloads.TINY, workloads.small_shape(dtype="bf16"),
                                   workloads.small_shape(dtype="f32", n_heads=4, n_kv_heads=1)])
def test_forward_library_composition(shape):
    w = workloads.make_weights(shape, seed=5)
    # random norm gains so that a dropped or misplaced gain shows
    g = torch.Generator().manual_seed(9)
    w["final_norm"] = torch.rand(shape.d_model, generator=g) + 0.5
    for lw in w["layers"]:
        lw["attn_norm"] = torch.rand(shape.d_model, generator=g) + 0.5
        lw["ffn_norm"] = torch.rand(shape.d_model, generator=g) + 0.5
    toks = workloads.make_prompt(shape.vocab, 13, seed=2)[0]
    got = model.forward(shape, w, toks)
    want = _library_forward(shape, w, toks)
    assert got.shape == (13, shape.vocab)
    assert torch.allclose(got, want, atol=1e-10, rtol=1e-10)
    last = model.forward(shape, w, toks, last=3)
    assert torch.allclose(last, got[-3:], atol=1e-12)


def test_causality():
    shape = workloads.TINY
    w = workloads.make_weights(shape, seed=1)
    toks = workloads.make_prompt(shape.vocab, 20, seed=3)[0]
    full = model.forward(shape, w, toks)
    part = model.forward(shape, w, toks[:12])
    assert torch.allclose(full[:12], part, atol=1e-12)
    other = toks.clone()
    other[15] = (other[15] + 1) % shape.vocab
    alt = model.forward(shape, w, other)
    assert torch.allclose(alt[:15], full[:15], atol=1e-12)
    assert not torch.allclose(alt[15:], full[15:])


# ---- the bf16 dataflow mode ------------------------------------------------

def test_round_bf16_nearest_even_by_hand():
    """bf16 keeps 8 significant bits: near 1 the spacing is 2^-7.  Halfway
    cases go to the even neighbour, everything else to the nearest."""
    x = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, 3.0, -(1 + 2 ** -8),
                      2 ** -130 * 3, 65280.0, 1 - 2 ** -9], dtype=torch.float64)
    want = [1.0, 1 + 2 ** -6, 1 + 2 ** -7, 3.0, -1.0, 2 ** -130 * 3, 65280.0, 1.0]
    assert model.round_bf16(x).tolist() == want


@pytest.mark.parametrize("shape", [workloads.TINY, workloads.small_shape(dtype="bf16")],
                         ids=lambda s: s.name)
def test_bf16_dataflow_without_rounding_is_the_definition(shape):
    """The bf16 dataflow's restructuring (gain before the GEMM and 1/rms on
    its sums; the softmax denominator apart from the weighted values) is the
    definition itself once the rounding is the identity; with the rounding on
    it moves the logits by a small, non-zero amount."""
    w = workloads.make_weights(shape, seed=3)
    g = torch.Generator().manual_seed(4)
    for lw in w["layers"]:   # non-trivial gains, so that the gain placement matters
        lw["attn_norm"] = 1 + 0.3 * torch.rand(shape.d_model, generator=g)
        lw["ffn_norm"] = 1 + 0.3 * torch.rand(shape.d_model, generator=g)
    w["final_norm"] = 1 + 0.3 * torch.rand(shape.d_model, generator=g)
    toks = workloads.make_prompt(shape.vocab, 24, seed=5)[0].tolist()
    ref = model.forward(shape, w, toks)
    same = model.forward(shape, w, toks, act="bf16", rnd=lambda t: t)
    assert (same - ref).abs().max() < 1e-11
    rounded = model.forward(shape, w, toks, act="bf16")
    d = (rounded - ref).abs().max().item()
    assert 1e-5 < d < 0.05, d


def test_rounded_attention_without_rounding_is_attention():
    g = torch.Generator().manual_seed(6)
    q = torch.randn(9, 4, 16, generator=g, dtype=torch.float64)
    k = torch.randn(9, 2, 16, generator=g, dtype=torch.float64)
    v = torch.randn(9, 2, 16, generator=g, dtype=torch.float64)
    a = model.causal_attention(q, k, v)
    b = model.causal_attention_rounded(q, k, v, lambda t: t)
    assert (a - b).abs().max() < 1e-13
