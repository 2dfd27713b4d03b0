"""Llama-style decoder forward in fp64 with no KV cache (host side).

Test infrastructure: see the package docstring.

The pages fix only what the target pass must return: one next-token
distribution at every position of (prefix, d_1..d_K), all from one forward
("Speculative decoding internals", 演算法核心, Step 2; "Speculative Decoding
101", Floor 3).  The model itself is fixed by the synthetic workloads, with
these readings where they are silent:

* pre-norm residual blocks, no biases;
* RMSNorm y = x / sqrt(mean(x^2) + eps) * g;
* rotate-half RoPE: pairs (i, i + hd/2) rotated by pos * theta^(-2i/hd);
* grouped-query attention: query head h reads KV head floor(h * h_kv / h_q),
  scores scaled by 1/sqrt(hd), causal;
* SwiGLU MLP: W_down(silu(W_gate x) * W_up x);
* untied LM head on the final RMSNorm.

Every position is recomputed from the token ids each call (the plain
definition of causal self-attention); nothing is cached.  Weights are read
exactly as given (bf16 or fp32 bits) and widened to fp64.

Two precisions (``act``):

* ``"f64"`` (default): the definition, every activation in fp64.
* ``"bf16"``: the dataflow of a bf16 model with fp32 accumulation -- the
  precision the benchmark's bf16 models are specified in.  Arithmetic stays
  fp64 (more exact than fp32 accumulation); activations are rounded to bf16
  (round to nearest even) where a bf16 model stores them between
  operations: every GEMM input (an RMSNorm'd input as bf16(x * gain), its
  1/rms applied to the GEMM's sums -- the same product as normalising
  first), q, k and v where attention reads them, the attention output and
  the SwiGLU output.  The residual stream, norms, RoPE, the softmax and its
  probabilities stay unrounded (the probabilities that weight v are kept to
  ~16 significant bits, a bf16 pair; rounded to one bf16 they would move a
  4096-wide model's logits by up to ~0.05, by an amount that depends on the
  order the keys are visited in).  With the rounding replaced by the
  identity this mode is the definition itself (a pinned property).
"""
import math

import torch

F64 = torch.float64


def _w(t):
    return t.detach().to("cpu").to(F64)


def rms_norm(x, gain, eps):
    ms = (x * x).mean(dim=-1, keepdim=True)
    return x / torch.sqrt(ms + eps) * _w(gain)


def rope_angles(positions, head_dim, theta):
    """[n, hd/2] angles pos * theta^(-2i/hd), in fp64."""
    i = torch.arange(head_dim // 2, dtype=F64)
    inv_freq = torch.pow(torch.tensor(float(theta), dtype=F64), -2.0 * i / head_dim)
    return torch.as_tensor(positions, dtype=F64)[:, None] * inv_freq[None, :]


def apply_rope(x, positions, theta):
    """Rotate-half RoPE on x [n, heads, hd]."""
    hd = x.shape[-1]
    ang = rope_angles(positions, hd, theta)
    cos, sin = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def causal_attention(q, k, v):
    """q [n, hq, hd], k/v [n, hkv, hd] -> [n, hq, hd]; GQA head map h -> h*hkv//hq."""
    n, hq, hd = q.shape
    hkv = k.shape[1]
    out = torch.empty_like(q)
    mask = torch.triu(torch.ones(n, n, dtype=torch.bool), diagonal=1)
    for h in range(hq):
        g = (h * hkv) // hq
        s = (q[:, h, :] @ k[:, g, :].T) / math.sqrt(hd)
        s = s.masked_fill(mask, float("-inf"))
        s = s - s.max(dim=-1, keepdim=True).values
        e = torch.exp(s)
        out[:, h, :] = (e / e.sum(dim=-1, keepdim=True)) @ v[:, g, :]
    return out


def causal_attention_rounded(q, k, v, rnd):
    """causal_attention in a bf16 model's dataflow: q, k and v as rnd(q),
    rnd(k), rnd(v); the softmax unrounded.  With rnd = identity this is
    causal_attention."""
    return causal_attention(rnd(q), rnd(k), rnd(v))


def silu(x):
    return x / (1.0 + torch.exp(-x))


def round_bf16(t):
    """Round fp64 values to the nearest bf16 (ties to even), widened back."""
    return t.to(torch.bfloat16).to(F64)


def _identity(t):
    return t


def _norm_input(x, gain, eps, rnd):
    """An RMSNorm'd GEMM input as (a, s) with rms_norm(x) = a * s, the GEMM
    applied to a and its sums scaled by s.  Definition (rnd None): a = the
    normalised x, s = 1.  bf16 dataflow: a = rnd(x * gain), s = 1 / rms(x)."""
    if rnd is None:
        return rms_norm(x, gain, eps), 1.0
    inv = 1.0 / torch.sqrt((x * x).mean(dim=-1, keepdim=True) + eps)
    return rnd(x * _w(gain)), inv


def decoder_layer(x, lw, shape, positions, rnd=None):
    """One pre-norm block.  rnd None: the fp64 definition; else the rounding
    of the bf16 dataflow (see the module docstring)."""
    n = x.shape[0]
    hq, hkv, hd = shape.n_heads, shape.n_kv_heads, shape.head_dim
    a, sa = _norm_input(x, lw["attn_norm"], shape.rms_eps, rnd)
    q = ((a @ _w(lw["wq"]).T) * sa).view(n, hq, hd)
    k = ((a @ _w(lw["wk"]).T) * sa).view(n, hkv, hd)
    v = ((a @ _w(lw["wv"]).T) * sa).view(n, hkv, hd)
    q = apply_rope(q, positions, shape.rope_theta)
    k = apply_rope(k, positions, shape.rope_theta)
    if rnd is None:
        o = causal_attention(q, k, v).reshape(n, hq * hd)
    else:
        o = rnd(causal_attention_rounded(q, k, v, rnd).reshape(n, hq * hd))
    x = x + o @ _w(lw["wo"]).T
    b, sb = _norm_input(x, lw["ffn_norm"], shape.rms_eps, rnd)
    h = silu((b @ _w(lw["w_gate"]).T) * sb) * ((b @ _w(lw["w_up"]).T) * sb)
    if rnd is not None:
        h = rnd(h)
    return x + h @ _w(lw["w_down"]).T


ACT_ROUNDING = {"f64": None, "bf16": round_bf16}


def hidden(shape, weights, tokens, rnd=None):
    """Residual stream [n, d] (fp64) after the last decoder layer, at every
    position of ``tokens`` (positions 0..n-1), before the final RMSNorm."""
    tok = torch.as_tensor(tokens, dtype=torch.long).reshape(-1)
    positions = torch.arange(tok.numel())
    x = _w(weights["embed"][tok.to(weights["embed"].device)])
    for lw in weights["layers"]:
        x = decoder_layer(x, lw, shape, positions, rnd)
    return x


def final_input(shape, weights, x, rnd=None):
    """The LM head's input for residual rows x, as (a, s) (see _norm_input)."""
    return _norm_input(x, weights["final_norm"], shape.rms_eps, rnd)


def forward(shape, weights, tokens, last=None, act="f64", rnd=None):
    """Logits [n, V] (fp64) at every position of ``tokens`` (positions 0..n-1).

    ``last``: if given, only the logits of the last ``last`` positions are
    returned (the LM head is applied to those rows only; the hidden states of
    all positions are still recomputed from scratch).
    ``act``: "f64" (the definition) or "bf16" (a bf16 model's dataflow, see
    the module docstring).  ``rnd`` overrides the dataflow's rounding function
    (tests replace it by the identity).
    """
    if rnd is None:
        rnd = ACT_ROUNDING[act]
    x = hidden(shape, weights, tokens, rnd)
    if last is not None:
        x = x[x.shape[0] - last:]
    a, s = final_input(shape, weights, x, rnd)
    return (a @ _w(weights["lm_head"]).T) * s
