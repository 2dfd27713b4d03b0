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


def silu(x):
    return x / (1.0 + torch.exp(-x))


def decoder_layer(x, lw, shape, positions):
    n = x.shape[0]
    hq, hkv, hd = shape.n_heads, shape.n_kv_heads, shape.head_dim
    a = rms_norm(x, lw["attn_norm"], shape.rms_eps)
    q = (a @ _w(lw["wq"]).T).view(n, hq, hd)
    k = (a @ _w(lw["wk"]).T).view(n, hkv, hd)
    v = (a @ _w(lw["wv"]).T).view(n, hkv, hd)
    q = apply_rope(q, positions, shape.rope_theta)
    k = apply_rope(k, positions, shape.rope_theta)
    o = causal_attention(q, k, v).reshape(n, hq * hd)
    x = x + o @ _w(lw["wo"]).T
    b = rms_norm(x, lw["ffn_norm"], shape.rms_eps)
    h = silu(b @ _w(lw["w_gate"]).T) * (b @ _w(lw["w_up"]).T)
    return x + h @ _w(lw["w_down"]).T


def forward(shape, weights, tokens, last=None):
    """Logits [n, V] (fp64) at every position of ``tokens`` (positions 0..n-1).

    ``last``: if given, only the logits of the last ``last`` positions are
    returned (the LM head is applied to those rows only; the hidden states of
    all positions are still recomputed from scratch).
    """
    tok = torch.as_tensor(tokens, dtype=torch.long).reshape(-1)
    n = tok.numel()
    positions = torch.arange(n)
    x = _w(weights["embed"][tok.to(weights["embed"].device)])
    for lw in weights["layers"]:
        x = decoder_layer(x, lw, shape, positions)
    if last is not None:
        x = x[n - last:]
    x = rms_norm(x, weights["final_norm"], shape.rms_eps)
    return x @ _w(weights["lm_head"]).T
