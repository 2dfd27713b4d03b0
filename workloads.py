"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds model shapes and random-input recipes only -- none of the
speculative-decoding arithmetic.  Both the CUDA path (through its tests and
``bench.py``) and the fp64 oracle read the tensors it makes, so both see the
same bits.  Nothing here imports the CUDA library or the oracle.

Recipes (all seeded, all synthetic; no dataset or trained weight is used):

* Weights: every matrix and embedding ~ N(0, 0.02^2), drawn in fp32 by
  ``torch.randn`` with a seeded ``torch.Generator`` on the requested device,
  then rounded to the model dtype.  RMSNorm gains are 1 (fp32).
* Tiny draft: the target's embedding, layer 0, final-norm gain and LM head,
  each plus N(0, 0.01^2) noise.
* Prefix draft: the target's first n layers with the shared final norm and
  LM head (views of the same buffers, no copy).
* Prompts: token ids uniform on [0, vocab).
* Acceptance rows: target logits ~ N(0, 3^2); draft logits = target rows
  1..K plus N(0, sigma^2).
* 4-bit weights (dtype "q4"): every matrix [n][k] gets codes uniform on
  [-8, 7] and one bf16 scale per 64-k group, uniform on [0.75, 1.25] x
  0.02 / 4.6 (weights of std ~0.02), laid out as the library takes them:
  codes packed two per byte (element 2b in the low nibble), then the scales
  group-major [k/64][n].  The embedding is bf16 N(0, 0.02^2), gains 1.
"""
from dataclasses import dataclass, replace

import torch

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-5
    dtype: str = "bf16"          # "f32", "bf16" or "q4" (4-bit weights, bf16 arithmetic)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self):
        """Bytes per streamed weight (q4: a nibble plus a bf16 scale per 64)."""
        return 4 if self.dtype == "f32" else 2 if self.dtype == "bf16" else 0.5 + 2 / 64

    @property
    def act_bytes(self):
        """Bytes per activation / KV element."""
        return 4 if self.dtype == "f32" else 2

    def layer_params(self):
        d, hd = self.d_model, self.head_dim
        attn = d * hd * (2 * self.n_heads + 2 * self.n_kv_heads)
        return attn + 3 * d * self.ffn_dim

    def weight_bytes(self, n_layers=None, head=True):
        """Bytes of matrices streamed by one forward pass (norm gains excluded)."""
        n = self.n_layers if n_layers is None else n_layers
        b = n * self.layer_params() * self.elem_bytes
        if head:
            b += self.vocab * self.d_model * self.elem_bytes
        return b

    def kv_bytes_per_token(self):
        return self.n_layers * 2 * self.n_kv_heads * self.head_dim * self.act_bytes


# Tiny speculative-generation model: 2 layers, d=128, 4 heads, SwiGLU 512,
# vocab 256, fp32.
TINY = ModelShape("tiny", 2, 128, 4, 4, 32, 512, 256, 10000.0, dtype="f32")
# 1B-shaped: 16 layers, d=2048, 32/8 heads (hd 64), FFN 8192, vocab 128256.
ONE_B = ModelShape("1b", 16, 2048, 32, 8, 64, 8192, 128256, 500000.0)
# 8B-shaped: 32 layers, d=4096, 32/8 heads (hd 128), FFN 14336, vocab 128256.
EIGHT_B = ModelShape("8b", 32, 4096, 32, 8, 128, 14336, 128256, 500000.0)


def small_shape(name="small", dtype="bf16", **kw):
    """A scaled-down Llama-style shape with GQA, for parity tests."""
    base = ModelShape(name, 2, 256, 8, 2, 32, 384, 1000, 500000.0, dtype=dtype)
    return replace(base, **kw)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, std, dtype):
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(std).to(dtype)


def make_weights(shape: ModelShape, seed: int, device="cpu", std=0.02):
    """Random-init weights in the layout the C-ABI takes (row-major [out][in])."""
    g = _gen(seed, device)
    dt = shape.torch_dtype
    d, hd, f = shape.d_model, shape.head_dim, shape.ffn_dim
    w = {
        "embed": _randn((shape.vocab, d), g, device, std, dt),
        "final_norm": torch.ones(d, dtype=torch.float32, device=device),
        "lm_head": None,
        "layers": [],
    }
    for _ in range(shape.n_layers):
        w["layers"].append({
            "attn_norm": torch.ones(d, dtype=torch.float32, device=device),
            "wq": _randn((shape.n_heads * hd, d), g, device, std, dt),
            "wk": _randn((shape.n_kv_heads * hd, d), g, device, std, dt),
            "wv": _randn((shape.n_kv_heads * hd, d), g, device, std, dt),
            "wo": _randn((d, shape.n_heads * hd), g, device, std, dt),
            "ffn_norm": torch.ones(d, dtype=torch.float32, device=device),
            "w_gate": _randn((f, d), g, device, std, dt),
            "w_up": _randn((f, d), g, device, std, dt),
            "w_down": _randn((d, f), g, device, std, dt),
        })
    w["lm_head"] = _randn((shape.vocab, d), g, device, std, dt)
    return w


def noisy_layer0_draft(shape: ModelShape, target_w, seed: int, sigma=0.01):
    """Draft = target embedding + layer 0 + final norm + LM head, each + N(0, sigma^2)."""
    dev = target_w["embed"].device
    g = _gen(seed, dev)

    def noisy(t):
        n = torch.randn(t.shape, generator=g, device=dev, dtype=torch.float32) * sigma
        return (t.float() + n).to(t.dtype)

    lay = {k: noisy(v) for k, v in target_w["layers"][0].items()}
    dw = {"embed": noisy(target_w["embed"]), "final_norm": noisy(target_w["final_norm"]),
          "lm_head": noisy(target_w["lm_head"]), "layers": [lay]}
    return replace(shape, name=shape.name + "-draft", n_layers=1), dw


def prefix_draft(shape: ModelShape, target_w, n_layers: int):
    """Draft = target's first n layers + shared final norm and LM head (views)."""
    dw = {"embed": target_w["embed"], "final_norm": target_w["final_norm"],
          "lm_head": target_w["lm_head"], "layers": target_w["layers"][:n_layers]}
    return replace(shape, name=f"{shape.name}-first{n_layers}", n_layers=n_layers), dw


def make_prompt(vocab: int, length: int, seed: int, batch: int = 1):
    g = _gen(seed, "cpu")
    return torch.randint(0, vocab, (batch, length), generator=g, dtype=torch.int64).to(torch.int32)


def make_accept_rows(rows: int, k: int, vocab: int, sigma: float, seed: int,
                     device="cpu", target_std=3.0):
    """Acceptance-kernel inputs: target logits [rows, K+1, V] ~ N(0, 3^2) and
    draft logits [rows, K, V] = target rows 1..K + N(0, sigma^2) (fp32)."""
    g = _gen(seed, device)
    p = torch.randn(rows, k + 1, vocab, generator=g, device=device, dtype=torch.float32)
    p.mul_(target_std)
    q = torch.randn(rows, k, vocab, generator=g, device=device, dtype=torch.float32)
    q.mul_(sigma).add_(p[:, :k, :])
    return p, q


def q4_matrix(n, k, g, device, scale=0.02 / 4.6):
    """One 4-bit matrix in the library's layout (uint8 buffer: packed codes
    [n][k/2], then bf16 scales [k/64][n])."""
    codes = torch.randint(-8, 8, (n, k), generator=g, device=device, dtype=torch.int16)
    nib = (codes & 0xF).to(torch.uint8)
    packed = nib[:, 0::2] | (nib[:, 1::2] << 4)
    scales = (torch.rand(k // 64, n, generator=g, device=device, dtype=torch.float32) * 0.5 + 0.75) * scale
    sb = scales.to(torch.bfloat16).contiguous().view(torch.uint8).reshape(-1)
    return torch.cat([packed.reshape(-1), sb])


def q4_parts(buf, n, k):
    """(packed codes [n][k/2] uint8, scales [n][k/64] fp32 holding bf16 values)
    of a 4-bit matrix buffer, as host tensors."""
    b = buf.detach().cpu()
    packed = b[: n * k // 2].reshape(n, k // 2)
    scales = b[n * k // 2:].view(torch.bfloat16).reshape(k // 64, n).t().float()
    return packed, scales


def make_q4_weights(shape: ModelShape, seed: int, device="cpu"):
    """Random 4-bit weights (see the module docstring), same dict layout as
    make_weights; the matrices are uint8 buffers."""
    g = _gen(seed, device)
    d, hd, f = shape.d_model, shape.head_dim, shape.ffn_dim
    w = {"embed": _randn((shape.vocab, d), g, device, 0.02, torch.bfloat16),
         "final_norm": torch.ones(d, dtype=torch.float32, device=device), "layers": []}
    for _ in range(shape.n_layers):
        w["layers"].append({
            "attn_norm": torch.ones(d, dtype=torch.float32, device=device),
            "wq": q4_matrix(shape.n_heads * hd, d, g, device),
            "wk": q4_matrix(shape.n_kv_heads * hd, d, g, device),
            "wv": q4_matrix(shape.n_kv_heads * hd, d, g, device),
            "wo": q4_matrix(d, shape.n_heads * hd, g, device),
            "ffn_norm": torch.ones(d, dtype=torch.float32, device=device),
            "w_gate": q4_matrix(f, d, g, device),
            "w_up": q4_matrix(f, d, g, device),
            "w_down": q4_matrix(d, f, g, device),
        })
    w["lm_head"] = q4_matrix(shape.vocab, d, g, device)
    return w


def make_heads(shape: ModelShape, k: int, seed: int, device="cpu", std=0.02):
    """Random self-draft heads: K stacked row-major d x d matrices [K, d, d]
    in the target's arithmetic dtype (bf16 for bf16 and 4-bit targets)."""
    g = _gen(seed, device)
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    return _randn((k, shape.d_model, shape.d_model), g, device, std, dt)


# matrix name -> (rows, k) of a shape
def matrix_dims(shape: ModelShape, name):
    d, hd, f = shape.d_model, shape.head_dim, shape.ffn_dim
    return {"wq": (shape.n_heads * hd, d), "wk": (shape.n_kv_heads * hd, d), "wv": (shape.n_kv_heads * hd, d),
            "wo": (d, shape.n_heads * hd), "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f),
            "lm_head": (shape.vocab, d)}[name]
