"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/specverify.h declares, and rejects bad
arguments with the documented codes before touching the device.  Without a
GPU, a valid spec_init fails with SPEC_E_CUDA: there is no CPU fallback."""
import ctypes
import os
import re

import pytest
import torch

import speculative_decoding_verification_step_gb300 as sv
from speculative_decoding_verification_step_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "specverify.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return sv.lib()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^SPEC_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
        assert n in sv.SIGNATURES, n
    assert set(sv.SIGNATURES) == set(names)


def test_version(L):
    assert b"sm_103a" in L.spec_version()


def _desc(vocab=256, head_dim=32, dtype=sv.SPEC_DTYPE_F32, layers=None):
    fake = 0x1000
    lay = (sv.LayerWeights * 1)()
    for n in sv._LAYER_FIELDS:
        setattr(lay[0], n, fake)
    d = sv.ModelDesc(1, 128, 4, 4, head_dim, 512, vocab, 10000.0, 1e-5, dtype, fake, fake, fake,
                     lay if layers is None else layers)
    return d, lay


def _init(L, t, d, k=4, max_ctx=128, batch=1, mix=0.0, lookup=0, heads=0):
    opts = sv.Opts(batch, max_ctx, 1.0, 0, mix, None, 0, lookup, heads)
    h = ctypes.c_void_p()
    rc = L.spec_init(ctypes.byref(t) if t is not None else None,
                     ctypes.byref(d) if d is not None else None, k, ctypes.byref(opts), ctypes.byref(h))
    return rc, h


def test_init_argument_errors(L):
    t, _a = _desc()
    d, _b = _desc()
    assert _init(L, None, d)[0] == -1                       # SPEC_E_ARG
    bad, _c = _desc(vocab=300)
    rc, h = _init(L, t, bad)
    assert rc == -2 and not h.value                         # SPEC_E_VOCAB
    assert b"vocabular" in L.spec_last_error(None)
    hd, _d = _desc(head_dim=48)
    assert _init(L, t, hd)[0] == -3                         # SPEC_E_SHAPE
    assert _init(L, t, d, k=0)[0] == -1
    assert _init(L, t, d, k=17)[0] == -1
    bf, _e = _desc(dtype=sv.SPEC_DTYPE_BF16)                # d_model 128 ok, ffn 512 ok
    bf.d_model = 96                                         # not a multiple of 64
    assert _init(L, bf, d)[0] == -3
    nulls = (sv.LayerWeights * 1)()
    nl, _f = _desc(layers=nulls)
    assert _init(L, nl, d)[0] == -1


def test_heads_argument_errors(L):
    """Self-draft heads replace the draft model: batch 1, no lookup, no mix,
    K <= 8, aligned weights, and no second (different) draft model."""
    t, _a = _desc()
    d, _b = _desc()
    heads = 0x2000
    assert _init(L, t, None, heads=heads, batch=2)[0] == -1
    assert _init(L, t, None, heads=heads, lookup=2)[0] == -1
    assert _init(L, t, None, heads=heads, mix=0.5)[0] == -1
    assert _init(L, t, None, heads=heads, k=9)[0] == -1
    assert _init(L, t, None, heads=heads + 4)[0] == -1      # not 16-byte aligned
    rc, h = _init(L, t, d, heads=heads)                     # a separate draft model as well
    assert rc == -1 and not h.value
    assert b"draft" in L.spec_last_error(None)


def test_lookup_argument_errors(L):
    t, _a = _desc()
    d, _b = _desc()
    assert _init(L, t, d, lookup=-1)[0] == -1
    assert _init(L, t, d, lookup=9)[0] == -1                # suffix matches of at most 8 tokens
    assert _init(L, t, d, lookup=3, mix=0.5)[0] == -1       # no draft logits to mix
    assert b"draft_mix_lambda" in L.spec_last_error(None)


def test_batch_argument_errors(L):
    t, _a = _desc()
    d, _b = _desc()
    assert _init(L, t, d, batch=0)[0] == -1
    assert _init(L, t, d, batch=sv.SPEC_MAX_BATCH + 1)[0] == -1
    assert _init(L, t, d, batch=2)[0] == -1                 # batch > 1 needs bf16 models
    assert b"bf16" in L.spec_last_error(None)
    bt, _c = _desc(dtype=sv.SPEC_DTYPE_BF16)
    bd, _d = _desc(dtype=sv.SPEC_DTYPE_BF16)
    assert _init(L, bt, bd, batch=2, mix=0.5)[0] == -1      # no draft mixing in batches
    assert b"draft_mix_lambda" in L.spec_last_error(None)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_no_cpu_fallback(L):
    t, _a = _desc()
    d, _b = _desc()
    rc, h = _init(L, t, d)
    assert rc == -5 and not h.value                         # SPEC_E_CUDA
    assert L.spec_last_error(None)


def test_stateless_argument_errors(L):
    rc = L.spec_accept_rows(None, 0, None, 0, None, 1, 4, 10, 1.0, 0, 0, None, None, None, None)
    assert rc == -1
    p = ctypes.c_void_p(0x1000)
    assert L.spec_accept_rows(p, 0, p, 0, p, 1, 17, 10, 1.0, 0, 0, p, p, None, None) == -1
    assert L.spec_accept_rows(p, 0, p, 0, p, 0, 4, 10, 1.0, 0, 0, p, p, None, None) == -1
    assert L.spec_sample_rows(None, 0, 1, 10, 1.0, 0, 0, 1, None, None) == -1
    assert L.spec_sample_rows(p, 0, 1, 10, -1.0, 0, 0, 1, p, None) == -1


def test_null_context_calls(L):
    L.spec_free(None)
    assert L.spec_prefill(None, None, 0) == -1
    assert L.spec_step(None, None, None, None) == -1
    assert L.spec_ar_step(None, None) == -1
    assert L.spec_prefill_synthetic(None, 16, 0) == -1
    assert L.spec_seq_context(None, 0, None, None) == -1
    assert L.spec_get_stats(None, None) == -1
    assert L.spec_last_error(None)


def test_binding_refuses_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(sv, "_lib", None)
    monkeypatch.setattr(sv, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        sv.lib()


def test_fault_hook_argument_errors(L):
    """spec_inject_fault checks its arguments before any device work; with no
    context and no allocation, no device memory is held."""
    assert L.spec_inject_fault(None, 99, 0) == -1                       # unknown kind
    assert L.spec_inject_fault(None, sv.SPEC_FAULT_ALLOC, 0) == -1      # n >= 1
    assert L.spec_inject_fault(None, sv.SPEC_FAULT_WAIT_TIMEOUT, 5) == -1   # needs a context
    assert L.spec_inject_fault(None, sv.SPEC_FAULT_ALLOC, 3) == 0
    assert L.spec_inject_fault(None, sv.SPEC_FAULT_CLEAR, 0) == 0
    assert L.spec_device_bytes_held() == 0
