"""GPU parity of the forward pass and of whole speculative steps, through the
C ABI, against the fp64 oracle.

* Forward: logits of the target/draft forward over 150 tokens (three prefill
  chunks, ragged tail) within 2e-2 (bf16 models, fp32 accumulation) or 5e-5
  (fp32 models) of the oracle's full causal recompute.
* Batch invariance: the same positions scored one at a time, or as a
  (K+1)-token verify block, give bit-identical logits.
* Steps (tiny speculative-generation workload, K = 4, prompt 16, 64 new
  tokens, greedy and T = 1, Philox seed 0): teacher-forced step by step --
  stage (i) the draft/target logits of each step against the oracle's own
  forward on the same context (up to the first draft that differs from the
  oracle's); stage (ii) the oracle's draft draw on the GPU's draft rows and
  its acceptance on the GPU's logits and drafts must reproduce the GPU's
  drafts and emitted tokens exactly, except flagged near-boundary draws.
* Greedy speculative output equals greedy plain decoding on the GPU.
* A draft equal to the target accepts every draft.
"""
import numpy as np
import pytest
import torch

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads
from oracle import generate as gen
from oracle import model as omodel

pytestmark = pytest.mark.gpu

# bf16 shapes with head dims 64 and 128: attention items read V in halves
HD_SHAPES = [workloads.small_shape(name="hd64", dtype="bf16", n_heads=4, n_kv_heads=2, head_dim=64),
             workloads.small_shape(name="hd128", dtype="bf16", n_heads=2, n_kv_heads=1, head_dim=128)]
SHAPES = [workloads.TINY, workloads.small_shape(dtype="bf16"),
          workloads.small_shape(dtype="f32", n_heads=4, n_kv_heads=1, head_dim=64)] + HD_SHAPES


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s.name}-{s.dtype}-hd{s.head_dim}")
def test_forward_parity_and_batch_invariance(shape):
    w = workloads.make_weights(shape, seed=1)
    wc = helpers.to_device(w)
    dec = helpers.decoder(shape, wc, shape, wc, 4, 256)
    toks = workloads.make_prompt(shape.vocab, 150, seed=2)[0].tolist()
    full = torch.empty(150, shape.vocab, device="cuda")
    dec.model_forward(0, toks, 0, full)
    ref = omodel.forward(shape, w, toks).numpy()
    got = full.cpu().numpy()
    err = np.abs(got - ref).max()
    assert err < helpers.logit_tol(shape), err
    # one position at a time, then a 6-token block, over the cached prefix
    one = torch.empty(1, shape.vocab, device="cuda")
    for pos in range(100, 106):
        dec.model_forward(0, [toks[pos]], pos, one)
        assert torch.equal(one[0], full[pos]), pos
    blk = torch.empty(6, shape.vocab, device="cuda")
    dec.model_forward(0, toks[100:106], 100, blk)
    assert torch.equal(blk, full[100:106])
    dec.close()


def _tiny_pair():
    shape = workloads.TINY
    w = workloads.make_weights(shape, seed=0)
    dshape, dw = workloads.noisy_layer0_draft(shape, w, seed=1)
    prompt = workloads.make_prompt(shape.vocab, 16, seed=0)[0].tolist()
    return shape, w, dshape, dw, prompt


def _teacher_forced(shape, w, dshape, dw, prompt, k, temp, n_new, mix=0.0, seed=0, max_ctx=256):
    dec = helpers.decoder(shape, helpers.to_device(w), dshape, helpers.to_device(dw), k, max_ctx,
                          temperature=temp, seed=seed, mix=mix)
    try:
        return helpers.teacher_forced(dec, gen.Model(shape, w), gen.Model(dshape, dw), prompt, k, temp,
                                      n_new, helpers.logit_tol(shape), mix=mix, seed=seed, max_ctx=max_ctx,
                                      tie=helpers.tie_eps(shape))[:3]
    finally:
        dec.close()


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_tiny_generation_teacher_forced(temp):
    shape, w, dshape, dw, prompt = _tiny_pair()
    tokens, steps, skipped = _teacher_forced(shape, w, dshape, dw, prompt, 4, temp, 64)
    assert skipped <= steps // 5


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_tiny_generation_free_running(temp):
    """Config 1 compared free-running: the GPU's 64 tokens equal the oracle's."""
    shape, w, dshape, dw, prompt = _tiny_pair()
    dec = helpers.decoder(shape, helpers.to_device(w), dshape, helpers.to_device(dw), 4, 128,
                          temperature=temp, seed=0)
    dec.prefill(prompt)
    got = dec.generate(64)
    ref, steps = gen.generate(gen.Model(shape, w), gen.Model(dshape, dw), prompt, 64, 4, temp, 0)
    flagged = any(s.flags & helpers.SKIP_FLAGS for s in steps)
    if not flagged:
        assert got == ref
    else:   # a flagged near-boundary draw may legitimately diverge; compare up to it
        first = next(i for i, s in enumerate(steps) if s.flags & helpers.SKIP_FLAGS)
        upto = sum(len(s.emitted) for s in steps[:first])
        assert got[:upto] == ref[:upto]
    dec.close()


@pytest.mark.parametrize("mix", [0.5])
def test_small_bf16_mixed_draft_teacher_forced(mix):
    shape = workloads.small_shape(dtype="bf16")
    w = workloads.make_weights(shape, seed=4)
    dshape, dw = workloads.prefix_draft(shape, w, 1)
    prompt = workloads.make_prompt(shape.vocab, 40, seed=5)[0].tolist()
    _teacher_forced(shape, w, dshape, dw, prompt, 5, 1.0, 30, mix=mix)


@pytest.mark.parametrize("shape", HD_SHAPES, ids=lambda s: s.name)
def test_head_dims_teacher_forced(shape):
    """The persistent kernel's attention at head dims 64 and 128 (V read in
    halves by two items per row), step by step against the oracle."""
    w = workloads.make_weights(shape, seed=15)
    dshape, dw = workloads.prefix_draft(shape, w, 1)
    prompt = workloads.make_prompt(shape.vocab, 60, seed=16)[0].tolist()
    _teacher_forced(shape, w, dshape, dw, prompt, 5, 1.0, 24)


def test_long_context_forward_crosses_key_split():
    """Past 1024 keys a row's attention spans two key splits (merged by the
    last split in split order): forward logits against the oracle, and
    positions 1020..1027 scored alone or in a block from an odd position
    bit-identical to the full forward."""
    shape = workloads.small_shape(dtype="bf16")
    w = workloads.make_weights(shape, seed=11)
    wc = helpers.to_device(w)
    dec = helpers.decoder(shape, wc, shape, wc, 4, 1200)
    n = 1100
    toks = workloads.make_prompt(shape.vocab, n, seed=12)[0].tolist()
    full = torch.empty(n, shape.vocab, device="cuda")
    dec.model_forward(0, toks, 0, full)
    ref = omodel.forward(shape, w, toks).numpy()
    err = np.abs(full.cpu().numpy()[1000:] - ref[1000:]).max()
    assert err < helpers.logit_tol(shape), err
    one = torch.empty(1, shape.vocab, device="cuda")
    for pos in range(1020, 1028):
        dec.model_forward(0, [toks[pos]], pos, one)
        assert torch.equal(one[0], full[pos]), pos
    blk = torch.empty(6, shape.vocab, device="cuda")
    dec.model_forward(0, toks[1021:1027], 1021, blk)
    assert torch.equal(blk, full[1021:1027])
    dec.close()


def test_long_context_steps_teacher_forced():
    """Speculative steps at 1050+ positions: the persistent kernel's
    attention merges two key splits per row; draft and target logits and the
    emitted tokens are checked against the oracle step by step."""
    shape = workloads.small_shape(dtype="bf16")
    w = workloads.make_weights(shape, seed=13)
    dshape, dw = workloads.prefix_draft(shape, w, 1)
    prompt = workloads.make_prompt(shape.vocab, 1050, seed=14)[0].tolist()
    _teacher_forced(shape, w, dshape, dw, prompt, 5, 1.0, 20, max_ctx=1200)


def test_long_context_greedy_spec_equals_greedy_ar():
    """Past position 1024 the verify pass's attention takes every token of a
    KV head in one item (token-group mode) while plain decoding scores one
    token per item: a row's arithmetic must not depend on that, so greedy
    speculative output equals greedy plain decoding token for token."""
    shape = workloads.small_shape(dtype="bf16")
    w = workloads.make_weights(shape, seed=15)
    dshape, dw = workloads.prefix_draft(shape, w, 1)
    wc = helpers.to_device(w)
    dwc = {**wc, "layers": wc["layers"][:1]}
    dec = helpers.decoder(shape, wc, dshape, dwc, 5, 1200)
    prompt = workloads.make_prompt(shape.vocab, 1040, seed=16)[0].tolist()
    dec.prefill(prompt)
    spec = dec.generate(40)
    dec.prefill(prompt)
    ar = [dec.ar_step() for _ in range(40)]
    assert spec == ar
    dec.close()


@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: f"{s.name}-{s.dtype}")
def test_greedy_spec_equals_greedy_ar(shape):
    w = workloads.make_weights(shape, seed=6)
    dshape, dw = workloads.prefix_draft(shape, w, 1)
    wc = helpers.to_device(w)
    dwc = {**wc, "layers": wc["layers"][:1]}
    dec = helpers.decoder(shape, wc, dshape, dwc, 4, 256)
    prompt = workloads.make_prompt(shape.vocab, 30, seed=7)[0].tolist()
    dec.prefill(prompt)
    spec = dec.generate(60)
    dec.prefill(prompt)
    ar = [dec.ar_step() for _ in range(60)]
    assert spec == ar
    st = dec.stats()
    assert st["ar_steps"] == 60
    dec.close()


@pytest.mark.parametrize("temp", [0.0, 1.0])
@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: f"{s.name}-{s.dtype}")
def test_ar_step_teacher_forced(shape, temp):
    """Plain decoding (spec_ar_step, the speedup's denominator) against the
    oracle step by step: each pass's logits within tolerance of the oracle's
    forward on the GPU's committed context, and the token the oracle's
    plain-decoding draw (argmax, or inverse CDF with the step's stream-4
    uniform) takes on the GPU's logits -- exact except flagged draws."""
    w = workloads.make_weights(shape, seed=9)
    dshape, dw = workloads.prefix_draft(shape, w, 1)
    wc = helpers.to_device(w)
    dwc = {**wc, "layers": wc["layers"][:1]}
    dec = helpers.decoder(shape, wc, dshape, dwc, 4, 128, temperature=temp, seed=5)
    prompt = workloads.make_prompt(shape.vocab, 20, seed=10)[0].tolist()
    dec.prefill(prompt)
    T = gen.Model(shape, w)
    tol = helpers.logit_tol(shape)
    ctx, skipped = list(prompt), 0
    for s in range(16):
        tok = dec.ar_step()
        p, _, _, context = dec.last_step_debug(128)
        ref = T.logits(ctx, last=1)[0]
        assert np.abs(p[0] - ref).max() < tol, s
        exp, fl = gen.ar_token_flagged(p[0], temp, 5, s, tie_eps=0.0)
        if fl & helpers.SKIP_FLAGS:
            skipped += 1
        else:
            assert exp == tok, (s, exp, tok)
        assert [int(t) for t in context] == ctx + [tok]
        ctx.append(tok)
    assert skipped <= 3
    assert dec.stats()["ar_steps"] == 16
    dec.close()


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_draft_equal_target_accepts_all(temp):
    shape = workloads.small_shape(dtype="bf16")
    w = workloads.make_weights(shape, seed=8)
    wc = helpers.to_device(w)
    dec = helpers.decoder(shape, wc, shape, wc, 5, 256, temperature=temp, seed=3)
    dec.prefill(workloads.make_prompt(shape.vocab, 20, seed=1)[0].tolist())
    for _ in range(8):
        toks, flags = dec.step()
        assert len(toks) == 6 and flags & sv.SPEC_FLAG_ALL_ACCEPTED
    st = dec.stats()
    assert st["accept_hist"][5] == 8
    dec.close()


def test_state_and_capacity_errors():
    shape, w, dshape, dw, prompt = _tiny_pair()
    dec = helpers.decoder(shape, helpers.to_device(w), dshape, helpers.to_device(dw), 4, 32)
    with pytest.raises(sv.SpecError, match="SPEC_E_STATE"):
        dec.step()
    with pytest.raises(sv.SpecError, match="SPEC_E_CAPACITY"):
        dec.prefill(list(range(30)))
    with pytest.raises(sv.SpecError, match="SPEC_E_ARG"):
        dec.prefill([0, 999])
    dec.prefill(prompt)
    n = 0
    with pytest.raises(sv.SpecError, match="SPEC_E_CAPACITY"):
        for _ in range(40):
            n += len(dec.step()[0])
    assert n > 0
    dec.prefill(prompt)
    dec.ar_step()
    with pytest.raises(sv.SpecError, match="SPEC_E_STATE"):
        dec.step()
    dec.close()


def test_vocab_mismatch():
    shape = workloads.TINY
    w = helpers.to_device(workloads.make_weights(shape, seed=0))
    from dataclasses import replace
    other = replace(shape, vocab=128)
    ow = dict(w)
    ow["embed"] = w["embed"][:128].contiguous()
    ow["lm_head"] = w["lm_head"][:128].contiguous()
    with pytest.raises(sv.SpecError, match="SPEC_E_VOCAB"):
        helpers.decoder(shape, w, other, ow, 4, 64)
