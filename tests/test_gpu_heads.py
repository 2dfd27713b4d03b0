"""Self-draft heads (opts.draft_heads) against the oracle (oracle/heads.py).

"Speculative Decoding 101", Floor 6 and "Speculative decoding internals",
三條主流變體 (MTP): extra prediction heads on the target draft the next K
positions from its own final hidden state; the verification is unchanged.
The heads here are random (structure and cost only: no trained acceptance).

* Teacher-forced steps (helpers.teacher_forced with the heads oracle): every
  head row within the logit tolerance of the fp64 oracle, the drafts and the
  emitted tokens exact except flagged draws, the committed context equal --
  on the persistent kernel (bf16; 4-bit target with bf16 heads), on the
  one-kernel-per-operation bf16 path and on the fp32 path (5e-5).
* After plain-decoding steps the heads read the plain-decoding pass's row.
* Greedy speculative output with the heads equals greedy plain decoding.
* The 8B width (2 layers, vocabulary 128256) with K = 5 heads of 4096 x 4096,
  under the full-width tolerance (2e-2 plus the oracle's own
  bf16-dataflow-vs-fp64 gap, see test_gpu_fullwidth.py).
* Argument checks that need a context.
"""
from dataclasses import replace

import pytest
import torch

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads
from oracle import generate as gen

pytestmark = pytest.mark.gpu

K = 5
SMALL = workloads.small_shape()
Q4S = workloads.small_shape(name="q4small", dtype="q4", d_model=512, n_heads=8, n_kv_heads=2, head_dim=64,
                            ffn_dim=1024, vocab=1024)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


def _oracle(shape, w, act="f64"):
    return gen.Model(shape, helpers_cpu(w), act=act)


def helpers_cpu(w):
    return {"embed": w["embed"].cpu(), "final_norm": w["final_norm"].cpu(), "lm_head": w["lm_head"].cpu(),
            "layers": [{k: v.cpu() for k, v in lw.items()} for lw in w["layers"]]}


def _run(shape, w, T, heads, temp, flags=0, tol=2e-2, steps=24, prompt_len=30, seed=3, alt=None, max_ctx=256):
    prompt = workloads.make_prompt(shape.vocab, prompt_len, seed=seed)[0].tolist()
    dec = sv.SpecDecoder(shape, w, None, None, K, max_ctx, temperature=temp, seed=17, flags=flags, heads=heads)
    try:
        _, n, skipped, worst = helpers.teacher_forced(dec, T, None, prompt, K, temp, steps, tol, seed=17,
                                                      max_ctx=max_ctx, heads=heads.cpu(), alt=alt)
        assert skipped <= max(1, n // 4)
        return n, worst
    finally:
        dec.close()


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_heads_teacher_forced_bf16(temp):
    w = workloads.make_weights(SMALL, seed=51, device="cuda")
    heads = workloads.make_heads(SMALL, K, seed=52, device="cuda")
    n, worst = _run(SMALL, w, _oracle(SMALL, w), heads, temp)
    print(f"bf16 heads T={temp}: {n} steps, largest logit error {worst[0]:.4f}")


def test_heads_teacher_forced_bf16_per_operation():
    w = workloads.make_weights(SMALL, seed=53, device="cuda")
    heads = workloads.make_heads(SMALL, K, seed=54, device="cuda")
    _run(SMALL, w, _oracle(SMALL, w), heads, 1.0, flags=sv.SPEC_OPT_NO_PERSIST)


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_heads_teacher_forced_fp32(temp):
    w = workloads.make_weights(workloads.TINY, seed=55, device="cuda")
    heads = workloads.make_heads(workloads.TINY, K, seed=56, device="cuda", std=0.1)
    _run(workloads.TINY, w, _oracle(workloads.TINY, w), heads, temp, tol=5e-5, prompt_len=16)


def test_heads_teacher_forced_q4_target():
    from test_gpu_q4 import dense
    w = workloads.make_q4_weights(Q4S, seed=57, device="cuda")
    heads = workloads.make_heads(Q4S, K, seed=58, device="cuda")
    T = gen.Model(Q4S, dense(Q4S, w))
    _run(Q4S, w, T, heads, 1.0, prompt_len=40)


def test_heads_after_plain_decoding():
    w = workloads.make_weights(SMALL, seed=59, device="cuda")
    heads = workloads.make_heads(SMALL, K, seed=60, device="cuda")
    T = _oracle(SMALL, w)
    prompt = workloads.make_prompt(SMALL.vocab, 20, seed=61)[0].tolist()
    dec = sv.SpecDecoder(SMALL, w, None, None, K, 256, temperature=1.0, seed=19, heads=heads)
    try:
        dec.prefill(prompt)
        for _ in range(3):
            dec.ar_step()
        ctx = [int(t) for t in dec.seq_context(0)]
        assert len(ctx) == len(prompt) + 3
        helpers.teacher_forced(dec, T, None, ctx, K, 1.0, 10, 2e-2, seed=19, heads=heads.cpu(), prefilled=True)
    finally:
        dec.close()


def test_heads_greedy_spec_equals_greedy_ar():
    w = workloads.make_weights(SMALL, seed=62, device="cuda")
    heads = workloads.make_heads(SMALL, K, seed=63, device="cuda", std=0.05)
    prompt = workloads.make_prompt(SMALL.vocab, 24, seed=64)[0].tolist()
    dec = sv.SpecDecoder(SMALL, w, None, None, K, 256, heads=heads)
    try:
        dec.prefill(prompt)
        spec = dec.generate(48)
        st = dec.stats()
        dec.prefill(prompt)
        ar = [dec.ar_step() for _ in range(48)]
        assert spec == ar
        print(f"greedy heads: {st['steps']} steps for 48 tokens, accepted {st['drafts_accepted']}")
    finally:
        dec.close()


def test_heads_full_width():
    W8 = replace(workloads.EIGHT_B, n_layers=2)
    w = workloads.make_weights(W8, seed=65, device="cuda")
    heads = workloads.make_heads(W8, K, seed=66, device="cuda")
    cpu = {"embed": w["embed"].cpu(), "final_norm": w["final_norm"].cpu().double(),
           "lm_head": w["lm_head"].cpu().double(),
           "layers": [{k: v.cpu().double() for k, v in lw.items()} for lw in w["layers"]]}
    T, Tb = gen.Model(W8, cpu), gen.Model(W8, cpu, act="bf16")
    dec = sv.SpecDecoder(W8, w, None, None, K, 128, temperature=1.0, seed=23, heads=heads)
    try:
        lists = dec.phase_list(0)   # the heads pass
        gem = [p for p in lists if p[0] == 1]
        assert [p[1:4] for p in gem] == [(K * 4096, 4096, 1), (128256, 4096, K)]
        prompt = workloads.make_prompt(W8.vocab, 24, seed=67)[0].tolist()
        _, n, skipped, worst = helpers.teacher_forced(dec, T, None, prompt, K, 1.0, 8, 2e-2, seed=23,
                                                      max_ctx=128, heads=heads.cpu().double(), alt=(Tb, None))
        assert skipped <= max(1, n // 3)
        print(f"8B-width heads: {n} steps, largest logit error {worst[0]:.4f} (allowed {worst[1]:.4f})")
    finally:
        dec.close()


def test_heads_context_argument_checks():
    w = workloads.make_weights(SMALL, seed=68, device="cuda")
    heads = workloads.make_heads(SMALL, K, seed=69, device="cuda")
    dec = sv.SpecDecoder(SMALL, w, None, None, K, 256, heads=heads)
    try:
        out = torch.empty(2, SMALL.vocab, device="cuda")
        with pytest.raises(sv.SpecError, match="SPEC_E_ARG"):
            dec.model_forward(1, [1, 2], 0, out)   # no draft model
        with pytest.raises(sv.SpecError, match="SPEC_E_STATE"):
            dec.step()                              # before prefill
    finally:
        dec.close()
