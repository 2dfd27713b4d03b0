"""GPU parity of prompt-lookup drafting ("Speculative Decoding 101", Floor 6)
through the C ABI, against the oracle (oracle/lookup.py).

Prompts repeat a segment, so the suffix search finds matches.  Per step,
teacher-forced: the GPU's drafts equal the oracle's lookup on the GPU's own
committed context (integer work: exact), the q rows are one-hot at the
drafts, the target logits agree with the oracle's forward within the
forward tolerance, and the oracle's acceptance (row word b) on the GPU's
logits reproduces the emitted tokens except flagged near-boundary draws.
Covered: the tiny fp32 model (per-operation path), a bf16 model on the
persistent kernel, and a 3-sequence batch.  Greedy prompt-lookup output
equals greedy plain decoding on the persistent path.
"""
import numpy as np
import pytest

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads
from oracle import generate as gen
from oracle import lookup as lk

pytestmark = pytest.mark.gpu

BF16 = workloads.small_shape(name="hd64", dtype="bf16", n_heads=4, n_kv_heads=2, head_dim=64)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


def _prompt(vocab, seed, batch=1):
    """Random ids with a repeated segment: a b ... (12 tokens) x ... a b ..."""
    base = workloads.make_prompt(vocab, 28, seed=seed, batch=batch).tolist()
    return [row[:12] + row[12:20] + row[:12] for row in base]


@pytest.mark.parametrize("shape", [workloads.TINY, BF16], ids=lambda s: f"{s.name}-{s.dtype}")
@pytest.mark.parametrize("temp", [0.0, 1.0])
@pytest.mark.parametrize("nseq", [1, 3])
def test_lookup_teacher_forced(shape, temp, nseq):
    if nseq > 1 and shape.dtype != "bf16":
        pytest.skip("batches need bf16 models")
    k, n_max, max_ctx, steps, seed = 4, 3, 160, 8, 5
    w = workloads.make_weights(shape, seed=1)
    wd = helpers.to_device(w)
    dec = sv.SpecDecoder(shape, wd, shape, wd, k, max_ctx, temperature=temp, seed=seed, batch=nseq,
                         lookup=n_max)
    prompts = _prompt(shape.vocab, 3, nseq)
    dec.prefill(prompts if nseq > 1 else prompts[0])
    T = gen.Model(shape, w)
    tol = helpers.logit_tol(shape)
    ctxs = [list(p) for p in prompts]
    skipped = 0
    for step in range(steps):
        rows, _ = dec.step()
        if nseq == 1:
            rows = [rows]
        p, q, d, _ = dec.last_step_debug(max_ctx)
        if nseq == 1:
            p, q, d = p[None], q[None], d[None]
        for b in range(nseq):
            want = lk.lookup_drafts(ctxs[b], k, n_max)
            assert [int(x) for x in d[b]] == want, (step, b)
            for i in range(k):
                assert q[b, i, want[i]] == 0.0 and np.isneginf(np.delete(q[b, i], want[i])).all()
            ref_p = T.logits(ctxs[b] + want, last=k + 1)
            assert np.abs(p[b] - ref_p).max() < tol
            em, _, fl = gen.verify(p[b], q[b], want, temp, seed, step, row=b, tie_eps=0.0)
            if fl & helpers.SKIP_FLAGS:
                skipped += 1
            else:
                assert em == rows[b], (step, b, em, rows[b])
            ctx = dec.seq_context(b).tolist()
            assert ctx[len(ctxs[b]):] == rows[b]
            ctxs[b] = ctx
    assert skipped <= steps * nseq // 4
    dec.close()


def test_lookup_greedy_equals_plain_decoding():
    k, n_max, max_ctx, n = 5, 3, 160, 40
    w = workloads.make_weights(BF16, seed=2)
    wd = helpers.to_device(w)
    prompt = _prompt(BF16.vocab, 7)[0]
    spec = sv.SpecDecoder(BF16, wd, BF16, wd, k, max_ctx, temperature=0.0, lookup=n_max)
    spec.prefill(prompt)
    out = spec.generate(n)
    spec.close()
    ar = sv.SpecDecoder(BF16, wd, BF16, wd, k, max_ctx, temperature=0.0)
    ar.prefill(prompt)
    ref = [ar.ar_step() for _ in range(n)]
    ar.close()
    assert out == ref
