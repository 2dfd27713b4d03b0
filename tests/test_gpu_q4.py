"""4-bit group-quantized weight streaming (SPEC_DTYPE_Q4) against the oracle.

The pages' measurements run 4-bit models ("Speculative decoding internals",
section "怎麼測自己的加速倍率": Q4_K_M targets).  The method is exact with
respect to the model that verifies, here the quantized target: the oracle
runs its fp64 forward on the dequantized weights (oracle.quant: scale x code,
exact), the GPU streams the packed codes and scales and computes each 64-k
group's code . X sum on the tensor cores before weighting it by the scale.

* Small 4-bit pair (d 512, GQA 4:1, head dim 64, FFN 1024, vocabulary 1024):
  teacher-forced steps at T in {0, 1}, lambda in {0, 0.5}, K = 5 -- logits
  within 2e-2 of the fp64 oracle, drafts and emitted tokens exact except
  flagged draws; plain decoding the same; greedy speculative output equal to
  greedy plain decoding; a draft equal to the target accepts every draft.
* The 8B / 1B widths, 4-bit, one layer each (vocabulary 128256): the q/k/v,
  o, gate/up and LM-head phases with their input rows resident in shared
  memory and the 6-token, 14336-wide down-projection with its input rows
  streamed beside the codes; teacher-forced at T = 1 with the full-width
  tolerance (2e-2 plus the oracle's own bf16-dataflow-vs-fp64 gap, see
  test_gpu_fullwidth.py).
* Argument checks: 4-bit models need batch 1, the persistent kernel and
  prompts of at least 10 tokens.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads
from oracle import generate as gen
from oracle import quant

pytestmark = pytest.mark.gpu

MATS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
Q4S = workloads.small_shape(name="q4small", dtype="q4", d_model=512, n_heads=8, n_kv_heads=2, head_dim=64,
                            ffn_dim=1024, vocab=1024)
K = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


def dense(shape, w):
    """The oracle's copy of 4-bit weights: every matrix dequantized by
    oracle.quant to fp64 [n][k]; the embedding and the gains as given."""
    def mat(name, buf):
        n, k = workloads.matrix_dims(shape, name)
        packed, scales = workloads.q4_parts(buf, n, k)
        return torch.from_numpy(quant.dequantize_q4(packed.numpy(), scales.double().numpy()))

    return {"embed": w["embed"].cpu(), "final_norm": w["final_norm"].cpu().double(),
            "lm_head": mat("lm_head", w["lm_head"]),
            "layers": [{k: (mat(k, v) if k in MATS else v.cpu().double()) for k, v in lw.items()}
                       for lw in w["layers"]]}


@pytest.fixture(scope="module")
def small():
    w = workloads.make_q4_weights(Q4S, seed=41, device="cuda")
    dshape, dw = workloads.prefix_draft(Q4S, w, 1)
    wd = dense(Q4S, w)
    dd = {**wd, "layers": wd["layers"][:1]}
    return w, dshape, dw, gen.Model(Q4S, wd), gen.Model(dshape, dd)


@pytest.mark.parametrize("temp,mix", [(0.0, 0.0), (1.0, 0.0), (0.0, 0.5), (1.0, 0.5)])
def test_q4_teacher_forced(small, temp, mix):
    w, dshape, dw, T, D = small
    prompt = workloads.make_prompt(Q4S.vocab, 40, seed=42)[0].tolist()
    dec = sv.SpecDecoder(Q4S, w, dshape, dw, K, 256, temperature=temp, seed=9, mix_lambda=mix)
    try:
        _, steps, skipped, worst = helpers.teacher_forced(dec, T, D, prompt, K, temp, 30, 2e-2, mix=mix, seed=9,
                                                          max_ctx=256)
        assert skipped <= max(1, steps // 4)
        print(f"q4 T={temp} lambda={mix}: {steps} steps, largest logit error {worst[0]:.4f}")
    finally:
        dec.close()


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_q4_plain_decoding(small, temp):
    w, dshape, dw, T, _ = small
    prompt = workloads.make_prompt(Q4S.vocab, 24, seed=43)[0].tolist()
    dec = sv.SpecDecoder(Q4S, w, dshape, dw, K, 256, temperature=temp, seed=10)
    try:
        dec.prefill(prompt)
        ctx, skipped = list(prompt), 0
        for s in range(12):
            tok = dec.ar_step()
            p, _, _, context = dec.last_step_debug(256)
            ref = T.logits(ctx, last=1)[0]
            assert np.abs(p[0] - ref).max() < 2e-2, s
            exp, fl = gen.ar_token_flagged(p[0], temp, 10, s, tie_eps=0.0)
            if fl & helpers.SKIP_FLAGS:
                skipped += 1
            else:
                assert exp == tok, (s, exp, tok)
            assert [int(t) for t in context] == ctx + [tok]
            ctx.append(tok)
        assert skipped <= 2
    finally:
        dec.close()


def test_q4_greedy_spec_equals_greedy_ar(small):
    w, dshape, dw, _, _ = small
    prompt = workloads.make_prompt(Q4S.vocab, 30, seed=44)[0].tolist()
    dec = sv.SpecDecoder(Q4S, w, dshape, dw, K, 256)
    try:
        dec.prefill(prompt)
        spec = dec.generate(48)
        dec.prefill(prompt)
        ar = [dec.ar_step() for _ in range(48)]
        assert spec == ar
    finally:
        dec.close()


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_q4_draft_equal_target_accepts_all(small, temp):
    w, _, _, _, _ = small
    dec = sv.SpecDecoder(Q4S, w, Q4S, w, K, 256, temperature=temp, seed=3)
    try:
        dec.prefill(workloads.make_prompt(Q4S.vocab, 20, seed=1)[0].tolist())
        for _ in range(6):
            toks, flags = dec.step()
            assert len(toks) == K + 1 and flags & sv.SPEC_FLAG_ALL_ACCEPTED
    finally:
        dec.close()


def test_q4_full_width_teacher_forced():
    """8B-width 4-bit target (2 layers, vocabulary 128256) with a 1B-width
    4-bit draft (1 layer): every phase kind of the 4-bit benchmark pair.  The
    prefill chunks of 8 positions stream their RMSNorm'd 4096-wide inputs
    (they do not fit the X region sized for K + 1 rows); the second layer
    makes their 1/rms matter (every first-layer input is an embedding row of
    nearly the same rms), and every step's K + 1 target rows are compared
    with the oracle on the GPU's own drafts, whether or not the drafts agree."""
    W8 = replace(workloads.EIGHT_B, n_layers=2, dtype="q4")
    W1 = replace(workloads.ONE_B, n_layers=1, dtype="q4")
    tw = workloads.make_q4_weights(W8, seed=45, device="cuda")
    dw = workloads.make_q4_weights(W1, seed=46, device="cuda")
    t64, d64 = dense(W8, tw), dense(W1, dw)
    T, Tb = gen.Model(W8, t64), gen.Model(W8, t64, act="bf16")
    D, Db = gen.Model(W1, d64), gen.Model(W1, d64, act="bf16")
    prompt = workloads.make_prompt(W8.vocab, 24, seed=47)[0].tolist()
    dec = sv.SpecDecoder(W8, tw, W1, dw, K, 128, temperature=1.0, seed=11)
    try:
        lists = dec.phase_list(K)
        gemm = {p[1:3]: p for p in lists if p[0] == 1}
        assert gemm[(4096, 14336)][7] == 0 and gemm[(6144, 4096)][7] == 1   # streamed / resident input rows

        def target_rows(step, ctx, p, q, d, ref):
            seq = ctx + [int(t) for t in d]
            want = T.logits(seq, last=K + 1)
            allow = 2e-2 + np.abs(Tb.logits(seq, last=K + 1) - want).max()
            err = np.abs(p - want).max()
            assert err < allow, (step, err, allow)

        _, steps, skipped, worst = helpers.teacher_forced(dec, T, D, prompt, K, 1.0, 10, 2e-2, seed=11,
                                                          max_ctx=128, alt=(Tb, Db), extra=target_rows)
        assert skipped <= max(1, steps // 3)
        print(f"q4 full width: {steps} steps, largest logit error {worst[0]:.4f} (allowed {worst[1]:.4f})")
    finally:
        dec.close()


def test_q4_argument_checks(small):
    w, dshape, dw, _, _ = small
    with pytest.raises(sv.SpecError, match="SPEC_E_ARG"):
        sv.SpecDecoder(Q4S, w, dshape, dw, K, 256, batch=2)
    with pytest.raises(sv.SpecError, match="SPEC_E_ARG"):
        sv.SpecDecoder(Q4S, w, dshape, dw, K, 256, flags=sv.SPEC_OPT_NO_PERSIST)
    with pytest.raises(sv.SpecError, match="SPEC_E_ARG"):
        sv.SpecDecoder(Q4S, w, dshape, dw, 8, 256)
    dec = sv.SpecDecoder(Q4S, w, dshape, dw, K, 256)
    try:
        with pytest.raises(sv.SpecError, match="SPEC_E_ARG"):
            dec.prefill(list(range(8)))
        full = torch.empty(4, Q4S.vocab, device="cuda")
        with pytest.raises(sv.SpecError, match="SPEC_E_STATE"):
            dec.model_forward(0, [1, 2, 3, 4], 0, full)
    finally:
        dec.close()
