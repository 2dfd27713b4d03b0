"""Failure paths driven by the library's injection hooks, with no GPU fault:

* A forward kernel whose grid barrier can never complete (one arrival more
  than will come) gives up after a short probe bound, raises the context's
  error flag and leaves; the step reports SPEC_E_TIMEOUT, nothing is
  committed (context, length and step counter unchanged), and the next steps
  equal those of a context that never failed.  The same for plain decoding
  and for a prefill.
* The n-th device allocation of spec_init failing gives SPEC_E_OOM for every
  n and leaves no device memory held.
"""
import pytest

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


def _pair(seed=21):
    shape = workloads.small_shape(dtype="bf16")
    w = workloads.make_weights(shape, seed=seed)
    dshape, _ = workloads.prefix_draft(shape, w, 1)
    wc = helpers.to_device(w)
    dwc = {**wc, "layers": wc["layers"][:1]}
    return shape, wc, dshape, dwc


def test_wait_timeout_commits_nothing():
    shape, wc, dshape, dwc = _pair()
    prompt = workloads.make_prompt(shape.vocab, 24, seed=22)[0].tolist()
    kw = dict(temperature=1.0, seed=3, mix=0.5)
    ref = helpers.decoder(shape, wc, dshape, dwc, 5, 256, **kw)
    ref.prefill(prompt)
    ref_steps = [ref.step()[0] for _ in range(3)]
    ref_ctx = list(ref.seq_context(0))
    ref.close()

    dec = helpers.decoder(shape, wc, dshape, dwc, 5, 256, **kw)
    # a prefill whose forward gives up reports the timeout; a clean one after it works
    dec.inject_fault(sv.SPEC_FAULT_WAIT_TIMEOUT, 4096)
    with pytest.raises(sv.SpecError, match="SPEC_E_TIMEOUT"):
        dec.prefill(prompt)
    dec.inject_fault(sv.SPEC_FAULT_WAIT_TIMEOUT, 0)
    dec.prefill(prompt)
    assert dec.step()[0] == ref_steps[0]
    before = list(dec.seq_context(0))
    steps_before = dec.stats()["steps"]
    dec.inject_fault(sv.SPEC_FAULT_WAIT_TIMEOUT, 4096)
    for _ in range(2):
        with pytest.raises(sv.SpecError, match="SPEC_E_TIMEOUT"):
            dec.step()
        assert list(dec.seq_context(0)) == before
        assert dec.stats()["steps"] == steps_before
    with pytest.raises(sv.SpecError, match="SPEC_E_TIMEOUT"):
        dec.ar_step()
    assert list(dec.seq_context(0)) == before
    dec.inject_fault(sv.SPEC_FAULT_WAIT_TIMEOUT, 0)
    assert dec.step()[0] == ref_steps[1]
    assert dec.step()[0] == ref_steps[2]
    assert list(dec.seq_context(0)) == ref_ctx
    dec.close()


def test_alloc_failure_reports_oom_and_holds_nothing():
    shape, wc, dshape, dwc = _pair(seed=23)
    base = sv.device_bytes_held()
    fired = 0
    for n in range(1, 200):
        sv.inject_alloc_failure(n)
        try:
            dec = helpers.decoder(shape, wc, dshape, dwc, 5, 256)
        except sv.SpecError as e:
            assert "SPEC_E_OOM" in str(e), (n, str(e))
            assert sv.device_bytes_held() == base, n
            fired += 1
            continue
        # n beyond the allocation count: the injection never fired and is cleared
        assert sv.device_bytes_held() > base
        dec.prefill(workloads.make_prompt(shape.vocab, 12, seed=1)[0].tolist())
        assert 1 <= len(dec.step()[0]) <= 6
        dec.close()
        break
    assert fired >= 20, fired
    assert sv.device_bytes_held() == base
