"""The allocation-free acceptance entry point (spec_accept_rows_noalloc).

It serves callers that cannot allocate device memory while they verify
drafts (a serving process whose pool already holds nearly all of HBM, or a
latency-critical loop that must not trigger the device synchronisation an
allocation can cause): its scratch is a fixed 4 MiB array compiled into the
library.  Called through the C ABI, it must return exactly what the
allocating entry point spec_accept_rows returns (tokens, counts and flags
are integer decisions: bit-exact) -- on two calls in a row, so that the
shared array's leftover contents from the first call cannot leak into the
second.  Oversized requests are refused on the host with a clear error.

This file is collected last on purpose: it runs after every other test in a
full run, and also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import speculative_decoding_verification_step_gb300 as sv
import workloads

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _drafts(qc, temp, seed):
    R, K, V = qc.shape
    d = torch.empty(R, K, dtype=torch.int32, device="cuda")
    for i in range(1, K + 1):
        d[:, i - 1] = sv.sample_rows(qc[:, i - 1, :], temp, seed, position=i, row_stride=K * V, rows=R)
    return d


def test_noalloc_matches_allocating_entry_point_twice():
    sv.build()
    L = sv.lib()
    R, K, V = 96, 5, 5000
    stream = torch.cuda.current_stream().cuda_stream
    for call, (sigma, temp, seed) in enumerate([(1.0, 1.0, 3), (0.5, 0.0, 4)]):
        p, q = workloads.make_accept_rows(R, K, V, sigma, seed=seed)
        pc, qc = p.cuda(), q.cuda()
        d = _drafts(qc, temp, seed)
        ref_t, ref_c, ref_f = sv.accept_rows(pc, qc, d, temp, seed)
        tok = torch.full((R, K + 1), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        flg = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        rc = L.spec_accept_rows_noalloc(_p(pc), (K + 1) * V, _p(qc), K * V, _p(d), R, K, V,
                                        float(temp), seed, 0, _p(tok), _p(cnt), _p(flg),
                                        ctypes.c_void_p(stream))
        assert rc == 0, L.spec_last_error(None)
        torch.cuda.synchronize()
        assert torch.equal(cnt, ref_c), call
        assert torch.equal(flg, ref_f), call
        for r in range(R):
            c = int(ref_c[r])
            assert torch.equal(tok[r, :c], ref_t[r, :c]), (call, r)


def test_noalloc_refuses_oversized_requests():
    sv.build()
    L = sv.lib()
    x = torch.zeros(16, device="cuda")
    # 4096 rows of a 128256-token vocabulary need ~22 MB of scratch > 4 MiB
    rc = L.spec_accept_rows_noalloc(_p(x), 0, _p(x), 0, _p(x), 4096, 5, 128256, 1.0, 0, 0,
                                    _p(x), _p(x), None, None)
    assert rc == -1
    msg = L.spec_last_error(None).decode()
    assert "scratch" in msg and str(4 << 20) in msg
