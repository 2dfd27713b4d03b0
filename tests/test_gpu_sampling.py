"""GPU parity of the draft sampler and the fused acceptance kernel against the
fp64 oracle, through the C ABI (spec_sample_rows, spec_accept_rows).

Inputs follow the acceptance-kernel workload: target logits ~ N(0, 3^2) at
K+1 positions, draft logits = target rows 1..K + N(0, sigma^2), drafts drawn
from the draft softmax with the Philox draw layout (step = row index).
Token and count decisions must be bit-exact except where the oracle flags a
near-boundary draw (|r - ratio| < 1e-5, or an inverse-CDF target within 1e-6
of a bin edge).  Both sides read the same fp32 logits here, so greedy argmax
decisions are compared with no near-tie window.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads
from oracle import accept as acc
from oracle import generate as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


@pytest.mark.parametrize("V", [256, 5000, 128256])
@pytest.mark.parametrize("temp", [0.0, 1.0, 0.7])
def test_sample_rows(V, temp):
    R = 96
    g = torch.Generator().manual_seed(V)
    logits = torch.randn(R, V, generator=g) * 3.0
    if V == 5000:
        logits[3, 17] = logits[3, 4000] = logits[3].max() + 1.0   # argmax tie -> lowest id
    out = sv.sample_rows(logits.cuda(), temp, seed=7, step_base=11, position=3).cpu().numpy()
    skipped = 0
    for r in range(R):
        tok, fl = gen.draft_token(logits[r].double().numpy(), temp, 7, 11 + r, 3, tie_eps=0.0)
        if fl & helpers.SKIP_FLAGS:
            skipped += 1
            continue
        assert out[r] == tok, (r, out[r], tok)
    assert skipped <= R // 10
    if temp == 0.0 and V == 5000:
        assert out[3] == 17


def _draft_tokens(qc, temp, seed, step_base=0, rows=None, row_stride=None):
    R, K, V = qc.shape if rows is None else (rows, qc.shape[-2], qc.shape[-1])
    d = torch.empty(R, K, dtype=torch.int32, device="cuda")
    for i in range(1, K + 1):
        d[:, i - 1] = sv.sample_rows(qc[:, i - 1, :], temp, seed, step_base=step_base, position=i,
                                     row_stride=K * V if row_stride is None else row_stride, rows=R)
    return d


def _check_rows(p, q, d, tokens, counts, temp, seed, rows):
    skipped = 0
    for r in rows:
        em, n, fl = gen.verify(p[r], q[r], list(d[r]), temp, seed, int(r), tie_eps=0.0)
        c = int(counts[r])
        assert 1 <= c <= q.shape[1] + 1
        if fl & helpers.SKIP_FLAGS:
            skipped += 1
            continue
        assert list(tokens[r][:c]) == em, (r, list(tokens[r][:c]), em)
        assert c == n + 1
    return skipped


@pytest.mark.parametrize("sigma", [0.25, 1.0, 2.0])
@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_accept_rows_small(sigma, temp):
    R, K, V = 128, 5, 5000
    p, q = workloads.make_accept_rows(R, K, V, sigma, seed=3)
    pc, qc = p.cuda(), q.cuda()
    d = _draft_tokens(qc, temp, seed=5)
    tokens, counts, flags = sv.accept_rows(pc, qc, d, temp, seed=5)
    dn = d.cpu().numpy()
    pn, qn = p.double().numpy(), q.double().numpy()
    for r in range(R):   # the drafts themselves match the oracle's sampler
        for i in range(K):
            tok, fl = gen.draft_token(qn[r, i], temp, 5, r, i + 1, tie_eps=0.0)
            if not fl & helpers.SKIP_FLAGS:
                assert dn[r, i] == tok
    skipped = _check_rows(pn, qn, dn, tokens.cpu().numpy(), counts.cpu().numpy(), temp, 5, range(R))
    assert skipped <= R // 10


def test_accept_draft_equals_target():
    R, K, V = 64, 4, 3000
    p, _ = workloads.make_accept_rows(R, K, V, 1.0, seed=9)
    pc = p.cuda()
    qc = pc[:, :K, :].contiguous()
    for temp in (0.0, 1.0):
        d = _draft_tokens(qc, temp, seed=1)
        tokens, counts, flags = sv.accept_rows(pc, qc, d, temp, seed=1)
        assert torch.all(counts == K + 1)
        assert torch.all((flags.cpu() & sv.SPEC_FLAG_ALL_ACCEPTED) != 0)


def test_accept_worked_example():
    """V = 3 rows of the worked example (p = (.5,.3,.2), q = (.8,.1,.1)):
    the first emitted token over many steps follows p."""
    N, K, V = 40000, 1, 3
    p = torch.log(torch.tensor([[0.5, 0.3, 0.2], [0.2, 0.3, 0.5]]))[None].expand(N, 2, 3).contiguous()
    q = torch.log(torch.tensor([[0.8, 0.1, 0.1]]))[None].expand(N, 1, 3).contiguous()
    pc, qc = p.cuda(), q.cuda()
    d = _draft_tokens(qc, 1.0, seed=2)
    tokens, counts, _ = sv.accept_rows(pc, qc, d, 1.0, seed=2)
    first = tokens[:, 0].cpu().numpy()
    freq = np.bincount(first, minlength=3) / N
    assert np.allclose(freq, [0.5, 0.3, 0.2], atol=0.01)
    acc_rate = (counts.cpu().numpy() == 2)[d.cpu().numpy()[:, 0] == 0].mean()
    assert abs(acc_rate - 0.625) < 0.02


@pytest.mark.parametrize("sigma", [0.25, 0.5, 1.0, 2.0])
def test_accept_full_vocab_1024_rows(sigma):
    """Acceptance-kernel workload at full size: 1024 rows, V = 128256, K = 5.
    The oracle checks every row (tokens and counts exact except flagged
    near-boundary draws); every count is in 1..K+1."""
    R, K, V = 1024, 5, 128256
    pc, qc = workloads.make_accept_rows(R, K, V, sigma, seed=int(sigma * 100), device="cuda")
    d = _draft_tokens(qc, 1.0, seed=11)
    tokens, counts, flags = sv.accept_rows(pc, qc, d, 1.0, seed=11)
    torch.cuda.synchronize()
    cn = counts.cpu().numpy()
    assert cn.min() >= 1 and cn.max() <= K + 1
    ds, ts = d.cpu().numpy(), tokens.cpu().numpy()
    skipped = 0
    for c0 in range(0, R, 64):   # host copies in chunks of 64 rows
        ps = pc[c0:c0 + 64].cpu().numpy()
        qs = qc[c0:c0 + 64].cpu().numpy()
        for j in range(ps.shape[0]):
            r = c0 + j
            em, n, fl = gen.verify(ps[j], qs[j], list(ds[r]), 1.0, 11, r, tie_eps=0.0)
            if fl & helpers.SKIP_FLAGS:
                skipped += 1
                continue
            assert int(cn[r]) == n + 1, (r, int(cn[r]), n)
            assert list(ts[r][:cn[r]]) == em, r
    assert skipped <= R // 8   # flagged near-edge residual draws (~5% of rows at V = 128256)
    alpha = (cn - 1).sum() / (cn - 1 + (cn <= K)).sum()
    print(f"sigma={sigma}: per-draft acceptance {alpha:.3f}, mean tokens/step {cn.mean():.3f}")


def test_chi_square_first_token():
    """10^5 T=1 steps on one fixed row (V = 128256, K = 5, sigma = 1): the
    first emitted token follows the target p_1 (chi-square over 100
    equal-mass bins must not reject at 1%)."""
    K, V, N, half = 5, 128256, 100_000, 50_000
    p, q = workloads.make_accept_rows(1, K, V, 1.0, seed=21)
    pc, qc = p.cuda(), q.cuda()
    firsts = []
    for base in (0, half):
        d = _draft_tokens(qc, 1.0, seed=4, step_base=base, rows=half, row_stride=0)
        tokens, counts, _ = sv.accept_rows(pc, qc, d, 1.0, seed=4, step_base=base, rows=half,
                                           p_row_stride=0, q_row_stride=0)
        firsts.append(tokens[:, 0].cpu().numpy())
    first = np.concatenate(firsts)
    p1 = acc.softmax_t(p[0, 0].double().numpy(), 1.0)
    bins = helpers.equal_mass_bins(p1, 100)
    nb = bins.max() + 1
    obs = np.bincount(bins[first], minlength=nb)
    exp = np.bincount(bins, weights=p1, minlength=nb) * N
    assert exp.min() >= 5
    chi = stats.chisquare(obs, exp * obs.sum() / exp.sum())
    assert chi.pvalue > 0.01, chi


def test_chi_square_tiny_vocab():
    """Same at V = 256 with one bin per token (tiny workload's vocabulary)."""
    K, V, N = 4, 256, 60_000
    g = torch.Generator().manual_seed(5)
    p = torch.randn(1, K + 1, V, generator=g) * 0.5
    q = p[:, :K] + torch.randn(1, K, V, generator=g) * 0.5
    pc, qc = p.cuda(), q.contiguous().cuda()
    d = _draft_tokens(qc, 1.0, seed=8, rows=N, row_stride=0)
    tokens, _, _ = sv.accept_rows(pc, qc, d, 1.0, seed=8, rows=N, p_row_stride=0, q_row_stride=0)
    first = tokens[:, 0].cpu().numpy()
    p1 = acc.softmax_t(p[0, 0].double().numpy(), 1.0)
    obs = np.bincount(first, minlength=V)
    chi = stats.chisquare(obs, p1 * N)
    assert chi.pvalue > 0.01, chi
