"""Host-side logic of bench.py that needs no GPU: the per-phase fold of the
persistent kernel's timestamps (spec_phase_times / spec_phase_list layouts,
include/specverify.h), the gate on the committed verify-traffic record, and
the reference arm's behaviour on ranks other than 0 and on the 4-bit
workload (which the oracle arm does not run)."""
import json

import pytest

import bench


def _phase(kind, n, k, arrive_min, arrive_max, release, prep, work):
    return {"kind": kind, "n": n, "k": k, "arrive_min_ns": arrive_min, "arrive_max_ns": arrive_max,
            "release_ns": release, "prep_max_ns": prep, "work_max_ns": work}


def test_phase_summary_splits_and_rows():
    # embedding, a SwiGLU GEMM (n = 64 output rows, 8 tiles of 8 gate + 8 up
    # rows), attention, a plain GEMM (n = 32 rows, 2 tiles), the last phase
    # (no release)
    ph = [
        _phase(0, 4, 64, 900, 1000, 1200, -1, -1),
        _phase(1, 64, 128, 2800, 3000, 3500, 1700, 2600),
        _phase(2, 4, 4, 4500, 4800, 5000, 4300, 4600),
        _phase(1, 32, 128, 5900, 6000, -1, 5300, 5800),
    ]
    plist = [(0, 4, 64, 4, 0, 0, 0, 0), (1, 64, 128, 4, 8, 0, 4, 1),
             (2, 4, 2, 4, 4, 0, 0, 128), (1, 32, 128, 4, 2, 0, 4, 1)]
    out = bench.phase_summary(ph, plist)
    assert out["phases"] == 4 and out["total_us"] == 6.0
    g = out["gemm_shapes"]["64x128"]
    # previous release 1200 -> prep end 1700 -> last unit 2600 -> latest arrival 3000 -> release 3500
    assert (g["us"], g["prep_us"], g["stream_us"], g["tail_us"], g["barrier_us"]) == (2.3, 0.5, 0.9, 0.4, 0.5)
    # weight bytes from the tiles: 8 x 16 rows x 128 x 2 B over 2.3 us
    assert g["gbs"] == round(8 * 16 * 128 * 2 / 2300.0, 1)
    last = out["gemm_shapes"]["32x128"]
    assert last["us"] == 1.0 and last["barrier_us"] == 0.0
    assert last["gbs"] == round(2 * 16 * 128 * 2 / 1000.0, 1)
    attn = out["by_kind"]["attn"]
    assert (attn["us"], attn["prep_us"], attn["stream_us"], attn["tail_us"]) == (1.5, 0.8, 0.3, 0.2)
    # without the phase list the SwiGLU GEMM counts its n output rows only
    assert bench.phase_summary(ph)["gemm_shapes"]["64x128"]["gbs"] == round(64 * 128 * 2 / 2300.0, 1)


def test_phase_summary_rejects_mismatched_list():
    ph = [_phase(1, 32, 128, 900, 1000, -1, 300, 800)]
    with pytest.raises(ValueError):
        bench.phase_summary(ph, [])


def test_traffic_record_gated_by_source_hash(monkeypatch):
    rec = json.load(open(bench.os.path.join(bench.ROOT, "profiles", "persist_forward_verify_traffic.json")))
    assert rec["command"].startswith("python bench.py --ncu-mode")
    assert 0.99 < rec["traffic_ratio"] < 1.1
    # used when its hash is the sources' hash, ignored otherwise
    monkeypatch.setattr(bench, "persist_source_hash", lambda: rec["source_sha256_16"])
    assert bench.persist_traffic_record()["traffic_ratio"] == rec["traffic_ratio"]
    monkeypatch.setattr(bench, "persist_source_hash", lambda: "0" * 16)
    assert bench.persist_traffic_record() is None


def _bench(args, env_extra):
    import os
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_without_work():
    # under torchrun only rank 0 times the oracle and prints; the others leave
    r = _bench(["--impl", "reference", "--gpus", "2"], {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_4bit_workload_is_unavailable():
    r = _bench(["--impl", "reference", "--workload", "8b-q4"], {"RANK": "0"})
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line
