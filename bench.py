#!/usr/bin/env python3
"""Speculative-decoding verification step on GB300: accepted tokens/s at batch
1, K = 5, with an 8B-shaped bf16 target and a 1B-shaped bf16 draft (random
N(0, 0.02^2) weights, 512-token uniform-random prompts, 128 new tokens per
generation), plus verify-step HBM GB/s.

One "step" is one speculative step: K draft passes + samplers, one target
pass over the K+1 positions, the fused acceptance kernel and the commit.
The timed region runs whole generations (prompt -> 128 tokens) back to back;
each generation's prefill happens outside the timed region, with inputs
already resident.  Every step streams ~17.5 GB of weights, far larger than
the 129 MB L2, so no L2 flush is needed between steps.

--gpus N (torchrun) runs N independent replicas, one per GPU (the step does
not shard at batch 1): value = tokens of all ranks / max time over ranks.
--impl reference times the fp64 CPU oracle on this host instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("accepted tokens/s at batch 1, K=5 (8B-shaped bf16); verify-step HBM GB/s")
HBM_ROOFLINE_GBS = 8000.0          # the figure the step's roofline target is stated against


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=240)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--k", type=int, default=5)
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--mix", type=float, default=0.5, help="draft/target-previous-logit mix lambda")
    ap.add_argument("--prompt", type=int, default=512)
    ap.add_argument("--new-tokens", type=int, default=128)
    ap.add_argument("--workload", choices=["8b", "1b", "8b-q4"], default="8b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--ar-tokens", type=int, default=128)
    ap.add_argument("--ncu-mode", action="store_true",
                    help="profiling run: prefill, --warmup steps, then --steps steps inside "
                         "cudaProfilerStart/Stop, nothing else")
    ap.add_argument("--pdl", action="store_true", help="launch with programmatic dependent launch")
    ap.add_argument("--phase-times", action="store_true",
                    help="profiling: per-phase breakdown of the persistent verify, plain-decoding "
                         "and draft passes (globaltimer stamps)")
    ap.add_argument("--no-persist", action="store_true",
                    help="one kernel per phase instead of the persistent forward kernel")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: keep the first N layers of both models")
    ap.add_argument("--accept-bench", action="store_true",
                    help="acceptance-kernel microbench: 1024 verify rows, V 128256, K 5, draft noise "
                         "sigma in {0.25, 0.5, 1, 2} (one JSON line each)")
    ap.add_argument("--verify-sweep", action="store_true",
                    help="verify step alone over batch x K x context (one JSON line each): "
                         "latency, algorithmic bytes, GB/s, tensor FLOP/s")
    ap.add_argument("--k-sweep", action="store_true",
                    help="speculative vs plain decoding at batch 1 for K = 1..8 (one JSON line each): "
                         "tokens/s, speedup, tokens per step, acceptance, C and the modelled K a / (1 + K C)")
    ap.add_argument("--profile-batch", default="",
                    help="profiling: B,K,CONTEXT -- one batched speculative step launched kernel by kernel "
                         "(synthetic state) between cudaProfilerStart/Stop, after two unprofiled steps")
    ap.add_argument("--sweep-batches", default="1",
                    help="comma-separated batch sizes of --verify-sweep (batch > 1: synthetic KV)")
    ap.add_argument("--sweep-ks", default="1,2,3,4,5,6,8", help="comma-separated K of --verify-sweep")
    ap.add_argument("--sweep-contexts", default="512,4096,16384",
                    help="comma-separated contexts of --verify-sweep")
    return ap.parse_args()


def workload_shapes(name):
    import workloads
    from dataclasses import replace
    if name == "8b":
        return workloads.EIGHT_B, workloads.ONE_B, "8B-shaped target + 1B-shaped draft"
    if name == "8b-q4":
        return (replace(workloads.EIGHT_B, dtype="q4"), replace(workloads.ONE_B, dtype="q4"),
                "8B-shaped 4-bit target + 1B-shaped 4-bit draft")
    return workloads.ONE_B, None, "1B-shaped target + its first 2 layers as draft"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tflops_peak():
    """Dense bf16 tensor FLOP/s of a kernel timed alone (MEASURED_PEAKS.json
    burst figure, else the fallback), in TFLOP/s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.idx)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                mhz.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


PERSIST_SOURCES = ("persist.cu", "tma_dev.cuh", "dattn_dev.cuh", "gemm_dev.cuh", "embed_dev.cuh",
                   "common.cuh", "kernels.h")


def persist_source_hash():
    h = hashlib.sha256()
    for f in PERSIST_SOURCES:
        h.update(open(os.path.join(ROOT, "speculative_decoding_verification_step_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def persist_traffic_record():
    """DRAM traffic of the persistent verify forward from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "persist_forward_verify_traffic.json")
    try:
        rec = json.load(open(path))
        return rec if rec.get("source_sha256_16") == persist_source_hash() else None
    except Exception:
        return None


# ----------------------------------------------------------------------------- oracle
def truncated(shape, w, layers):
    """The first `layers` decoder layers of a model (same width and vocabulary)."""
    from dataclasses import replace
    return replace(shape, n_layers=layers), dict(w, layers=w["layers"][:layers])


def oracle_steps(tshape, tw, dshape, dw, k, temperature, mix, prompt_len, budget_s, max_steps, seed=0):
    """The fp64 oracle's speculative steps, run for real at full depth, width
    and vocabulary on prompts of prompt_len tokens: steps continue until
    max_steps or until budget_s seconds have been spent (at least one step).
    Each step starts from a fresh prompt (the oracle recomputes every position
    anyway).  Returns (tokens, seconds, steps, threads)."""
    import torch
    import workloads
    from oracle import generate as gen

    T, D = gen.Model(tshape, tw), gen.Model(dshape, dw)
    toks, secs, n = 0, 0.0, 0
    while n < max_steps and (n == 0 or secs < budget_s):
        prompt = workloads.make_prompt(tshape.vocab, prompt_len, seed=seed + n)[0].tolist()
        t0 = time.perf_counter()
        prev = gen.prefill_prev_logits(T, prompt, k) if mix else None
        res = gen.spec_step(T, D, prompt, k, temperature, 0, n, prev, mix)
        secs += time.perf_counter() - t0
        toks += len(res.emitted)
        n += 1
    return toks, secs, n, torch.get_num_threads()


def host_weights(shape, seed, layers=None):
    """Seeded weights of a model (only its first `layers` decoder layers when
    given), drawn on the GPU when there is one and copied to host."""
    import torch
    import workloads
    from dataclasses import replace
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if layers is not None:
        shape = replace(shape, n_layers=min(layers, shape.n_layers))
    w = workloads.make_weights(shape, seed, device=dev)
    if dev == "cuda":
        w = to_host(w)
        torch.cuda.empty_cache()
    return w


def to_host(w):
    return {k: ([{kk: vv.cpu() for kk, vv in l.items()} for l in v] if k == "layers" else v.cpu())
            for k, v in w.items()}


def run_reference(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    tshape, dshape, wl = workload_shapes(args.workload)
    if tshape.dtype == "q4":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm runs the bf16 workloads only"}))
        return 0
    tw = host_weights(tshape, 1)
    if dshape is None:
        import workloads
        dshape, dw = workloads.prefix_draft(tshape, tw, 2)
    else:
        dw = host_weights(dshape, 2)
    # warm-up: one step (not timed); then up to --steps real steps within ~150 s
    oracle_steps(tshape, tw, dshape, dw, args.k, args.temperature, args.mix, args.prompt, 0.0, 1, seed=500)
    toks, secs, n, threads = oracle_steps(tshape, tw, dshape, dw, args.k, args.temperature, args.mix,
                                          args.prompt, 150.0, args.steps, seed=100)
    v = toks / secs
    sample = (f"{n} complete fp64 oracle speculative steps ({wl}, full depth, K={args.k}, "
              f"T={args.temperature}, lambda={args.mix}, {args.prompt}-token prompts, every position "
              f"recomputed) after 1 untimed step; {toks} tokens in {secs:.1f} s measured")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": n, "steps_requested": args.steps, "warmup": 1,
            "ms_per_step": 1000 * secs / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl, "K": args.k, "temperature": args.temperature,
                       "mix_lambda": args.mix, "prompt": args.prompt, "batch": 1},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- ours
def phase_summary(ph, plist=None):
    """Fold per-phase stamps of one persistent pass.  Per phase: total time
    from the previous release to this one, split into prep (release -> latest
    end of X preparation; attention: latest end of a key walk), stream (->
    latest delivery of a CTA's last weight unit; attention: end of the items,
    i.e. the merges), tail (-> latest arrival: reductions and epilogues) and
    barrier (latest arrival -> release).  Summed per phase kind
    and per GEMM shape (with its weight GB/s over the whole phase, 2 B per
    weight).  plist: the pass's phase list (spec_phase_list), whose 16-row
    tiles give the weight rows a GEMM streams (a SwiGLU tile is 8 gate + 8 up
    rows of its n output rows: 2n rows); without it, n rows."""
    kinds = {0: "embed", 1: "gemm", 2: "attn"}
    out = {"phases": len(ph), "total_us": 0.0, "by_kind": {}, "gemm_shapes": {}}
    if plist is not None and len(plist) != len(ph):
        raise ValueError("phase list and phase times differ in length")
    rows_of = {}
    prev = 0
    for i, p in enumerate(ph):
        end = p["release_ns"] if p["release_ns"] >= 0 else p["arrive_max_ns"]
        prep_end = p["prep_max_ns"] if p["prep_max_ns"] >= 0 else prev
        work_end = p["work_max_ns"] if p["work_max_ns"] >= 0 else prep_end
        parts = {"us": (end - prev) / 1e3, "prep_us": (prep_end - prev) / 1e3,
                 "stream_us": (work_end - prep_end) / 1e3, "tail_us": (p["arrive_max_ns"] - work_end) / 1e3,
                 "barrier_us": ((p["release_ns"] - p["arrive_max_ns"]) / 1e3) if p["release_ns"] >= 0 else 0.0}
        k = kinds.get(p["kind"], str(p["kind"]))
        agg = out["by_kind"].setdefault(k, {"count": 0})
        agg["count"] += 1
        for f, v in parts.items():
            agg[f] = agg.get(f, 0.0) + v
        if p["kind"] == 1:
            key = f'{p["n"]}x{p["k"]}'
            rows_of[key] = plist[i][4] * 16 if plist is not None else p["n"]
            g = out["gemm_shapes"].setdefault(key, {"count": 0})
            g["count"] += 1
            for f, v in parts.items():
                g[f] = g.get(f, 0.0) + v
        prev = end
    out["total_us"] = round(prev / 1e3, 1)
    for key, g in out["gemm_shapes"].items():
        k = int(key.split("x")[1])
        g["gbs"] = round(g["count"] * rows_of[key] * k * 2 / (g["us"] * 1e3), 1)
    for table in (out["by_kind"], out["gemm_shapes"]):
        for agg in table.values():
            for f in list(agg):
                if f.endswith("_us") or f == "us":
                    agg[f] = round(agg[f] / agg["count"], 2)   # per phase
    return out


def combine_ranks(ms, toks, world, device):
    """Whole-job inputs of the throughput across replicas: the slowest rank's
    timed milliseconds (all_reduce MAX) and the tokens of all ranks (SUM)."""
    if world <= 1:
        return ms, float(toks)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, toks], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(t[1])


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist
    import workloads
    import speculative_decoding_verification_step_gb300 as sv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sv.build()
    sv.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    tshape, dshape, wl = workload_shapes(args.workload)
    if args.layers:
        from dataclasses import replace
        tshape = replace(tshape, n_layers=min(args.layers, tshape.n_layers))
        dshape = replace(dshape, n_layers=min(args.layers, dshape.n_layers)) if dshape else None
        wl += f" (first {args.layers} layers, profiling only)"
    K = args.k
    q4 = tshape.dtype == "q4"
    mk = workloads.make_q4_weights if q4 else workloads.make_weights
    tw = mk(tshape, 1, device="cuda")
    if dshape is None:
        dshape, dw = workloads.prefix_draft(tshape, tw, 2)
    else:
        dw = mk(dshape, 2, device="cuda")
    torch.cuda.synchronize()
    max_ctx = args.prompt + args.new_tokens + 4 * (K + 1) + 64
    stream = torch.cuda.Stream()

    base_flags = (sv.SPEC_OPT_PDL if args.pdl else 0) | (sv.SPEC_OPT_NO_PERSIST if args.no_persist else 0)

    def make(temp, mix, flags=0, lookup=0):
        return sv.SpecDecoder(tshape, tw, dshape, dw, K, max_ctx, temperature=temp, seed=0,
                              mix_lambda=mix, stream=stream.cuda_stream, flags=flags | base_flags,
                              lookup=lookup)

    def prompt(i):
        return workloads.make_prompt(tshape.vocab, args.prompt, seed=1000 * rank + i)[0].tolist()

    def repeat_prompt(i):
        """A 128-token uniform block repeated to the prompt length (prompt lookup finds matches)."""
        blk = workloads.make_prompt(tshape.vocab, 128, seed=1000 * rank + i)[0].tolist()
        return (blk * (args.prompt // 128 + 1))[:args.prompt]

    hist_acc = {}

    def timed_generations(dec, n_steps, gen_base, prompt_fn=None):
        """Run n_steps speculative steps as whole generations; returns (ms,
        tokens, steps).  The histogram of accepted drafts over all of them is
        left in hist_acc[id(dec)] (each prefill resets the context's own)."""
        ms, toks, done, g = 0.0, 0, 0, gen_base
        hist = [0] * 17
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        while done < n_steps:
            dec.prefill((prompt_fn or prompt)(g))
            g += 1
            emitted = 0
            e0.record(stream)
            while emitted < args.new_tokens and done < n_steps:
                t, _ = dec.step()
                emitted += len(t)
                done += 1
            e1.record(stream)
            e1.synchronize()
            ms += e0.elapsed_time(e1)
            toks += emitted
            hist = [x + y for x, y in zip(hist, dec.stats()["accept_hist"])]
        hist_acc[id(dec)] = hist
        return ms, toks, done

    if args.accept_bench:
        # the fused acceptance kernel alone over independent verify rows:
        # target logits N(0, 3^2), draft logits = target rows 1..K + N(0,
        # sigma^2), drafts drawn from the draft softmax (Philox stream 0 at
        # step = row index); inputs resident on the device, 5.78 GB > L2
        peak, peak_kind = peaks()
        R, KA, VA = 1024, 5, 128256
        for sigma in (0.25, 0.5, 1.0, 2.0):
            p, q = workloads.make_accept_rows(R, KA, VA, sigma, seed=7, device="cuda")
            drafts = torch.empty(R, KA, dtype=torch.int32, device="cuda")
            for i in range(KA):
                drafts[:, i] = sv.sample_rows(q[:, i, :], 1.0, 11, step_base=0, position=i + 1,
                                              row_stride=KA * VA, rows=R)
            for _ in range(3):
                sv.accept_rows(p, q, drafts, 1.0, 11)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = 10
            e0.record()
            for _ in range(n):
                toks, counts, flags = sv.accept_rows(p, q, drafts, 1.0, 11)
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1) / n
            nbytes = R * (2 * KA + 1) * VA * 4
            acc_mean = float(counts.float().mean()) - 1.0
            print(json.dumps({"accept_bench": True, "rows": R, "K": KA, "V": VA, "sigma": sigma,
                              "ms": ms, "bytes": nbytes, "GB_s": nbytes / (ms * 1e6),
                              "frac_of_measured": nbytes / (ms * 1e6) / peak, "peak_kind": peak_kind,
                              "rows_per_s": R / (ms * 1e-3), "accepted_per_row": acc_mean,
                              "acceptance_alpha_approx": acc_mean / KA}), flush=True)
            del p, q, drafts
            torch.cuda.empty_cache()
        return 0

    if args.verify_sweep:
        # the verify step (target over K+1 positions per sequence + fused
        # acceptance) replayed as a graph, after a prefill of `context`
        # uniform-random ids (batch 1) or a synthetic state of `context`
        # positions (batch > 1: random ids, KV caches filled with N(0, 1)
        # values -- the same bytes read, not the models' own keys and values)
        peak, peak_kind = peaks()
        tf_peak = tflops_peak()
        kv_tok = tshape.kv_bytes_per_token() + dshape.kv_bytes_per_token()
        for batch in [int(x) for x in args.sweep_batches.split(",")]:
            for ctx in [int(x) for x in args.sweep_contexts.split(",")]:
                prm = workloads.make_prompt(tshape.vocab, ctx, seed=77)[0].tolist()
                for k in [int(x) for x in args.sweep_ks.split(",")]:
                    cap = ctx + 2 * (k + 1) + 64
                    need = batch * cap * kv_tok * 1.05 + 2e9
                    free = torch.cuda.mem_get_info()[0]
                    line = {"verify_sweep": True, "workload": wl, "batch": batch, "K": k, "context": ctx}
                    if need > free:
                        line["skipped"] = f"KV caches need {need / 1e9:.0f} GB, {free / 1e9:.0f} GB free"
                        print(json.dumps(line), flush=True)
                        continue
                    d = sv.SpecDecoder(tshape, tw, dshape, dw, k, cap, temperature=args.temperature,
                                       seed=0, mix_lambda=0.0, stream=stream.cuda_stream, batch=batch)
                    if batch == 1:
                        d.prefill(prm)
                    else:
                        d.prefill_synthetic(ctx, seed=77)
                    prof = d.profile(iters=10 if batch == 1 else 3)
                    st = d.stats()
                    L = ctx - 1                      # committed positions before the pending token
                    nbytes = (st["verify_weight_bytes"] + batch * (L + k + 1) * st["kv_bytes_per_token_target"]
                              + batch * (k + 1) * tshape.vocab * 4)
                    sec = prof["verify_ms"] * 1e-3
                    gbs = nbytes / sec / 1e9
                    # dense GEMM flops: 2 x (weight elements) x verify rows
                    tfl = 2.0 * st["verify_weight_bytes"] / 2 * batch * (k + 1) / sec / 1e12
                    line.update({"kv": "prefill" if batch == 1 else "synthetic N(0,1)",
                                 "verify_step_ms": prof["verify_ms"],
                                 "target_forward_ms": prof["verify_forward_ms"],
                                 "positions_per_s": batch * (k + 1) / sec,
                                 "bytes": nbytes, "GB_s": gbs, "frac_of_measured": gbs / peak,
                                 "peak_kind": peak_kind, "gemm_TFLOP_s": tfl, "frac_of_bf16_peak": tfl / tf_peak,
                                 "kernels_per_verify": prof["kernels_verify"],
                                 "persistent": prof["kernels_verify"] <= 2})
                    print(json.dumps(line), flush=True)
                    d.close()
                    torch.cuda.synchronize()
        return 0

    if args.phase_times:
        dec = make(args.temperature, args.mix, sv.SPEC_OPT_PHASE_TIMES)
        dec.prefill(prompt(0))
        for _ in range(max(args.warmup, 3)):
            dec.step()
        dec.profile(3)   # runs the verify-only and plain-decoding passes too
        print(json.dumps({"phase_times": True, "workload": wl,
                          "passes": {name: phase_summary(dec.phase_times(i), dec.phase_list(i))
                                     for name, i in (("draft_1", 0), ("draft_2", 1), ("verify", K),
                                                     ("ar", K + 1))}}), flush=True)
        return 0

    if args.k_sweep:
        # plain decoding once (its pass does not depend on K), then per K:
        # whole generations as in the headline run, and the graph-replayed
        # phase times for C
        ar = make(args.temperature, 0.0)
        ar.prefill(prompt(0))
        for _ in range(3):
            ar.ar_step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ar.prefill(prompt(1))
        e0.record(stream)
        for _ in range(args.ar_tokens):
            ar.ar_step()
        e1.record(stream)
        e1.synchronize()
        ar_tok_s = args.ar_tokens / (e0.elapsed_time(e1) / 1000.0)
        ar.close()
        for k in (1, 2, 3, 4, 5, 6, 8):
            d = sv.SpecDecoder(tshape, tw, dshape, dw, k, args.prompt + args.new_tokens + 4 * (k + 1) + 64,
                               temperature=args.temperature, seed=0, mix_lambda=args.mix,
                               stream=stream.cuda_stream, flags=base_flags)
            d.prefill(prompt(0))
            d.step()
            ms, toks, nsteps = timed_generations(d, 90, 400)
            hist = hist_acc[id(d)][:k + 1]
            acc_n = sum(i * h for i, h in enumerate(hist))
            alpha = acc_n / max(1, acc_n + sum(hist[:k]))
            d.prefill(prompt(0))
            prof = d.profile(iters=10)
            c_ratio = prof["draft_loop_ms"] / max(1e-9, k * prof["verify_ms"])
            tok_s = toks / (ms / 1000.0)
            print(json.dumps({"k_sweep": True, "workload": wl, "K": k, "temperature": args.temperature,
                              "mix_lambda": args.mix, "tokens_per_s": tok_s, "ar_tokens_per_s": ar_tok_s,
                              "speedup_vs_ar": tok_s / ar_tok_s, "tokens_per_step": toks / nsteps,
                              "acceptance_alpha": alpha,
                              "expected_tokens_per_step": (1 - alpha ** (k + 1)) / (1 - alpha) if alpha < 1 else k + 1,
                              "verify_ms": prof["verify_ms"], "draft_loop_ms": prof["draft_loop_ms"],
                              "C": c_ratio, "K_alpha_over_1_plus_KC": k * alpha / (1 + k * c_ratio),
                              "expected_tokens_over_1_plus_KC": ((1 - alpha ** (k + 1)) / (1 - alpha) if alpha < 1
                                                                 else k + 1) / (1 + k * c_ratio),
                              "persistent": prof["kernels_verify"] <= 2}), flush=True)
            d.close()
        return 0

    if args.profile_batch:
        pb, pk, pctx = [int(x) for x in args.profile_batch.split(",")]
        d = sv.SpecDecoder(tshape, tw, dshape, dw, pk, pctx + 2 * (pk + 1) + 64, temperature=args.temperature,
                           seed=0, mix_lambda=0.0, stream=stream.cuda_stream, flags=sv.SPEC_OPT_NO_GRAPH,
                           batch=pb)
        d.prefill_synthetic(pctx, seed=3)
        d.step()
        d.step()
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        d.step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        print(json.dumps({"profile_batch": True, "batch": pb, "K": pk, "context": pctx, "workload": wl,
                          "kernels_per_step": d.stats()["kernels_per_step"]}), flush=True)
        d.close()
        return 0

    if args.ncu_mode:
        dec = make(args.temperature, args.mix)
        dec.prefill(prompt(0))
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            dec.step()
        torch.cuda.synchronize()
        warm_tokens = dec.stats()["tokens_emitted"]
        torch.cuda.profiler.start()
        for _ in range(args.steps):
            dec.step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        st = dec.stats()
        # algorithmic bytes of the first profiled verify forward (context: prompt + warm-up tokens)
        L0 = args.prompt - 1 + warm_tokens
        vb = st["verify_weight_bytes"] + (L0 + K + 1) * st["kv_bytes_per_token_target"] + (K + 1) * tshape.vocab * 4
        print(json.dumps({"ncu_mode": True, "kernels_per_step": st["kernels_per_step"], "steps": st["steps"],
                          "workload": wl, "verify_forward_bytes_approx": vb}), flush=True)
        return 0

    # ---- headline run ----
    dec = make(args.temperature, args.mix)
    dec.prefill(prompt(0))
    for _ in range(args.warmup):
        dec.step()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        ms, toks, nsteps = timed_generations(dec, args.steps, 1)
        wall = time.perf_counter() - wall0
    clocks = clk.summary()
    st = dec.stats()
    ms_max, toks_all = combine_ranks(ms, toks, world, "cuda")
    value = toks_all / (ms_max / 1000.0)
    hist = hist_acc[id(dec)][:K + 1]    # every timed generation (each prefill resets the context's)
    steps_in_stats = max(1, sum(hist))
    tokens_per_step = sum((i + 1) * h for i, h in enumerate(hist)) / steps_in_stats
    alpha = sum(i * h for i, h in enumerate(hist)) / max(1, sum(i * h for i, h in enumerate(hist)) +
                                                         sum(hist[:K]))

    # ---- phase times (graph replay): verify pass, draft loop, plain decoding ----
    dec.prefill(prompt(0))
    prof = dec.profile(iters=20)
    L = args.prompt + args.new_tokens // 2     # mid-generation context for the byte count
    kv_t, kv_d = st["kv_bytes_per_token_target"], st["kv_bytes_per_token_draft"]
    verify_bytes = st["verify_weight_bytes"] + (L + K + 1) * kv_t + (K + 1) * tshape.vocab * 4
    draft_bytes = K * st["draft_weight_bytes"] + K * (L + K) * kv_d
    verify_gbs = verify_bytes / (prof["verify_ms"] * 1e6)
    hbm_peak, peak_kind = peaks()
    step_bytes = verify_bytes + draft_bytes
    roofline_tok_s = tokens_per_step / (step_bytes / (HBM_ROOFLINE_GBS * 1e9))

    # ---- plain autoregressive decoding on the same kernels ----
    ar = make(args.temperature, 0.0)
    ar.prefill(prompt(0))
    for _ in range(3):
        ar.ar_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ar.prefill(prompt(1))
    e0.record(stream)
    for _ in range(args.ar_tokens):
        ar.ar_step()
    e1.record(stream)
    e1.synchronize()
    ar_tok_s = args.ar_tokens / (e0.elapsed_time(e1) / 1000.0)
    ar_kernels = ar.stats()["kernels_per_ar_step"]
    ar.close()

    # ---- dominant kernel: the verify pass's target forward (one persistent
    # launch), timed live with CUDA events on the context's stream ----
    Lp = args.prompt - 1                       # context length at the profile (prefill of prompt(0))
    fwd_bytes = (st["verify_weight_bytes"] + (Lp + K + 1) * kv_t + (K + 1) * tshape.vocab * 4)
    fwd_achieved = fwd_bytes / (prof["verify_forward_ms"] * 1e6)
    # the record was taken on the 8B-shaped bf16 verify launch: other workloads'
    # launches (other shapes, 4-bit phases) are not covered by it
    traffic = persist_traffic_record() if args.workload == "8b" else None
    roofline = {"bound": "hbm",
                "kernel": "persist_forward (target verify pass over the K+1 positions)",
                "achieved": fwd_achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": fwd_achieved / hbm_peak, "peak_kind": peak_kind,
                "bytes_per_launch": fwd_bytes, "ms_per_launch": prof["verify_forward_ms"],
                "launches_timed": 20, "frac_of_8TBs": fwd_achieved / HBM_ROOFLINE_GBS,
                "traffic": traffic["traffic_ratio"] * fwd_bytes if traffic else None}

    # ---- sweep of the other draft settings of this workload ----
    sweep = []
    if not args.no_sweep:
        for temp, mix in [(1.0, 0.0), (1.0, 0.9), (0.0, 0.0), (0.0, 0.9)]:
            if (temp, mix) == (args.temperature, args.mix):
                continue
            d2 = make(temp, mix)
            d2.prefill(prompt(0))
            d2.step()
            m2, t2, n2 = timed_generations(d2, 60, 50)
            sweep.append({"temperature": temp, "mix_lambda": mix, "tokens_per_s": t2 / (m2 / 1000),
                          "tokens_per_step": t2 / n2,
                          "speedup_vs_ar": (t2 / (m2 / 1000)) / ar_tok_s})
            d2.close()
        # prompt-lookup drafting (n-gram suffix match up to 3 tokens) on prompts
        # of a repeated 128-token block; with random-init weights the target
        # does not follow the repetition, so this measures the step cost of
        # lookup drafting (one launch instead of the K draft passes)
        for temp in (1.0, 0.0):
            d2 = make(temp, 0.0, lookup=3)
            d2.prefill(repeat_prompt(0))
            d2.step()
            m2, t2, n2 = timed_generations(d2, 60, 70, repeat_prompt)
            sweep.append({"drafter": "prompt lookup (n-gram up to 3)", "temperature": temp,
                          "prompt": "128-token uniform block repeated", "tokens_per_s": t2 / (m2 / 1000),
                          "tokens_per_step": t2 / n2, "ms_per_step": m2 / n2,
                          "speedup_vs_ar": (t2 / (m2 / 1000)) / ar_tok_s})
            d2.close()

        # self-draft heads: K random d x d heads on the target's final hidden
        # state draft all K positions in one pass (structure and cost only:
        # random heads have no trained acceptance)
        if not q4:
            heads = workloads.make_heads(tshape, K, seed=5, device="cuda")
            for temp in (1.0, 0.0):
                d2 = sv.SpecDecoder(tshape, tw, None, None, K, max_ctx, temperature=temp, seed=0,
                                    stream=stream.cuda_stream, flags=base_flags, heads=heads)
                d2.prefill(prompt(0))
                d2.step()
                m2, t2, n2 = timed_generations(d2, 60, 90)
                d2.prefill(prompt(0))
                pr = d2.profile(iters=10)
                sweep.append({"drafter": f"self-draft heads ({K} random {tshape.d_model}x{tshape.d_model} heads on "
                                         f"the target's final hidden state, shared LM head)",
                              "temperature": temp, "tokens_per_s": t2 / (m2 / 1000), "tokens_per_step": t2 / n2,
                              "ms_per_step": m2 / n2, "heads_pass_ms": pr["draft_loop_ms"],
                              "heads_pass_kernels": pr["kernels_draft_loop"], "verify_ms": pr["verify_ms"],
                              "speedup_vs_ar": (t2 / (m2 / 1000)) / ar_tok_s})
                d2.close()
            del heads

    # ---- end to end through the C ABI with host buffers ----
    e2e_reqs, e2e_toks, e2e_steps = 2, 0, 0
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for i in range(e2e_reqs):
        dec.prefill(prompt(200 + i))       # host prompt -> device, prefill
        out = dec.generate(args.new_tokens)   # host token buffer
        e2e_toks += len(out)
        e2e_steps += dec.stats()["steps"]
    e2e_s = time.perf_counter() - w0
    e2e_steps = max(1, e2e_steps)
    e2e = {"value": e2e_toks / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": round(e2e_reqs * args.prompt * 4 / e2e_steps, 1),
           "d2h_bytes_per_step": (2 * K + 3) * 4,
           "includes": f"prompt upload ({args.prompt} int32) + prefill + {args.new_tokens} tokens per request"}

    # ---- oracle on the host cores (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not q4:
        del dec
        thw, dhw = to_host(tw), to_host(dw)      # the same weights the GPU ran
        n, secs, nsteps_cpu, threads = oracle_steps(tshape, thw, dshape, dhw, K, args.temperature, args.mix,
                                                    args.prompt, 20.0, 3)
        cpu = {"value": n / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{nsteps_cpu} complete fp64 oracle speculative step(s) of this workload (full "
                         f"depth, K={K}, {args.prompt}-token prompt, every position recomputed): "
                         f"{n} tokens in {secs:.1f} s measured"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": nsteps, "warmup": args.warmup, "ms_per_step": ms_max / max(1, nsteps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (4-bit weights)" if q4 else "bf16",
        "data": ("synthetic (random 4-bit codes with bf16 group scales, weights of std ~0.02, uniform-random prompts)"
                 if q4 else "synthetic (random N(0,0.02^2) weights, uniform-random prompts)"),
        "config": {"workload": wl, "batch": 1, "K": K, "prompt": args.prompt,
                   "new_tokens_per_generation": args.new_tokens, "temperature": args.temperature,
                   "mix_lambda": args.mix, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({(st['verify_weight_bytes'] + st['draft_weight_bytes']) / 1e9:.1f} "
                         f"GB of weights per step)"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": st["kernels_per_step"] * nsteps,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "verify_step": {"ms": prof["verify_ms"], "bytes": verify_bytes, "GB_s": verify_gbs,
                        "frac_of_8TBs": verify_gbs / HBM_ROOFLINE_GBS,
                        "frac_of_measured": verify_gbs / hbm_peak, "kernels": prof["kernels_verify"]},
        "draft_loop": {"ms": prof["draft_loop_ms"], "bytes": draft_bytes,
                       "GB_s": draft_bytes / (prof["draft_loop_ms"] * 1e6),
                       "kernels": prof["kernels_draft_loop"]},
        "ar_decoding": {"tokens_per_s": ar_tok_s, "ms_per_token": 1000.0 / ar_tok_s,
                        "pass_ms": prof["ar_ms"], "kernels_per_token": ar_kernels},
        "speedup_vs_ar": value / ar_tok_s,
        "tokens_per_step": tokens_per_step, "acceptance_alpha": alpha,
        "accepted_tokens_s_frac_of_8TBs_roofline": value / roofline_tok_s,
        "modelled_speedup": {"C": prof["draft_loop_ms"] / max(1e-9, K * prof["verify_ms"]),
                             "K_alpha_over_1_plus_KC": K * alpha / (1 + K * prof["draft_loop_ms"] /
                                                                    max(1e-9, K * prof["verify_ms"]))},
        "sweep": sweep,
        "wall_s_timed": wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
