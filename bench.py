#!/usr/bin/env python3
"""Benchmark of the GDN sublayer hot path on GB300 (one JSON line on stdout, rank 0).

One step = one pass of the prefill sublayer over the 4 x 4096-token batch (conv1d+SiLU kernel,
then the chunk-wise gated delta rule kernel with the sigmoid-gated RMSNorm fused; conv and
recurrent states written), inputs resident in HBM.  The headline value is prefill tokens/s.
The same line carries the fused decode step (256 sequences, one token each, 64 pre-generated
steps cycled) in seq-steps/s, with the recurrent state fp32 and again stored as binary16, the roofline of the dominant kernels, an end-to-end number
through host buffers, the fp64 CPU oracle timed on this host's cores, and the SM clocks seen
during the timed region.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun every rank runs an independent replica (the path has no exchange step); the
reported value is the sum over ranks of the tokens processed divided by the slowest rank's
time.  `--impl reference` times the CPU oracle itself on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s and decode seq-steps/s on 1 GB300; % of roofline"
# algorithmic bytes of the chunk-prefill kernel: per token qkv 20480 + g 192 + beta 192 + z 12288
# + out 12288; per sequence the fp32 state read and written (2 x 48 x 128 x 128 x 4)
CHUNK_BYTES_PER_TOKEN = 20480 + 192 + 192 + 12288 + 12288
STATE_BYTES_PER_SEQ = 2 * 48 * 128 * 128 * 4
# algorithmic bytes of one decode step per sequence: state in+out, conv state in+out (3 x 10240
# bf16 each way), x 20480, g+beta 384, z 12288, out 12288
DECODE_BYTES_PER_SEQ = STATE_BYTES_PER_SEQ + 2 * 10240 * 3 * 2 + 20480 + 384 + 12288 + 12288


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=640)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--varlen-steps", type=int, default=10)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--profile-verify", type=int, default=0, metavar="B",
                    help="profiler mode: only the verify leg (8 rows) on B sequences, --warmup + --steps transactions")
    ap.add_argument("--profile-case", default=None,
                    help="run only the prefill (conv + chunk) on these comma-separated sequence lengths, "
                         "--steps times after --warmup, for profiling; prints one timing line")
    ap.add_argument("--profile-kda-prefill", default=None, metavar="LENGTHS",
                    help="run only the KDA prefill (conv + KDA recurrence, 64 heads x 128) on these "
                         "comma-separated sequence lengths, --steps times after --warmup; prints one timing line")
    return ap.parse_args()


def run_profile_verify(args, local):
    """The verify leg alone for profilers: B sequences x 8 rows, verify + commit per transaction."""
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import linear_attention_ssm_gb300 as gdn
    from linear_attention_ssm_gb300.synth import decode_inputs
    B, K = args.profile_verify, VERIFY_ROWS
    d = decode_inputs(B, K, seed=5)
    vx, vg, vb, vz = (d[k].transpose(0, 1).contiguous().to(dev) for k in ("x", "g", "beta", "z"))
    w, nw = d["conv_w"].to(dev), d["norm_w"].to(dev)
    st, cs = d["state0"].to(dev), d["conv_state0"].to(dev)
    cm = torch.randint(1, K + 1, (B,), generator=torch.Generator().manual_seed(5), dtype=torch.int32).to(dev)
    out = torch.empty((B, K, 48, 128), dtype=torch.bfloat16, device=dev)
    stash = torch.empty(gdn.gdn_verify_stash_size(B, K), dtype=torch.uint8, device=dev)

    def step():
        gdn.gdn_verify(vx, w, cs, vg, vb, st, vz, nw, d["q_scale"], out=out, stash=stash)
        gdn.gdn_verify_commit(cm, stash, cs, st, K)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    print(json.dumps({"profile_verify": B, "rows": K, "ms_per_transaction": e0.elapsed_time(e1) / max(args.steps, 1)}))


def run_profile_kda_prefill(args, local):
    """A KDA prefill workload for profilers: --warmup untimed calls, then --steps calls."""
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import linear_attention_ssm_gb300 as gdn
    from linear_attention_ssm_gb300.synth import KDA_GEO, kda_prefill_inputs
    lengths = [int(v) for v in args.profile_kda_prefill.split(",")]
    geo, T = KDA_GEO, sum(lengths)
    d = kda_prefill_inputs(lengths, seed=11, geo=geo)
    x, cu, g, beta, z = (d[k].to(dev) for k in ("x", "cu_seqlens", "g", "beta", "z"))
    w, nw, st0 = d["conv_w"].to(dev), d["norm_w"].to(dev), d["state0"].to(dev)
    st = torch.empty_like(st0)
    qkv = torch.empty_like(x)
    out = torch.empty((T, geo.num_v_heads, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gdn.gdn_kda_chunk_prefill_workspace_size(len(lengths), T, geometry=geo), dtype=torch.uint8,
                     device=dev)

    def step():
        gdn.gdn_kda_prefill(x, w, cu, g, beta, z, nw, geo.q_scale, state_in=st0, state_out=st, qkv_buf=qkv, out=out,
                            workspace=ws, geometry=geo)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    print(json.dumps({"profile_kda_prefill": lengths, "tokens": T, "ms_per_step": e0.elapsed_time(e1) / max(args.steps, 1)}))


def run_profile_case(args, local):
    """A small prefill workload for profilers: --warmup untimed calls, then --steps calls."""
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import linear_attention_ssm_gb300 as gdn
    from linear_attention_ssm_gb300.synth import prefill_inputs
    lengths = [int(v) for v in args.profile_case.split(",")]
    inp = prefill_inputs(lengths, seed=2)
    N, T = len(lengths), sum(lengths)
    x, w, cu = inp["x"].to(dev), inp["conv_w"].to(dev), inp["cu_seqlens"].to(dev)
    g, beta, z, nw = inp["g"].to(dev), inp["beta"].to(dev), inp["z"].to(dev), inp["norm_w"].to(dev)
    state_in = inp["state0"].to(dev)
    state_out = torch.empty_like(state_in)
    qkv = torch.empty_like(x)
    out = torch.empty((T, 48, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gdn.gdn_chunk_prefill_workspace_size(N, T), dtype=torch.uint8, device=dev)

    def step():
        gdn.gdn_conv1d_prefill(x, w, cu, None, None, qkv)
        gdn.gdn_chunk_prefill(qkv, g, beta, cu, inp["q_scale"], 1e-6, state_in, state_out, z, nw, 1e-6, out,
                              workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    print(json.dumps({"profile_case": lengths, "tokens": T, "ms_per_step": e0.elapsed_time(e1) / max(args.steps, 1)}))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def code_digest(text):
    """Hash of a kernel source's code: `//` comments, trailing blanks and empty lines left out, so
    that a comment-only edit keeps a traffic record while any change to the code drops it."""
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()[:16]


def traffic_record(kernel):
    """ncu DRAM bytes per launch of `kernel`, if captured on the current code."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        src = os.path.join(ROOT, "linear_attention_ssm_gb300", "csrc", rec["source"])
        with open(src) as f:
            if code_digest(f.read()) != rec["code_sha256_16"]:
                return None
        return rec
    except Exception:
        return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        import torch
        ident = None
        try:
            ident = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ident = vis.split(",")[device_index] if vis else str(device_index)
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.06)
        self.proc.terminate()
        return self.summarize(self.proc.communicate(timeout=10)[0])

    @classmethod
    def summarize(cls, text):
        """Median SM clock, the largest maximum clock and every throttle reason seen Active in the
        sampler's CSV lines (sm, max sm, power, then the four reasons; unparsable lines skipped)."""
        sm, mx, reasons = [], [], set()
        for line in text.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(cls.NAMES, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def slowest_rank_ms(ms, world, device):
    """The largest of the ranks' timings (every rank calls this; world 1 needs no group)."""
    if world == 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, world, slowest_ms):
    """Whole-job throughput of `world` independent replicas: all ranks' units / slowest time."""
    return world * units_per_rank / (slowest_ms / 1000.0)


def dist_stats(ms):
    """Mean, median and the 10th / 90th percentiles of per-run times (ms)."""
    xs = sorted(float(v) for v in ms)
    n = len(xs)

    def pct(p):  # nearest-rank percentile
        return xs[min(n - 1, max(0, int(round(p / 100.0 * n + 0.5)) - 1))]
    return {"runs": n, "mean_ms": statistics.mean(xs), "p10_ms": pct(10), "p50_ms": statistics.median(xs),
            "p90_ms": pct(90)}


def step_bytes(tokens, seqs):
    """Algorithmic bytes of one fully fused prefill pass: per token x 20480 + z 12288 + g, beta 384 +
    out 12288; per sequence the fp32 state and the conv state, each read and written; the conv and
    norm weights once."""
    return 45440 * tokens + (STATE_BYTES_PER_SEQ + 2 * 10240 * 3 * 2) * seqs + 10240 * 4 * 2 + 128 * 2


def time_small_configs(gdn, dev, hbm_peak, runs=60, warm=10):
    """The correctness-sized workloads: one sequence of 16 tokens from a zero state, and separate
    sequences of 63, 64, 65, 80 and 128 tokens from a nonzero state.  Each prefill call (conv1d,
    then the chunk prefill with the fused gate) is captured in a CUDA graph and replayed, so that
    the host's per-call work leaves no gaps; one pair of CUDA events per replay."""
    import torch
    from linear_attention_ssm_gb300.synth import CHUNK_BOUNDARY_LENGTHS, prefill_inputs
    cases = [("S16_zero_state", 16, 0, True)] + [(f"S{S}", S, 1000 + S, False) for S in CHUNK_BOUNDARY_LENGTHS]
    res = {}
    for name, S, seed, zero in cases:
        inp = prefill_inputs([S], seed=seed, zero_state=zero)
        x, w, cu = inp["x"].to(dev), inp["conv_w"].to(dev), inp["cu_seqlens"].to(dev)
        g, beta, z, nw = inp["g"].to(dev), inp["beta"].to(dev), inp["z"].to(dev), inp["norm_w"].to(dev)
        st_in, cs_in = inp["state0"].to(dev), inp["conv_state0"].to(dev)
        st_out, cs_out = torch.empty_like(st_in), torch.empty_like(cs_in)
        qkv, out = torch.empty_like(x), torch.empty((S, 48, 128), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(gdn.gdn_chunk_prefill_workspace_size(1, S), dtype=torch.uint8, device=dev)

        def call():
            gdn.gdn_conv1d_prefill(x, w, cu, cs_in, cs_out, qkv)
            gdn.gdn_chunk_prefill(qkv, g, beta, cu, inp["q_scale"], 1e-6, None if zero else st_in, st_out, z, nw,
                                  1e-6, out, workspace=ws)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                call()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                call()
            for _ in range(warm):
                graph.replay()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
            for a, b in evs:
                a.record(side)
                graph.replay()
                b.record(side)
        torch.cuda.synchronize()
        gdn.gdn_check_device_errors()
        st = dist_stats([a.elapsed_time(b) for a, b in evs])
        roof = S / (step_bytes(S, 1) / (hbm_peak * 1e9))
        tps = S / (st["p50_ms"] / 1000.0)
        res[name] = {"tokens": S, "tokens_per_s": tps, "roofline_tokens_per_s": roof, "frac": tps / roof,
                     "algorithmic_bytes": step_bytes(S, 1), **st}
        del graph
    return res


def cpu_oracle_sample(inp, tokens_per_seq, nthreads=0):
    """The oracle (conv -> recurrence -> gated norm, fp64, all V heads) on the first
    `tokens_per_seq` tokens of every sequence, on `nthreads` threads (0: every core).  Returns
    (tokens/s, threads used, description)."""
    import torch
    import oracle
    from linear_attention_ssm_gb300.synth import cu_seqlens_of
    lengths = inp["lengths"]
    cu = inp["cu_seqlens"].tolist()
    idx = torch.cat([torch.arange(cu[n], cu[n] + min(tokens_per_seq, lengths[n])) for n in range(len(lengths))])
    sub = [min(tokens_per_seq, L) for L in lengths]
    t0 = time.perf_counter()
    oracle.prefill(inp["x"][idx], inp["conv_w"], cu_seqlens_of(sub), inp["g"][idx], inp["beta"][idx], inp["z"][idx],
                   inp["norm_w"], 16, 48, 128, 128, inp["q_scale"], state_in=inp["state0"], nthreads=nthreads)
    dt = time.perf_counter() - t0
    ntok = sum(sub)
    used = min(nthreads if nthreads > 0 else oracle.num_threads(), len(lengths) * 48)
    return ntok / dt, used, (f"first {tokens_per_seq} tokens of each of the {len(lengths)} "
                             f"sequences ({ntok} tokens, all 48 V heads), fp64, {used} threads, {dt:.2f} s")


def run_reference(args, rank, world):
    if rank != 0:
        return
    import torch  # noqa: F401
    import oracle
    from linear_attention_ssm_gb300.synth import BATCHED_LENGTHS, prefill_inputs
    oracle.build()
    inp = prefill_inputs(BATCHED_LENGTHS, seed=2)
    per_step = 64
    for _ in range(args.warmup):
        cpu_oracle_sample(inp, per_step)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        tps, cores, desc = cpu_oracle_sample(inp, per_step)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    tokens = per_step * len(BATCHED_LENGTHS) * args.steps
    value = tokens / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill 4 x 4096 tokens (sampled: first 64 tokens of each sequence per step)",
                   "global_batch": 4, "seq_len": 4096, "parallelism": "cpu threads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_kda_decode(args, gdn, dev, stream, barrier, max_over_ranks, world, hbm_peak):
    """KDA decode step (decay per key channel) on the pages' 64-head geometry, 256 sequences, 8
    pre-generated steps cycled."""
    import torch
    from linear_attention_ssm_gb300.synth import KDA_GEO, kda_decode_inputs
    geo, B, S = KDA_GEO, 256, 8
    d = kda_decode_inputs(B, S, seed=7)
    kx, kg, kb, kz = (d[k].to(dev) for k in ("x", "g", "beta", "z"))
    kw, knw = d["conv_w"].to(dev), d["norm_w"].to(dev)
    kst, kcs = d["state0"].to(dev), d["conv_state0"].to(dev)
    kout = torch.empty((B, geo.num_v_heads, 128), dtype=torch.bfloat16, device=dev)

    def step(s):
        gdn.gdn_kda_decode_step(kx[s], kw, kcs, kg[s], kb[s], kst, kz[s], knw, d["q_scale"], out=kout, geometry=geo)

    for s in range(max(args.warmup, 1)):
        step(s % S)
    barrier()
    n = max(args.decode_steps // 2, 4)
    s6, e6 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s6.record(stream)
    for s in range(n):
        step(s % S)
    e6.record(stream)
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    ms = max_over_ranks(s6.elapsed_time(e6)) / n
    C, hv = geo.conv_dim, geo.num_v_heads
    per_seq = 2 * hv * 128 * 128 * 4 + 2 * C * 3 * 2 + C * 2 + hv * 128 * 4 + hv * 4 + 2 * hv * 128 * 2
    nbytes = per_seq * B
    gbs = nbytes / (ms / 1e3) / 1e9
    del kx, kg, kb, kz, kst, kcs
    return {"metric": "KDA decode seq-steps/s", "value": world * B / (ms / 1e3), "unit": "seq-steps/s",
            "ms_per_step": ms, "steps": n, "batch": B,
            "workload": "KDA decode, 256 sequences x one token, 64 heads x 128 (q, k, v), per-channel decay",
            "roofline": {"kernel": "decode_step_kernel (per-channel decay)", "bound": "hbm", "achieved": gbs,
                         "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "traffic": (traffic_record("decode_kda") or {}).get("bytes_per_launch"),
                         "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": ms}}


def kda_prefill_bytes(tokens, seqs, hv):
    """Algorithmic bytes of one KDA recurrence call (in either form): per (token, V head) q, k, v, z
    (bf16 rows of 128), g (fp32 row of 128) and beta in, the bf16 output row out; per (sequence,
    V head) the fp32 state in and out."""
    return tokens * hv * (4 * 256 + 512 + 4 + 256) + 2 * seqs * hv * 128 * 128 * 4


def time_kda_prefill(args, gdn, dev, stream, barrier, max_over_ranks, world):
    """KDA prefill on the pages' 64-head geometry, 4 sequences x 4096 tokens: conv1d, then the KDA
    recurrence in its chunk-wise form with the gated RMSNorm fused (both timed with events, and
    the chunk call alone for its roofline); the sequential recurrence kernel is timed beside it.
    x alone is 805 MB per step, larger than L2."""
    import torch
    from linear_attention_ssm_gb300.synth import KDA_GEO, kda_prefill_inputs
    geo, lengths = KDA_GEO, [4096] * 4
    T, N = sum(lengths), len(lengths)
    d = kda_prefill_inputs(lengths, seed=11, geo=geo)
    x, cu, g, beta, z = (d[k].to(dev) for k in ("x", "cu_seqlens", "g", "beta", "z"))
    w, nw, st0 = d["conv_w"].to(dev), d["norm_w"].to(dev), d["state0"].to(dev)
    del d
    st = torch.empty_like(st0)
    qkv = torch.empty((T, geo.conv_dim), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, geo.num_v_heads, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gdn.gdn_kda_chunk_prefill_workspace_size(N, T, geometry=geo), dtype=torch.uint8, device=dev)
    qs = geo.q_scale

    def whole():
        gdn.gdn_kda_prefill(x, w, cu, g, beta, z, nw, qs, state_in=st0, state_out=st, qkv_buf=qkv, out=out,
                            workspace=ws, geometry=geo)

    def chunk():
        gdn.gdn_kda_chunk_prefill(qkv, g, beta, cu, qs, state_in=st0, state_out=st, z=z, norm_w=nw, out=out,
                                  workspace=ws, geometry=geo)

    def sequential():
        gdn.gdn_kda_recurrence(qkv, g, beta, cu, qs, state_in=st0, state_out=st, z=z, norm_w=nw, out=out,
                               geometry=geo)

    n = 5
    timed = {}
    for name, fn in (("whole", whole), ("chunk", chunk), ("sequential", sequential)):
        for _ in range(max(args.warmup, 1)):
            fn()
        barrier()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(n):
            fn()
        e0.record(stream)
        torch.cuda.synchronize()
        gdn.gdn_check_device_errors()
        timed[name] = max_over_ranks(s0.elapsed_time(e0)) / n
    del x, cu, g, beta, z, st0, st, qkv, out, ws
    torch.cuda.empty_cache()
    hbm_peak, _, peak_kind = peaks()
    nbytes = kda_prefill_bytes(T, N, geo.num_v_heads)
    gbs = nbytes / (timed["chunk"] / 1e3) / 1e9
    rec = traffic_record("kda_chunk_prefill")
    return {"metric": "KDA prefill tokens/s", "value": world * T / (timed["whole"] / 1e3), "unit": "tokens/s",
            "ms_per_step": timed["whole"], "steps": n,
            "workload": "KDA prefill, 4 sequences x 4096 tokens, 64 heads x 128 (q, k, v), per-channel decay, "
                        "conv1d -> chunk-wise KDA recurrence (prep + state kernels) -> sigmoid-gated RMSNorm",
            "sequential_recurrence_ms": timed["sequential"],
            "roofline": {"kernel": "kda_chunk_prefill (schedule + prep + state kernels, tcgen05, fused gated norm)",
                         "bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "peak_kind": peak_kind + " (copy bandwidth)",
                         "traffic": rec["bytes_per_launch"] if rec else None,
                         "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": timed["chunk"]}}


VERIFY_ROWS = 8
VERIFY_RECORD = 53440  # stash bytes per (sequence, row): raw inputs, keys, deltas, g


def time_verify(args, gdn, dev, stream, barrier, max_over_ranks, world, hbm_peak, state_dtype=None):
    """Verify of 8 rows for each of 256 sequences, then the commit of a seeded verdict in 1..8
    (the accepted proposals plus one correction row).  Both kernels are timed with events."""
    import torch
    from linear_attention_ssm_gb300.synth import DECODE_BATCH, decode_inputs
    B, K = DECODE_BATCH, VERIFY_ROWS
    d = decode_inputs(B, K, seed=5)
    vx, vg, vb, vz = (d[k].transpose(0, 1).contiguous().to(dev) for k in ("x", "g", "beta", "z"))
    w, nw = d["conv_w"].to(dev), d["norm_w"].to(dev)
    st0, cs0 = d["state0"].to(dev).to(state_dtype or torch.float32), d["conv_state0"].to(dev)
    st, cs = st0.clone(), cs0.clone()
    gen = torch.Generator().manual_seed(5)
    committed = torch.randint(1, K + 1, (B,), generator=gen, dtype=torch.int32)
    cm = committed.to(dev)
    out = torch.empty((B, K, 48, 128), dtype=torch.bfloat16, device=dev)
    stash = torch.empty(gdn.gdn_verify_stash_size(B, K), dtype=torch.uint8, device=dev)

    def step(ev=None):
        if ev: ev[0].record(stream)
        gdn.gdn_verify(vx, w, cs, vg, vb, st, vz, nw, d["q_scale"], out=out, stash=stash)
        if ev: ev[1].record(stream)
        gdn.gdn_verify_commit(cm, stash, cs, st, K)
        if ev: ev[2].record(stream)

    for _ in range(max(args.warmup, 1)):
        step()
    barrier()
    n = max(args.decode_steps // 4, 10)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    v_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / n)
    c_ms = max_over_ranks(sum(e[1].elapsed_time(e[2]) for e in evs) / n)
    step_ms = max_over_ranks(sum(e[0].elapsed_time(e[2]) for e in evs) / n)
    C, hv = 10240, 48
    state_bytes = B * hv * 128 * 128 * st0.element_size()
    v_bytes = (state_bytes + B * K * C * 2 + B * C * 3 * 2 + B * K * hv * 8 + 2 * B * K * hv * 128 * 2
               + B * K * VERIFY_RECORD)
    m = committed.tolist()
    c_bytes = (2 * state_bytes + 2 * B * C * 3 * 2
               + sum(r * (16 * 128 * 4 + hv * 128 * 4 + hv * 4) + min(r, 3) * C * 2 for r in m))
    sfx = "_fp16_state" if st0.element_size() == 2 else ""
    roof = lambda nbytes, ms, kernel, rec: {"kernel": kernel, "bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                                            "peak": hbm_peak, "unit": "GB/s",
                                            "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                                            "traffic": (traffic_record(rec) or {}).get("bytes_per_launch"),
                                            "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": ms}
    return {"metric": "verify rows/s", "value": world * B * K / (step_ms / 1e3), "unit": "rows/s",
            "ms_per_step": step_ms, "steps": n, "batch": B, "rows": K,
            "committed_rows_mean": sum(m) / B,
            "workload": f"256 sequences x 8 verify rows ({'binary16' if st0.element_size() == 2 else 'fp32'} state), "
                        "then the commit of a seeded verdict in 1..8",
            "roofline_verify": roof(v_bytes, v_ms, "verify_kernel", "verify" + sfx),
            "roofline_commit": roof(c_bytes, c_ms, "commit_kernel", "verify_commit" + sfx)}


def _r(v, d=4):
    """A number rounded to `d` significant digits (None passes through)."""
    if v is None:
        return None
    return float(f"{float(v):.{d}g}")


def compact_summary(line, step_dist):
    """Every leg's figures in a few hundred characters, placed last on the line so that a reader
    that keeps only the line's end still sees them."""
    def leg(d, unit_key="value", scale=1e6):
        if not d or "error" in d:
            return d and {"error": d["error"][:80]}
        r = d.get("roofline") or {}
        return {"M_per_s": _r(d[unit_key] / scale), "ms": _r(d.get("ms_per_step")), "frac": _r(r.get("frac"), 3)}
    out = {"prefill": {"M_tok_s": _r(line["value"] / 1e6), "frac": _r(line["roofline"]["frac"], 3),
                       "p10_p50_p90_ms": [_r(step_dist[k]) for k in ("p10_ms", "p50_ms", "p90_ms")],
                       "runs": step_dist["runs"]}}
    out["decode"] = leg(line["decode"])
    out["decode_fused_gates"] = leg(line["decode_fused_gates"])
    out["prefill_fused_gates"] = {"M_tok_s": _r(line["prefill_fused_gates"]["value"] / 1e6),
                                  "ms": _r(line["prefill_fused_gates"]["ms_per_step"])}
    out["decode_f16"] = leg(line["decode_fp16_state"])
    out["decode_kda"] = leg(line["decode_kda"])
    v = line.get("varlen")
    if v:
        out["varlen"] = {"M_tok_s": _r(v["value"] / 1e6), "ms": _r(v["ms_per_step"]), "frac": _r(v["frac"], 3)}
    for key in ("verify", "verify_fp16_state"):
        d = line.get(key) or {}
        if d and "error" not in d:
            out[key] = {"M_rows_s": _r(d.get("value", 0) / 1e6), "ms": _r(d.get("ms_per_step")),
                        "frac": _r((d.get("roofline_verify") or {}).get("frac"), 3),
                        "commit_frac": _r((d.get("roofline_commit") or {}).get("frac"), 3)}
    out["kda_prefill"] = leg(line.get("kda_prefill"))
    out["small_configs"] = {k: {"M_tok_s": _r(d["tokens_per_s"] / 1e6, 3), "p50_us": _r(1e3 * d["p50_ms"], 3),
                                "frac": _r(d["frac"], 3)} for k, d in line["small_configs"].items()}
    c = line.get("cpu_baseline")
    if c:
        out["cpu"] = {"tok_s_all": _r(c["value"]), "threads": c["cores"],
                      "tok_s_1thread": _r(c["single_thread"]["value"]), "nproc": c.get("nproc")}
    return out


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import linear_attention_ssm_gb300 as gdn
    from linear_attention_ssm_gb300 import build as gdn_build
    from linear_attention_ssm_gb300.synth import (BATCHED_LENGTHS, DECODE_BATCH, DECODE_STEPS, VARLEN_LENGTHS,
                                                  decode_inputs, prefill_inputs)
    if not os.path.exists(gdn.binding.LIB_PATH):
        gdn_build.build()
    gdn.load_library()
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return slowest_rank_ms(v, world, dev)

    hbm_peak, _, peak_kind = peaks()
    stream = torch.cuda.current_stream()

    # ---------------- prefill, 4 x 4096 tokens
    inp = prefill_inputs(BATCHED_LENGTHS, seed=2)
    N, T = len(BATCHED_LENGTHS), sum(BATCHED_LENGTHS)
    x, w, cu = inp["x"].to(dev), inp["conv_w"].to(dev), inp["cu_seqlens"].to(dev)
    g, beta, z, nw = inp["g"].to(dev), inp["beta"].to(dev), inp["z"].to(dev), inp["norm_w"].to(dev)
    state_in = inp["state0"].to(dev)
    state_out = torch.empty_like(state_in)
    cs_in = inp["conv_state0"].to(dev)
    cs_out = torch.empty_like(cs_in)
    qkv = torch.empty_like(x)
    out = torch.empty((T, 48, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gdn.gdn_chunk_prefill_workspace_size(N, T), dtype=torch.uint8, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ev_conv = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def prefill_step(i=None):
        if i is not None:
            ev_conv[i][0].record(stream)
        gdn.gdn_conv1d_prefill(x, w, cu, cs_in, cs_out, qkv)
        if i is not None:
            ev_conv[i][1].record(stream)
            ev[i][0].record(stream)
        gdn.gdn_chunk_prefill(qkv, g, beta, cu, inp["q_scale"], 1e-6, state_in, state_out, z, nw, 1e-6, out,
                              workspace=ws)
        if i is not None:
            ev[i][1].record(stream)

    for _ in range(max(args.warmup, 1)):
        prefill_step()
    gdn.gdn_check_device_errors()
    barrier()
    clocks = ClockSampler(local)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        prefill_step(i)
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    gdn.gdn_check_device_errors()
    ms = max_over_ranks(start.elapsed_time(end))
    ms_per_step = ms / args.steps
    value = replica_throughput(T, world, ms_per_step)
    chunk_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    conv_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_conv)
    chunk_bytes = CHUNK_BYTES_PER_TOKEN * T + STATE_BYTES_PER_SEQ * N
    chunk_gbs = chunk_bytes / (chunk_ms / 1000.0) / 1e9
    rec = traffic_record("chunk_prefill_split")
    roofline = {"kernel": "chunk_prefill (schedule + prep + state kernels, tcgen05, fused gated norm)",
                "bound": "hbm", "achieved": chunk_gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": chunk_gbs / hbm_peak,
                "peak_kind": peak_kind + " (copy bandwidth)",
                "traffic": rec["bytes_per_launch"] if rec else None,
                "algorithmic_bytes_per_launch": chunk_bytes, "avg_launch_ms": chunk_ms}
    conv_bytes = T * 10240 * 2 * 2 + N * 10240 * 3 * 2 * 2 + 10240 * 4 * 2
    crec = traffic_record("conv1d_prefill")
    conv_roof = {"kernel": "conv1d_prefill", "bound": "hbm", "achieved": conv_bytes / (conv_ms / 1000) / 1e9,
                 "peak": hbm_peak, "unit": "GB/s", "avg_launch_ms": conv_ms,
                 "algorithmic_bytes_per_launch": conv_bytes, "traffic": crec["bytes_per_launch"] if crec else None}
    conv_roof["frac"] = conv_roof["achieved"] / hbm_peak

    # the prefill step with the gates derived in the prep kernel from the a / b projections
    from linear_attention_ssm_gb300.synth import gate_inputs as _gate_inputs
    gpi = _gate_inputs(T, seed=6)
    pa, pb, pal, pdb = (gpi[k].to(dev) for k in ("a", "b", "A_log", "dt_bias"))

    def prefill_fg_step():
        gdn.gdn_conv1d_prefill(x, w, cu, cs_in, cs_out, qkv)
        gdn.gdn_chunk_prefill_fused_gates(qkv, pa, pb, pal, pdb, cu, inp["q_scale"], 1e-6, state_in, state_out, z, nw,
                                          1e-6, out, workspace=ws)
    for _ in range(max(args.warmup, 1)):
        prefill_fg_step()
    barrier()
    sfg, efg = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sfg.record(stream)
    for _ in range(args.steps):
        prefill_fg_step()
    efg.record(stream)
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    fg_ms = max_over_ranks(sfg.elapsed_time(efg)) / args.steps
    prefill_fg = {"workload": "the headline step with the gates derived in the prep kernel from a, b (bf16), "
                              "A_log, dt_bias", "value": replica_throughput(T, world, fg_ms), "unit": "tokens/s",
                  "ms_per_step": fg_ms, "steps": args.steps}
    del pa, pb, pal, pdb

    # distribution of per-step times over a separate pass of at least 50 steps (the headline above
    # times exactly --steps steps between two events): whole step, and the chunk prefill alone
    nd = max(50, args.steps)
    evd = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nd)]
    barrier()
    for e0, e1, e2 in evd:
        e0.record(stream)
        gdn.gdn_conv1d_prefill(x, w, cu, cs_in, cs_out, qkv)
        e1.record(stream)
        gdn.gdn_chunk_prefill(qkv, g, beta, cu, inp["q_scale"], 1e-6, state_in, state_out, z, nw, 1e-6, out,
                              workspace=ws)
        e2.record(stream)
    torch.cuda.synchronize()
    step_dist = dist_stats([e0.elapsed_time(e2) for e0, _, e2 in evd])
    chunk_dist = dist_stats([e1.elapsed_time(e2) for _, e1, e2 in evd])
    roofline["launch_ms_distribution"] = chunk_dist

    # ---------------- end to end through host buffers (pinned): every step copies its inputs from
    # host to device, runs the prefill and reads its outputs back to the host.  Device inputs and
    # outputs are double-buffered and the copies run on two copy streams, so the H2D copy of step
    # i + 1 and the D2H read of step i - 1 overlap the prefill of step i (a serving loop's layout).
    h_x, h_g, h_b, h_z = (inp["x"].pin_memory(), inp["g"].pin_memory(), inp["beta"].pin_memory(),
                          inp["z"].pin_memory())
    h_state, h_cs = inp["state0"].pin_memory(), inp["conv_state0"].pin_memory()
    h_out = torch.empty((T, 48, 128), dtype=torch.bfloat16).pin_memory()
    h_state_out = torch.empty_like(h_state).pin_memory()
    h_cs_out = torch.empty_like(h_cs).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_x, h_g, h_b, h_z, h_state, h_cs))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_state_out, h_cs_out))
    cin, cin2, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    bufs = [dict(x=x, g=g, beta=beta, z=z, st=state_in, cs=cs_in, out=out, st_out=state_out, cs_out=cs_out)]
    bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "in2", "comp", "out")}

    def e2e_step(i):
        bi = i % 2
        B = bufs[bi]
        # two H2D streams (x on one, the rest on the other): two copy engines in flight
        for st_, key, pairs in ((cin, "in", (("x", h_x),)),
                                (cin2, "in2", (("g", h_g), ("beta", h_b), ("z", h_z), ("st", h_state), ("cs", h_cs)))):
            with torch.cuda.stream(st_):
                st_.wait_event(ev["comp"][bi])  # the prefill two steps back has read this buffer's inputs
                for k, h in pairs:
                    B[k].copy_(h, non_blocking=True)
                ev[key][bi].record(st_)
        stream.wait_event(ev["in"][bi])
        stream.wait_event(ev["in2"][bi])
        stream.wait_event(ev["out"][bi])  # the outputs two steps back have been read out
        gdn.gdn_prefill(B["x"], w, cu, B["g"], B["beta"], B["z"], nw, inp["q_scale"], 1e-6, 1e-6, state_in=B["st"],
                        state_out=B["st_out"], conv_state_in=B["cs"], conv_state_out=B["cs_out"], qkv_buf=qkv,
                        out=B["out"], workspace=ws)
        ev["comp"][bi].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(ev["comp"][bi])
            h_out.copy_(B["out"], non_blocking=True)
            h_state_out.copy_(B["st_out"], non_blocking=True)
            h_cs_out.copy_(B["cs_out"], non_blocking=True)
            ev["out"][bi].record(cout)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    cin.wait_stream(stream)  # no copy of the timed steps starts before the start mark
    cin2.wait_stream(stream)
    for i in range(args.e2e_steps):
        e2e_step(i)
    stream.wait_stream(cout)
    stream.wait_stream(cin)
    stream.wait_stream(cin2)
    e2.record(stream)
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2)) / args.e2e_steps
    e2e_value = replica_throughput(T, world, e2e_ms)

    # the host link alone: the same copies without the prefill, host to device on the two input
    # streams, device to host on the output stream, and both at once
    def copies(i, h2d_on, d2h_on):
        B = bufs[i % 2]
        if h2d_on:
            with torch.cuda.stream(cin):
                B["x"].copy_(h_x, non_blocking=True)
            with torch.cuda.stream(cin2):
                for k, h in (("g", h_g), ("beta", h_b), ("z", h_z), ("st", h_state), ("cs", h_cs)):
                    B[k].copy_(h, non_blocking=True)
        if d2h_on:
            with torch.cuda.stream(cout):
                h_out.copy_(B["out"], non_blocking=True)
                h_state_out.copy_(B["st_out"], non_blocking=True)
                h_cs_out.copy_(B["cs_out"], non_blocking=True)

    def time_copies(h2d_on, d2h_on):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for st_ in (cin, cin2, cout):
            st_.wait_stream(stream)
        for i in range(args.e2e_steps):
            copies(i, h2d_on, d2h_on)
        for st_ in (cin, cin2, cout):
            stream.wait_stream(st_)
        b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b)) / args.e2e_steps

    h2d_ms, d2h_ms, both_ms = time_copies(True, False), time_copies(False, True), time_copies(True, True)
    host_link = {"h2d_gbs": h2d / (h2d_ms / 1e3) / 1e9, "d2h_gbs": d2h / (d2h_ms / 1e3) / 1e9,
                 "copies_only_ms_per_step": both_ms,
                 "note": "the e2e step's pinned copies alone (no prefill): its floor"}
    del h_x, h_g, h_b, h_z, bufs

    # ---------------- varlen prefill: 8 packed sequences, 31,735 tokens (same path)
    del x, qkv, z, out, ws
    torch.cuda.empty_cache()
    varlen = None
    if args.varlen_steps > 0:
        vin = prefill_inputs(VARLEN_LENGTHS, seed=3)
        vN, vT = len(VARLEN_LENGTHS), sum(VARLEN_LENGTHS)
        vx, vcu = vin["x"].to(dev), vin["cu_seqlens"].to(dev)
        vg, vb, vz = vin["g"].to(dev), vin["beta"].to(dev), vin["z"].to(dev)
        vs_in = vin["state0"].to(dev)
        vs_out = torch.empty_like(vs_in)
        vcs_in = vin["conv_state0"].to(dev)
        vcs_out = torch.empty_like(vcs_in)
        vqkv = torch.empty_like(vx)
        vout = torch.empty((vT, 48, 128), dtype=torch.bfloat16, device=dev)
        vws = torch.empty(gdn.gdn_chunk_prefill_workspace_size(vN, vT), dtype=torch.uint8, device=dev)

        def varlen_step():
            gdn.gdn_conv1d_prefill(vx, w, vcu, vcs_in, vcs_out, vqkv)
            gdn.gdn_chunk_prefill(vqkv, vg, vb, vcu, vin["q_scale"], 1e-6, vs_in, vs_out, vz, nw, 1e-6, vout,
                                  workspace=vws)

        for _ in range(max(args.warmup, 1)):
            varlen_step()
        barrier()
        s4, e4 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s4.record(stream)
        for _ in range(args.varlen_steps):
            varlen_step()
        e4.record(stream)
        torch.cuda.synchronize()
        gdn.gdn_check_device_errors()
        v_ms = max_over_ranks(s4.elapsed_time(e4)) / args.varlen_steps
        v_roof = hbm_peak * 1e9 / (CHUNK_BYTES_PER_TOKEN + STATE_BYTES_PER_SEQ * vN / vT)
        varlen = {"workload": "varlen prefill, 8 packed sequences {1,17,63,64,65,1000,8191,22334} = 31,735 tokens",
                  "value": world * vT / (v_ms / 1000.0), "unit": "tokens/s", "ms_per_step": v_ms,
                  "steps": args.varlen_steps, "roofline_tokens_per_s": v_roof,
                  "frac": vT / (v_ms / 1000.0) / v_roof,
                  "frac_note": "conv1d + chunk prefill step against the chunk prefill's HBM roofline (the "
                               "algorithmic bytes of the chunk stage, as for the headline)"}
        del vin, vx, vqkv, vz, vout, vws
        torch.cuda.empty_cache()

    # ---------------- decode: 256 sequences, 64 pre-generated steps cycled
    d = decode_inputs(DECODE_BATCH, DECODE_STEPS, seed=4)
    B = DECODE_BATCH
    dx, dg, db, dz = d["x"].to(dev), d["g"].to(dev), d["beta"].to(dev), d["z"].to(dev)
    dw, dnw = d["conv_w"].to(dev), d["norm_w"].to(dev)
    dout = torch.empty((B, 48, 128), dtype=torch.bfloat16, device=dev)

    def time_decode(state_dtype, state_bytes_per_seq, kernel):
        dstate, dcs = d["state0"].to(dev).to(state_dtype), d["conv_state0"].to(dev)

        def decode_step(s):
            gdn.gdn_decode_step(dx[s], dw, dcs, dg[s], db[s], dstate, dz[s], dnw, d["q_scale"], out=dout)

        for s in range(max(args.warmup, 1)):
            decode_step(s % DECODE_STEPS)
        barrier()
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s3.record(stream)
        for s in range(args.decode_steps):
            decode_step(s % DECODE_STEPS)
        e3.record(stream)
        torch.cuda.synchronize()
        gdn.gdn_check_device_errors()
        dec_ms = max_over_ranks(s3.elapsed_time(e3)) / args.decode_steps
        dec_bytes = (DECODE_BYTES_PER_SEQ - STATE_BYTES_PER_SEQ + state_bytes_per_seq) * B
        dec_gbs = dec_bytes / (dec_ms / 1000) / 1e9
        del dstate, dcs
        return {"metric": "decode seq-steps/s", "value": world * B / (dec_ms / 1000), "unit": "seq-steps/s",
                "ms_per_step": dec_ms, "steps": args.decode_steps, "batch": B,
                "roofline": {"kernel": kernel, "bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak,
                             "unit": "GB/s", "frac": dec_gbs / hbm_peak,
                             "traffic": (traffic_record(kernel) or {}).get("bytes_per_launch"),
                             "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_ms": dec_ms},
                "roofline_seq_steps_per_s": hbm_peak * 1e9 / (dec_bytes / B)}

    decode = time_decode(torch.float32, STATE_BYTES_PER_SEQ, "decode_step")

    # the same step with the gates derived in the kernel from the a / b projections (bf16) and the
    # per-head A_log, dt_bias: 4 bytes of gate input per (sequence, V head) instead of 8
    from linear_attention_ssm_gb300.synth import gate_inputs
    gsteps = [gate_inputs(B, seed=40 + s) for s in range(DECODE_STEPS)]
    ga_all = torch.stack([gs["a"] for gs in gsteps]).to(dev)
    gb_all = torch.stack([gs["b"] for gs in gsteps]).to(dev)
    gal, gdb = gsteps[0]["A_log"].to(dev), gsteps[0]["dt_bias"].to(dev)

    def time_decode_fused_gates():
        dstate, dcs = d["state0"].to(dev), d["conv_state0"].to(dev)

        def step(s):
            gdn.gdn_decode_step_fused_gates(dx[s], dw, dcs, ga_all[s], gb_all[s], gal, gdb, dstate, dz[s], dnw,
                                            d["q_scale"], out=dout)
        for s in range(max(args.warmup, 1)):
            step(s % DECODE_STEPS)
        barrier()
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s3.record(stream)
        for s in range(args.decode_steps):
            step(s % DECODE_STEPS)
        e3.record(stream)
        torch.cuda.synchronize()
        gdn.gdn_check_device_errors()
        ms_ = max_over_ranks(s3.elapsed_time(e3)) / args.decode_steps
        nbytes = (DECODE_BYTES_PER_SEQ - 384 + 48 * 4) * B + 2 * 48 * 4
        gbs = nbytes / (ms_ / 1000) / 1e9
        del dstate, dcs
        return {"metric": "decode seq-steps/s", "value": world * B / (ms_ / 1000), "unit": "seq-steps/s",
                "ms_per_step": ms_, "steps": args.decode_steps, "batch": B,
                "gates": "derived in the decode kernel from a, b (bf16) and A_log, dt_bias",
                "roofline": {"kernel": "decode_step (fused gates)", "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                             "unit": "GB/s", "frac": gbs / hbm_peak, "algorithmic_bytes_per_launch": nbytes,
                             "avg_launch_ms": ms_}}

    decode_fg = time_decode_fused_gates()
    del ga_all, gb_all
    decode_kda = time_kda_decode(args, gdn, dev, stream, barrier, max_over_ranks, world, hbm_peak)
    # the same workload with the recurrent state stored as binary16 (half the state bytes)
    decode_f16 = time_decode(torch.float16, STATE_BYTES_PER_SEQ // 2, "decode_step_fp16_state")
    decode_f16["state"] = "binary16 in memory, fp32 arithmetic, rounded once per step"

    del d, dx, dg, db, dz
    torch.cuda.empty_cache()

    # ---------------- gates from their projections for the 4 x 4096 tokens (elementwise, HBM)
    from linear_attention_ssm_gb300.synth import gate_inputs
    gi = gate_inputs(T, seed=6)
    ga, gb_, gal, gdb = (gi[k].to(dev) for k in ("a", "b", "A_log", "dt_bias"))
    g_out = torch.empty((T, 48), dtype=torch.float32, device=dev)
    b_out = torch.empty((T, 48), dtype=torch.float32, device=dev)
    for _ in range(max(args.warmup, 1)):
        gdn.gdn_gates(ga, gb_, gal, gdb, g_out, b_out)
    # a microseconds-long kernel: its launches are captured in a CUDA graph so that the host's
    # per-call work does not leave gaps on the GPU between them
    ng = 50
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(ng):
                gdn.gdn_gates(ga, gb_, gal, gdb, g_out, b_out)
    stream.wait_stream(side)
    graph.replay()
    barrier()
    s5, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 4
    s5.record(stream)
    for _ in range(reps):
        graph.replay()
    e5.record(stream)
    torch.cuda.synchronize()
    gdn.gdn_check_device_errors()
    g_ms = max_over_ranks(s5.elapsed_time(e5)) / (ng * reps)
    g_bytes = T * 48 * (2 + 2 + 4 + 4)
    gates = {"workload": "gates g, beta from the a / b projections, 16,384 tokens x 48 V heads",
             "ms_per_launch": g_ms, "achieved_gbs": g_bytes / (g_ms / 1e3) / 1e9,
             "algorithmic_bytes_per_launch": g_bytes, "launches": ng * reps,
             "timing": "a CUDA graph of 50 launches, replayed 4 times",
             "note": "9.4 MB per launch: launch latency, not HBM, sets its time"}
    del graph, ga, gb_, gal, gdb, g_out, b_out

    # ---------------- multi-token verify: 256 sequences x 8 rows, then the commit of a verdict
    verify = time_verify(args, gdn, dev, stream, barrier, max_over_ranks, world, hbm_peak)
    verify_f16 = time_verify(args, gdn, dev, stream, barrier, max_over_ranks, world, hbm_peak, torch.float16)

    # ---------------- KDA prefill: conv1d, then the KDA recurrence (per-channel decay), 4 x 4096 tokens
    try:
        kda_prefill = time_kda_prefill(args, gdn, dev, stream, barrier, max_over_ranks, world)
    except Exception as exc:  # a secondary leg reports its failure without taking the line down
        kda_prefill = {"error": f"{type(exc).__name__}: {exc}"}

    # ---------------- the correctness-sized workloads (16 tokens; 63 / 64 / 65 / 80 / 128 tokens)
    small = time_small_configs(gdn, dev, hbm_peak)

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        tps, cores, desc = cpu_oracle_sample(inp, 2048)
        tps1, _, desc1 = cpu_oracle_sample(inp, 96, nthreads=1)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc,
               "single_thread": {"value": tps1, "unit": "tokens/s", "sample": desc1},
               "nproc": os.cpu_count()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "GDN prefill sublayer, 4 sequences x 4096 tokens (conv1d+SiLU -> chunk-wise "
                                   "gated delta rule -> sigmoid-gated RMSNorm), Hk=16 Hv=48 Dk=Dv=128, chunk 64",
                       "global_batch": 4 * world, "seq_len": 4096, "tokens_per_step_per_gpu": T,
                       "l2": "inputs larger than L2 (x 335 MB per step)", "parallelism": f"replicas x{world}"},
            "roofline": roofline, "roofline_conv": conv_roof,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": args.e2e_steps,
                    "pipelined": "H2D of step i+1 and D2H of step i-1 overlap the prefill of step i",
                    "host_link": host_link},
            "decode": decode, "decode_fused_gates": decode_fg, "prefill_fused_gates": prefill_fg,
            "decode_fp16_state": decode_f16, "decode_kda": decode_kda, "verify": verify,
            "verify_fp16_state": verify_f16,
            "gates": gates, "kda_prefill": kda_prefill,
            "varlen": varlen, "small_configs": small, "cpu_baseline": cpu, "clocks": clk,
            # per step: conv1d + conv-state kernels, the chunk prefill's schedule and segment / part
            # table kernels, then for each of its three chunk segments a prep, a state and a parts
            # launch (the state kernel of split sequences; with nothing split its CTAs return at once)
            "gpu_launches": (2 + 2 + 3 * 3) * args.steps,
            "arithmetic": "bf16 tensor-core operands (fp32 operands split into bf16 hi+lo), fp32 accumulate and state",
        }
        line["summary"] = compact_summary(line, step_dist)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.profile_verify:
        run_profile_verify(args, local)
    elif args.profile_case:
        run_profile_case(args, local)
    elif args.profile_kda_prefill:
        run_profile_kda_prefill(args, local)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
