#!/usr/bin/env python
"""Benchmark of the DSA sparse-MLA hot path on GB300.

One step = one pass of the whole path over one batch: causal top-k over the
indexer scores, the sparse MLA Partial over the selected FP8 rows and, when
the launch splits the KV range, the Combine.  Inputs are seeded synthetic
tensors with the shapes of the GLM-5.3-Flash serving workloads (default: 128
decode requests at 64K context sharing a 99.9% prefix, top-k 2048, 64 heads,
latent 512 + rope 64, FP8 E4M3 KV with per-token scales).

Prints one JSON line: whole-job query-tokens/s with inputs resident in HBM
(`value`), the same through host buffers with the copies timed (`e2e`), the
dominant kernel against its roofline, the fp64 oracle's speed on the host
cores (`cpu_baseline`) and the SM clocks seen during the timed region.
`--impl reference` times the fp64 oracle itself, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA query-tokens/s (top-k 2048, FP8 KV) and % of GB300 roofline"
UNIT = "query-tokens/s"
L2_FLUSH_BYTES = 512 << 20
NOMINAL_TFLOPS, NOMINAL_GBS = 2250.0, 8000.0
FALLBACK_GBS, FALLBACK_TFLOPS = 6800.0, 1900.0

# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture, keyed by the SHA-1 of the kernel sources it was taken on (reported
# as null once those sources change).
TRAFFIC_BY_SOURCE: dict[str, dict[str, int]] = {
    # mla_tc.cu + topk_row.cuh: the single-kernel path (--fused: top-k + attention)
    "a3ed308717ea26f427364930d9f7ab09e9d1a7d4": {"decode_64k_prefix99.9": 84_485_888},
    # mla_tc.cu: the attention kernel as its own call; verify_64k_8tok's figure is
    # the 19-request capture (152 query tokens, one wave) scaled by 128 / 19
    # requests: the requests share no rows, so the traffic grows in proportion
    "062c3281273413a49a357d84e58fbd63b9c04be3": {"decode_64k_prefix99.9": 49_795_840,
                                                 "verify_64k_8tok_19req": 191_791_872,
                                                 "verify_64k_8tok": 191_791_872 * 128 // 19},
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_64k_prefix99.9", help="the headline workload")
    ap.add_argument("--also", default="verify_64k_8tok",
                    help="further workloads measured in the same run (comma separated; '' for none)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the timed block of --steps passes until about this much timed load")
    ap.add_argument("--max-blocks", type=int, default=400)
    ap.add_argument("--fused", action="store_true",
                    help="run top-k and attention in one kernel where the shape allows (slower than the default "
                         "path on every workload measured)")
    ap.add_argument("--no-fused", action="store_true", help="the default path (kept for old commands)")
    ap.add_argument("--splits", type=int, default=0, help="KV splits (0 = library's rule)")
    ap.add_argument("--cpu-sample", type=int, default=64, help="query tokens the oracle baseline times")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="also write the raw clock samples to this CSV ({rank} is replaced by the rank)")
    ap.add_argument("--copy-streams", type=int, default=2,
                    help="copy streams of the end-to-end leg; q and scores are split over them by rows")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--l2-flush", choices=["write", "clean"], default="write",
                    help="before every timed step: write a 512 MiB buffer (write), or write it and then read a "
                         "second 512 MiB buffer so that L2 holds no dirty lines (clean)")
    ap.add_argument("--kv-write-rows", type=int, default=32768,
                    help="rows of the separate KV-write measurement (0 = skip)")
    return ap.parse_args()


def algorithmic(w, q_pos_host):
    """FLOPs and bytes of one pass, counted from the method's definition:
    per query token with k_eff = min(k, visible) selected rows,
    FLOPs = 2 H k_eff (dqk + d_latent); bytes of the attention step = gathered
    rows + scales + Q + O (bf16) + LSE + indices read; the top-k step reads the
    visible scores and writes k indices."""
    H, dqk, dl, k = w.heads, w.dqk, w.d_latent, w.k
    flops = bytes_fwd = bytes_topk = 0
    for p in q_pos_host:
        vis = int(p) + 1
        ke = min(k, vis)
        flops += 2 * H * ke * (dqk + dl)
        bytes_fwd += ke * (dqk + 4) + H * dqk * 2 + H * dl * 2 + H * 4 + ke * 4
        bytes_topk += vis * 4 + k * 4
    return flops, bytes_fwd, bytes_topk


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
    except Exception:
        return {"hbm_gbs": FALLBACK_GBS, "bf16_tflops": FALLBACK_TFLOPS, "bf16_tflops_sustained": None,
                "source": "fallback"}

    def find(pred):
        stack = [d]
        while stack:
            x = stack.pop()
            if isinstance(x, dict):
                for kk, v in x.items():
                    if isinstance(v, (int, float)) and pred(kk.lower()):
                        return float(v)
                    if isinstance(v, (dict, list)):
                        stack.append(v)
            elif isinstance(x, list):
                stack.extend(x)
        return None

    hbm = find(lambda s: "hbm" in s and ("gbs" in s or "gb_s" in s or "gbps" in s))
    bf = find(lambda s: "bf16" in s and "tflops" in s and "sustained" not in s)
    bfs = find(lambda s: "bf16" in s and "sustained" in s)
    return {"hbm_gbs": hbm or FALLBACK_GBS, "bf16_tflops": bf or FALLBACK_TFLOPS, "bf16_tflops_sustained": bfs,
            "source": "measured" if hbm else "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, out_path: str | None):
        self.uuid = uuid
        self.path = out_path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w") if self.path else subprocess.PIPE
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        if self.path:
            self.f.close()
            self.text = open(self.path).read()
        else:
            self.text = out or ""
        return False

    def summary(self):
        rows = []
        for line in self.text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's `value` (the job's time is its slowest
    rank's); `device` is where the collective's tensor lives."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank_step: int, steps: int, total_ms: float) -> float:
    """Units all ranks processed per second: every rank does the same work
    (weak scaling) and the job takes the slowest rank's time."""
    return world * units_per_rank_step * steps / (total_ms / 1e3)


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u.replace("GPU-", "")
    except Exception:
        return None


def run_oracle_sample(w, host, rows, nthreads=0):
    """Oracle top-k + attention over the given query tokens; returns seconds."""
    import numpy as np
    import oracle

    rows = np.asarray(rows)
    t0 = time.perf_counter()
    idx = oracle.topk(host["scores"][rows], host["q_pos"][rows], w.k, nthreads=nthreads)
    oracle.sparse_mla(host["q"][rows], host["kv"], host["kv_scale"], host["block_table"], host["q_req"][rows], idx,
                      d_latent=w.d_latent, d_rope=w.d_rope, page_size=w.page_size, softmax_scale=w.scale,
                      nthreads=nthreads)
    return time.perf_counter() - t0


def host_copies(inp):
    import torch
    return {"scores": inp.scores.cpu().numpy(), "q_pos": inp.q_pos.cpu().numpy(),
            "q": inp.q.view(torch.int16).cpu().numpy(), "kv": inp.kv.cpu().numpy(),
            "kv_scale": inp.kv_scale.cpu().numpy(), "block_table": inp.block_table.cpu().numpy(),
            "q_req": inp.q_req.cpu().numpy()}


def workload_config(w, splits, extra=None, l2="flushed (512 MiB write) before every timed step"):
    cfg = {"workload": w.name, "requests": w.num_req, "query_tokens": w.num_q, "heads": w.heads,
           "d_latent": w.d_latent, "d_rope": w.d_rope, "context": w.ctx, "shared_prefix": w.shared_prefix,
           "page_size": w.page_size, "top_k": w.k, "kv_splits": splits, "kv_dtype": "fp8_e4m3+fp32 scale/token",
           "l2": l2}
    if extra:
        cfg.update(extra)
    return cfg


def bench_reference(args):
    """The fp64 oracle timed on the host cores (rank 0 only)."""
    import numpy as np
    from dsa_sparse_mla_topk_gb300 import workloads as wl

    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = wl.lookup(args.workload)
    inp = wl.make_inputs(w, device="cpu")
    import torch
    host = host_copies(inp)
    n = min(w.num_q, max(1, args.cpu_sample // 4))
    rng = np.random.default_rng(0)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        run_oracle_sample(w, host, rng.choice(w.num_q, size=n, replace=False))
    total = 0.0
    for _ in range(args.steps):
        total += run_oracle_sample(w, host, np.sort(rng.choice(w.num_q, size=n, replace=False)))
    value = args.steps * n / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, 1, {"sample_query_tokens_per_step": n}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n} random query tokens of the workload per step (top-k + attention)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def prepare(w, dev, dsa, wl, args, torch):
    """Inputs, buffers and launch choices of one workload."""
    inp = wl.make_inputs(w, device=dev)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    S = args.splits or dsa.pick_num_splits(w.num_q, w.heads, w.d_latent, w.d_rope, w.k, num_sms)
    fused = args.fused and not args.no_fused and dsa.fused_path_supported(
        w.num_q, w.heads, w.d_latent, w.d_rope, inp.scores.shape[1], w.k, S)
    bufs = {"idx": torch.empty((w.num_q, w.k), dtype=torch.int32, device=dev),
            "out": torch.empty((w.num_q, w.heads, w.d_latent), dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((w.num_q, w.heads), dtype=torch.float32, device=dev)}
    if S > 1:
        bufs["o_part"] = torch.empty((S, w.num_q, w.heads, w.d_latent), dtype=torch.float32, device=dev)
        bufs["lse_part"] = torch.empty((S, w.num_q, w.heads), dtype=torch.float32, device=dev)
    ws_bytes = dsa.sparse_mla_workspace_size(w.num_q, w.heads, w.d_latent, w.d_rope, w.k)
    if ws_bytes:
        bufs["workspace"] = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    topk_ws = dsa.topk_workspace_size(w.num_q, inp.scores.shape[1], w.k)
    if topk_ws:
        bufs["topk_workspace"] = torch.empty(topk_ws, dtype=torch.uint8, device=dev)
    flops, bytes_fwd, bytes_topk = algorithmic(w, inp.q_pos.cpu().numpy())
    kw = dict(d_latent=w.d_latent, d_rope=w.d_rope, page_size=w.page_size, softmax_scale=w.scale)
    # kernels of this library launched by one pass
    two = not fused and dsa.two_kernel_path_supported(w.heads, w.d_latent, w.d_rope, inp.scores.shape[1])
    if fused:
        launches, path = 1, "fused"
    elif two:
        launches, path = 2 + (1 if S > 1 else 0), "two kernels (top-k with the page lookup, attention)"
    else:
        launches, path = (2 if topk_ws else 1) + (2 if ws_bytes else 1) + (1 if S > 1 else 0), "separate calls"
    return {"w": w, "inp": inp, "S": S, "fused": fused, "bufs": bufs, "kw": kw, "flops": flops,
            "bytes_fwd": bytes_fwd, "bytes_topk": bytes_topk, "launches": launches, "ws_bytes": ws_bytes,
            "path": path}


def one_pass(dsa, c, stream, status):
    """One pass of the whole path through the public call (top-k -> Partial
    -> Combine when split: on the tensor-core shape the top-k with the page
    lookup, then the attention kernel; top-k and Partial in one kernel on the
    fused path)."""
    w, inp = c["w"], c["inp"]
    dsa.sparse_mla_topk(inp.q, inp.kv, inp.kv_scale, inp.block_table, inp.q_req, inp.q_pos, inp.scores, w.k,
                        num_splits=c["S"], buffers=c["bufs"], dev_status=status, stream=stream, fused=c["fused"],
                        **c["kw"])


def separate_calls(dsa, c, stream, status, evs):
    """The same pass as separate calls with events between them: top-k,
    the attention call (resolve + Partial), the Combine."""
    w, inp, S, bufs, kw = c["w"], c["inp"], c["S"], c["bufs"], c["kw"]
    evs[0].record(stream)
    idx = dsa.topk_select(inp.scores, inp.q_pos, w.k, idx=bufs["idx"], dev_status=status, stream=stream,
                          workspace=bufs.get("topk_workspace"))
    evs[1].record(stream)
    if S == 1:
        dsa.sparse_mla_fwd(inp.q, inp.kv, inp.kv_scale, inp.block_table, inp.q_req, idx, num_splits=1, out=bufs["out"],
                           lse=bufs["lse"], workspace=bufs.get("workspace"), dev_status=status, stream=stream, **kw)
    else:
        dsa.sparse_mla_fwd(inp.q, inp.kv, inp.kv_scale, inp.block_table, inp.q_req, idx, num_splits=S,
                           o_part=bufs["o_part"], lse_part=bufs["lse_part"], workspace=bufs.get("workspace"),
                           dev_status=status, stream=stream, **kw)
    evs[2].record(stream)
    if S > 1:
        dsa.combine(bufs["o_part"], bufs["lse_part"], out=bufs["out"], lse=bufs["lse"], stream=stream)
    evs[3].record(stream)


class L2Flush:
    """Evicts the step's inputs from L2 before every timed step.  "write"
    writes L2_FLUSH_BYTES; "clean" then also reads a second buffer of that
    size, so that the lines left in L2 are clean and the timed step does not
    pay for writing the flush's own data back to HBM."""

    def __init__(self, torch, dev, mode):
        self.torch, self.mode = torch, mode
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        if mode == "clean":
            self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
            self.acc = torch.zeros((), dtype=torch.int64, device=dev)

    def describe(self):
        return ("flushed (512 MiB write) before every timed step" if self.mode == "write" else
                "flushed (512 MiB write, then a 512 MiB read: no dirty lines left) before every timed step")

    def zero_(self):
        self.w.zero_()
        if self.mode == "clean":
            self.torch.sum(self.r, 0, out=self.acc)


def measure(dsa, c, args, torch, dev, stream, status, flush, world, barrier, peaks):
    """Time exactly K = args.steps passes per block, L2 flushed before every
    pass, blocks repeated until about args.min_seconds of timed load; then the
    separate calls once more for the per-kernel breakdown.  Returns the
    workload's report."""
    w = c["w"]
    K = args.steps
    for _ in range(args.warmup):
        flush.zero_()
        one_pass(dsa, c, stream, status)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    def block():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        barrier()
        for s in range(K):
            flush.zero_()
            evs[s][0].record(stream)
            one_pass(dsa, c, stream, status)
            evs[s][1].record(stream)
        barrier()
        return [a.elapsed_time(b) for a, b in evs]

    t0 = time.perf_counter()
    first = block()
    wall = max_over_ranks(time.perf_counter() - t0, world, dev)
    nblocks = max(1, min(args.max_blocks, int(max_over_ranks(args.min_seconds / max(wall, 1e-6), world, dev)) + 1))
    per_block, step_ms = [], []
    for _ in range(nblocks):
        ms = block()
        step_ms += ms
        per_block.append(max_over_ranks(sum(ms), world, dev))
    del first
    block_ms = statistics.median(per_block)
    value = whole_job_rate(world, w.num_q, K, block_ms)
    ms_per_step = block_ms / K

    # per-kernel breakdown from the separate calls (the fused path runs them as one kernel)
    comp = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(max(10, K))]
    for e in comp:
        flush.zero_()
        separate_calls(dsa, c, stream, status, e)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    t_topk = statistics.median(e[0].elapsed_time(e[1]) for e in comp)
    t_fwd = statistics.median(e[1].elapsed_time(e[2]) for e in comp)
    t_comb = statistics.median(e[2].elapsed_time(e[3]) for e in comp)
    t_sep = statistics.median(e[0].elapsed_time(e[3]) for e in comp)

    flops, bytes_fwd, bytes_topk = c["flops"], c["bytes_fwd"], c["bytes_topk"]
    bytes_path = bytes_fwd + bytes_topk
    ai_path = flops / bytes_path
    ns_roof = min(NOMINAL_TFLOPS * 1e12, NOMINAL_GBS * 1e9 * ai_path)
    meas_roof = min(peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9 * ai_path)
    achieved_flops = flops / (ms_per_step / 1e3)
    src_files = ["mla_tc.cu", "topk_row.cuh"] if c["fused"] else ["mla_tc.cu"]
    sha = hashlib.sha1(b"".join(open(os.path.join(ROOT, "dsa_sparse_mla_topk_gb300", "csrc", f), "rb").read()
                                for f in src_files)).hexdigest()
    traffic = TRAFFIC_BY_SOURCE.get(sha, {}).get(w.name)
    if c["fused"]:
        # the one kernel is the whole pass: its algorithmic bytes are the pass's
        kern, kbytes, kms = "sparse_mla_topk_fwd (top-k + attention, one kernel)", bytes_path, ms_per_step
    else:
        kern, kbytes, kms = "sparse_mla_fwd (resolve + attention)", bytes_fwd, t_fwd
    achieved_gbs = kbytes / (kms / 1e3) / 1e9
    att_ms = t_fwd + (t_comb if c["S"] > 1 else 0.0)
    return {
        "workload": w.name, "value": value, "unit": UNIT, "query_tokens": w.num_q, "steps": K, "blocks": nblocks,
        "ms_per_step": ms_per_step,
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms),
                    "count": len(step_ms)},
        "path": c["path"], "kv_splits": c["S"],
        "gpu_launches_per_step": c["launches"],
        "roofline": {"kernel": kern, "bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": peaks["source"], "algorithmic_bytes_per_launch": kbytes, "avg_launch_ms": kms,
                     "achieved_tflops": flops / (kms / 1e3) / 1e12},
        "path_roofline": {"ai_flops_per_byte": ai_path, "achieved_tflops": achieved_flops / 1e12,
                          "frac_nominal": achieved_flops / ns_roof, "frac_measured": achieved_flops / meas_roof,
                          "nominal_roofline_tflops": ns_roof / 1e12},
        "kernel_ms_separate_calls": {"topk": t_topk, "sparse_mla_fwd": t_fwd, "combine": t_comb, "pass": t_sep},
        "attention_only": {"value": w.num_q / (att_ms / 1e3), "unit": UNIT,
                           "note": "the attention call (resolve + Partial) plus the Combine when split, timed as "
                                   "separate calls with L2 flushed",
                           "achieved_gbs": bytes_fwd / (att_ms / 1e3) / 1e9,
                           "frac_hbm": bytes_fwd / (att_ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
    }


def bench_ours(args):
    import numpy as np
    import torch

    import dsa_sparse_mla_topk_gb300 as dsa
    from dsa_sparse_mla_topk_gb300 import build as lib_build
    from dsa_sparse_mla_topk_gb300 import workloads as wl

    world, rank, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lib_build.build()
    dsa.load_library()
    peaks = read_peaks()

    names = [args.workload] + [n for n in args.also.split(",") if n and n != args.workload]
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(torch, dev, args.l2_flush)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    clock_path = args.clocks_csv.format(rank=rank) if args.clocks_csv else None
    sampler = ClockSampler(gpu_uuid(torch, dev), clock_path) if not args.no_clocks else None
    reports = {}
    head = None
    if sampler:
        sampler.__enter__()
    wall0 = time.perf_counter()
    for n in names:
        c = prepare(wl.lookup(n), dev, dsa, wl, args, torch)
        reports[n] = measure(dsa, c, args, torch, dev, stream, status, flush, world, barrier, peaks)
        if head is None:
            head = c
        else:
            del c
            torch.cuda.empty_cache()
    wall = time.perf_counter() - wall0
    if sampler:
        sampler.__exit__(None, None, None)
    w, inp, S, bufs, kw = head["w"], head["inp"], head["S"], head["bufs"], head["kw"]
    rep = reports[w.name]

    # ---- end to end through host buffers: copies timed every step ----
    # Every step copies its own inputs from pinned host memory and reads its
    # own out + lse back.  As in a serving loop, step i+1's input copies run on
    # two copy streams while step i computes; inputs and outputs are double
    # buffered, and L2 is still flushed before every step's compute.
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "scores", "q_pos", "q_req", "block_table")
        pin = {n: getattr(inp, n).cpu().pin_memory() for n in names_in}
        NB = 2
        dsts = [{n: torch.empty_like(getattr(inp, n)) for n in names_in} for _ in range(NB)]
        outs = [torch.empty_like(bufs["out"]) for _ in range(NB)]
        lses = [torch.empty_like(bufs["lse"]) for _ in range(NB)]
        idxs = [torch.empty_like(bufs["idx"]) for _ in range(NB)]
        out_h = [torch.empty(bufs["out"].shape, dtype=bufs["out"].dtype).pin_memory() for _ in range(NB)]
        lse_h = [torch.empty(bufs["lse"].shape, dtype=bufs["lse"].dtype).pin_memory() for _ in range(NB)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = out_h[0].numel() * out_h[0].element_size() + lse_h[0].numel() * lse_h[0].element_size()
        cs = [torch.cuda.Stream(dev) for _ in range(max(1, args.copy_streams))]

        def rows_of(t, ci):  # stream ci's share of tensor t's rows
            nrow = t.shape[0]
            return slice(nrow * ci // len(cs), nrow * (ci + 1) // len(cs))

        def ev():
            return torch.cuda.Event(enable_timing=True)

        def pipeline(nsteps):
            h2d_done = [[ev() for _ in cs] for _ in range(nsteps)]
            comp_done = [ev() for _ in range(nsteps)]
            d2h_done = [ev() for _ in range(nsteps)]

            def issue_h2d(i):
                b = i % NB
                for ci, stream_c in enumerate(cs):
                    if i >= NB:
                        stream_c.wait_event(comp_done[i - NB])  # that step's compute has read these inputs
                    with torch.cuda.stream(stream_c):
                        for n in names_in:
                            if n in ("q", "scores"):
                                r = rows_of(pin[n], ci)
                                dsts[b][n][r].copy_(pin[n][r], non_blocking=True)
                            elif ci == 0:
                                dsts[b][n].copy_(pin[n], non_blocking=True)
                    h2d_done[i][ci].record(stream_c)

            start, end = ev(), ev()
            start.record(cs[0])
            for stream_c in cs[1:]:
                stream_c.wait_event(start)
            issue_h2d(0)
            for i in range(nsteps):
                b = i % NB
                if i + 1 < nsteps:
                    issue_h2d(i + 1)
                for ci in range(len(cs)):
                    stream.wait_event(h2d_done[i][ci])
                if i >= NB:
                    stream.wait_event(d2h_done[i - NB])  # that step's outputs have been read back
                flush.zero_()
                d = dsts[b]
                sb = dict(bufs, out=outs[b], lse=lses[b], idx=idxs[b])
                out, lse, _ = dsa.sparse_mla_topk(d["q"], inp.kv, inp.kv_scale, d["block_table"], d["q_req"],
                                                  d["q_pos"], d["scores"], w.k, num_splits=S, buffers=sb,
                                                  dev_status=status, stream=stream, fused=head["fused"], **kw)
                comp_done[i].record(stream)
                cs[0].wait_event(comp_done[i])
                with torch.cuda.stream(cs[0]):
                    out_h[b].copy_(out, non_blocking=True)
                    lse_h[b].copy_(lse, non_blocking=True)
                d2h_done[i].record(cs[0])
            end.record(cs[0])
            end.synchronize()
            return start.elapsed_time(end)

        pipeline(max(2, args.warmup))
        barrier()
        e_ms = max_over_ranks(pipeline(args.steps), world, dev)
        # the pipelined results are the device-timed pass's, bit for bit
        one_pass(dsa, head, stream, status)
        torch.cuda.synchronize(dev)
        last = (args.steps - 1) % NB
        if not (torch.equal(out_h[last], bufs["out"].cpu()) and torch.equal(lse_h[last], bufs["lse"].cpu())):
            raise RuntimeError("end-to-end outputs differ from the device-timed pass")
        e2e = {"value": whole_job_rate(world, w.num_q, args.steps, e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps,
               "note": "KV cache resident in HBM; every step copies its inputs (q, scores, q_pos, q_req, block "
                       "table) from pinned host memory and reads out + lse back inside the timed region; step "
                       "i+1's input copies overlap step i's compute (double buffers, copies split over "
                       f"{len(cs)} copy streams); L2 flushed before every step's compute"}
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # ---- the KV cache write path (a separate measurement, not in the step):
    # n new bf16 rows quantised to FP8 and scattered through the block table,
    # timed per call with the L2 flushed before each ----
    kvw = None
    if args.kv_write_rows > 0 and w.heads == 64:
        n = args.kv_write_rows
        g = torch.Generator(device=dev).manual_seed(5)
        rows = torch.randn((n, w.dqk), generator=g, device=dev).to(torch.bfloat16)
        kv_w = torch.zeros_like(inp.kv)
        sc_w = torch.zeros_like(inp.kv_scale)
        slots = inp.kv.shape[0]
        perm = torch.randperm(slots, generator=g, device=dev)[:n].to(torch.int32)
        bt_w = torch.arange(slots // w.page_size, dtype=torch.int32, device=dev)[None, :]
        req_w = torch.zeros(n, dtype=torch.int32, device=dev)
        for _ in range(max(1, args.warmup)):
            dsa.kv_write(rows, req_w, perm, bt_w, kv_w, sc_w, page_size=w.page_size, dev_status=status, stream=stream)
        t_kvw = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dsa.kv_write(rows, req_w, perm, bt_w, kv_w, sc_w, page_size=w.page_size, dev_status=status, stream=stream)
            b.record(stream)
            b.synchronize()
            t_kvw.append(a.elapsed_time(b))
        ms = statistics.median(t_kvw)
        kbytes = n * (w.dqk * 2 + 4 + w.dqk + 4 + 4)  # rows read, req + pos read, codes + scale written
        kvw = {"rows": n, "ms": ms, "rows_per_s": n / (ms / 1e3), "algorithmic_bytes": kbytes,
               "achieved_gbs": kbytes / (ms / 1e3) / 1e9, "bound": "hbm", "peak_gbs": peaks["hbm_gbs"],
               "frac": kbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
               "note": "random distinct slots of the workload's pool; L2 flushed before every call; median"}
        torch.cuda.synchronize(dev)
        assert int(status.item()) == 0, f"device status {int(status.item())}"

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        host = host_copies(inp)
        n = min(w.num_q, args.cpu_sample)
        rows = np.sort(np.random.default_rng(0).choice(w.num_q, size=n, replace=False))
        secs = run_oracle_sample(w, host, rows)
        cpu = {"value": n / secs, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
               "sample": f"{n} of {w.num_q} query tokens (seeded), top-k + attention, fp64 C on all host cores",
               "seconds": secs}

    line = {"metric": METRIC, "value": rep["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rep["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded; shapes of the GLM-5.3-Flash workloads)",
            "config": workload_config(w, S, l2=flush.describe(), extra={"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                             "path": rep["path"],
                                             "timing": f"{rep['blocks']} blocks of exactly {args.steps} passes; "
                                                       "value and ms_per_step from the median block"}),
            "roofline": rep["roofline"], "path_roofline": rep["path_roofline"], "step_ms": rep["step_ms"],
            "kernel_ms": rep["kernel_ms_separate_calls"], "attention_only": rep["attention_only"],
            "workloads": reports, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": rep["gpu_launches_per_step"] * args.steps * rep["blocks"],
            "kv_write": kvw, "clocks": sampler.summary() if sampler else None, "wall_s": wall}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return bench_reference(args)
    return bench_ours(args)


if __name__ == "__main__":
    sys.exit(main())
