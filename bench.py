"""Benchmark: batched byte-level BPE encoding on GB300.

Default workload: the serving batch — 4,194,304 ASCII documents of 64-448
bytes (about 1 GiB), a merge table trained on a 32 MiB corpus of the same
generator. A step is one bpe_encode_batch call over the whole batch (split,
byte -> symbol, merge loop, id output, per-document offsets), inputs resident
in HBM. The input is far larger than L2, so no flush is needed between steps.

Prints one JSON line. ``--impl reference`` times the CPU oracle instead (a
bounded sample of the same workload on the host cores).

Multi-GPU: one process per GPU under torchrun; every rank encodes its own
distinct documents (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "encoded input MB/s and tokens/s on 1 GB300; achieved HBM GB/s vs peak"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "k_encode_serving_batch.md")
KERNEL_SRC = os.path.join(ROOT, "byte_level_bpe_pretokenize_gb300", "csrc", "bpe_kernels.cu")


def kernel_hash() -> str:
    return hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_from_profile():
    """dram bytes per launch of the encode kernel from the committed ncu
    summary, when it was taken on the current kernel source."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    kv = {}
    for line in open(PROFILE_SUMMARY):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    if kv.get("kernel_source_sha256_16") != kernel_hash():
        return None
    try:
        return int(float(kv["dram_bytes_per_full_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard(cfg: int, rank: int, n_docs: int | None = None) -> tuple[int, int]:
    """(first document, count) a rank encodes: every rank takes a full
    workload's worth of its own documents of the same generator (weak
    scaling; no data is exchanged between ranks)."""
    n = n_docs or workloads.n_docs(cfg)
    return rank * n, n


def load_workload(cfg: int, rank: int, n_docs: int | None = None):
    first, n = shard(cfg, rank, n_docs)
    data, offsets = workloads.docs(cfg, first, n)
    merges, vb, vo = workloads.table(cfg)
    return data, offsets, merges, vb, vo


def reduce_ranks(dist, device, times: list[float], counts: list[float]) -> tuple[list[float], list[float]]:
    """Max over ranks of each time, sum over ranks of each count (a no-op
    without a process group)."""
    if dist is None:
        return list(times), list(counts)
    import torch
    t = torch.tensor(times, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    c = torch.tensor(counts, dtype=torch.float64, device=device)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return t.tolist(), c.tolist()


def algorithmic_bytes(n_bytes: int, n_docs: int, n_tokens: int) -> int:
    # input bytes + doc offsets read; int32 ids + int64 doc offsets written
    return n_bytes + 8 * (n_docs + 1) + 4 * n_tokens + 8 * (n_docs + 1)


def oracle_sample(cfg: int, data, offsets, merges, vb, vo, budget_s: float, gpu_ids=None, gpu_off=None):
    """Time the oracle on whole documents from the start of the batch until
    about budget_s of CPU time; optionally check those documents against the
    GPU output."""
    import oracle
    o = oracle.Oracle(merges, vb, vo)
    n_docs = len(offsets) - 1
    done, nbytes, ntok, t_used = 0, 0, 0, 0.0
    step = 64
    mismatch = 0
    while done < n_docs and t_used < budget_s:
        cnt = min(step, n_docs - done)
        t0 = time.perf_counter()
        ids, ioff = o.encode_batch(data, offsets, done, cnt)
        t_used += time.perf_counter() - t0
        if gpu_ids is not None:
            g = gpu_ids[gpu_off[done]:gpu_off[done + cnt]]
            if not np.array_equal(g, ids) or not np.array_equal(gpu_off[done:done + cnt + 1] - gpu_off[done], ioff):
                mismatch += 1
        nbytes += int(offsets[done + cnt] - offsets[done])
        ntok += len(ids)
        done += cnt
        step = min(step * 2, 4096)
    return {"docs": done, "bytes": nbytes, "tokens": ntok, "seconds": t_used, "mismatched_groups": mismatch}


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = args.cfg
    n = workloads.n_docs(cfg)
    # A bounded sample per step: the first documents of the batch.
    lens = workloads.doc_lengths(cfg, 0, min(n, 200_000))
    data, offsets = workloads.docs(cfg, 0, len(lens))
    merges, vb, vo = workloads.table(cfg)
    per_step = max(0.5, args.reference_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(cfg, data, offsets, merges, vb, vo, per_step)
    rates, trates, samples = [], [], []
    for _ in range(args.steps):
        s = oracle_sample(cfg, data, offsets, merges, vb, vo, per_step)
        rates.append(s["bytes"] / s["seconds"] / 1e6)
        trates.append(s["tokens"] / s["seconds"])
        samples.append(s)
    v = statistics.median(rates)
    out = {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "MB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * statistics.median([s["seconds"] for s in samples]), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "tokens_per_s": round(statistics.median(trates), 1),
        "config": {"workload": workloads.NAMES[cfg], "n_docs_sampled": samples[-1]["docs"],
                   "bytes_sampled": samples[-1]["bytes"], "merges": int(len(merges))},
        "cpu_baseline": {"value": round(v, 3), "unit": "MB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {samples[-1]['docs']} documents ({samples[-1]['bytes']} bytes) of the "
                                   f"workload per step, single-threaded"},
        "e2e": {"value": round(v, 3), "unit": "MB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_gpu(args, world, rank, local):
    import torch
    import byte_level_bpe_pretokenize_gb300 as bpe

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()

    cfg = args.cfg
    data, offsets, merges, vb, vo = load_workload(cfg, rank, args.n_docs)
    n_bytes, n_docs = int(data.size), int(len(offsets) - 1)
    handle = bpe.bpe_build(merges, vb, vo, local)
    stream = torch.cuda.current_stream()
    s_ptr = stream.cuda_stream

    d_data = torch.from_numpy(data).to(dev)
    d_off = torch.from_numpy(offsets).to(dev)
    d_ids = torch.empty(n_bytes, dtype=torch.int32, device=dev)
    d_out = torch.empty(n_docs + 1, dtype=torch.int64, device=dev)

    def step(want_total=False):
        return bpe.bpe_encode_batch(handle, d_data.data_ptr(), n_bytes, d_off.data_ptr(), n_docs, d_ids.data_ptr(),
                                    n_bytes, d_out.data_ptr(), want_total, s_ptr)

    n_tokens = step(True)
    for _ in range(max(0, args.warmup - 1)):
        step()
    bpe.bpe_sync_status(handle, s_ptr)

    # Timed region: K steps; the encode kernel is timed by its own event pair.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:  # materialise the CUDA events
        a.record(stream)
        b.record(stream)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local)
    if rank == 0:
        clocks.start()
        time.sleep(0.5)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for a, b in ev:
        bpe.bpe_set_timing_events(handle, a.cuda_event, b.cuda_event)
        step()
    t_end.record(stream)
    bpe.bpe_set_timing_events(handle, None, None)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    bpe.bpe_sync_status(handle, s_ptr)
    step_ms = t_start.elapsed_time(t_end) / args.steps
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # Secondary: the same steps with the word cache off (every pre-token runs
    # the merge loop), timed the same way, outside the headline region.
    bpe.bpe_set_word_cache(handle, False)
    step()
    nc0, nc1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nc_steps = max(1, min(args.steps, 3))
    torch.cuda.synchronize()
    nc0.record(stream)
    for _ in range(nc_steps):
        step()
    nc1.record(stream)
    torch.cuda.synchronize()
    nocache_ms = nc0.elapsed_time(nc1) / nc_steps
    bpe.bpe_set_word_cache(handle, True)
    bpe.bpe_sync_status(handle, s_ptr)

    # End to end through the C ABI's host-buffer call: page-locked host input,
    # copies in, encode and copies out of ids and offsets, pipelined in slices
    # inside bpe_encode_batch_host; one untimed call first sizes its buffers.
    h_data = torch.from_numpy(data).pin_memory()
    h_off = torch.from_numpy(offsets).pin_memory()
    h_ids = torch.empty(n_bytes, dtype=torch.int32).pin_memory()
    h_out = torch.empty(n_docs + 1, dtype=torch.int64).pin_memory()

    def host_step():
        return bpe.bpe_encode_batch_host(handle, h_data.data_ptr(), n_bytes, h_off.data_ptr(), n_docs,
                                         h_ids.data_ptr(), n_bytes, h_out.data_ptr(), True, s_ptr)

    if host_step() != n_tokens:
        raise RuntimeError("host-buffer call gave a different token count")
    e2e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_step()
    e2e_s = (time.perf_counter() - e0) / e2e_steps
    (step_ms, kern_ms, e2e_s), (all_bytes, all_tokens, all_docs) = reduce_ranks(
        dist, dev, [step_ms, kern_ms, e2e_s], [n_bytes, n_tokens, n_docs])

    out = None
    if rank == 0:
        peak, peak_kind = peaks()
        alg = algorithmic_bytes(n_bytes, n_docs, n_tokens)
        achieved = alg / (kern_ms / 1e3) / 1e9
        value = all_bytes / (step_ms / 1e3) / 1e6
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            g_ids = d_ids[:n_tokens].cpu().numpy()
            g_off = d_out.cpu().numpy()
            s = oracle_sample(cfg, data, offsets, merges, vb, vo, args.cpu_budget, g_ids, g_off)
            cpu = {"value": round(s["bytes"] / s["seconds"] / 1e6, 3), "unit": "MB/s", "cores": 1,
                   "kind": "oracle",
                   "sample": f"first {s['docs']} documents ({s['bytes']} bytes) of the same batch, single-threaded",
                   "tokens_per_s": round(s["tokens"] / s["seconds"], 1),
                   "parity_vs_gpu": "identical" if s["mismatched_groups"] == 0 else
                   f"{s['mismatched_groups']} groups differ"}
        out = {
            "metric": METRIC, "value": round(value, 3), "unit": "MB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "tokens_per_s": round(all_tokens / (step_ms / 1e3), 1),
            "hbm_gbs_achieved": round(achieved, 2),
            "config": {"workload": workloads.NAMES[cfg], "n_docs": n_docs, "n_bytes": n_bytes,
                       "tokens": int(n_tokens), "merges": int(len(merges)), "n_vocab": int(len(vo) - 1),
                       "l2": (f"inputs ({n_bytes / 2**20:.0f} MiB) larger than L2 (129 MB); no flush" if n_bytes > 129e6 else f"inputs ({n_bytes / 2**20:.0f} MiB) fit in L2: a profiling case, not a bench number"), "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                         "kernel": "k_pretokenize..k_compact", "kernel_ms": round(kern_ms, 4),
                         "algorithmic_bytes_per_launch": alg, "traffic": traffic_from_profile()},
            "cpu_baseline": cpu,
            "e2e": {"value": round(all_bytes / e2e_s / 1e6, 3),
                    "unit": "MB/s", "h2d_bytes_per_step": n_bytes + 8 * (n_docs + 1),
                    "d2h_bytes_per_step": 4 * int(n_tokens) + 8 * (n_docs + 1)},
            "without_word_cache": {"value": round(n_bytes / (nocache_ms / 1e3) / 1e6, 3), "unit": "MB/s",
                                   "ms_per_step": round(nocache_ms, 4),
                                   "hbm_frac": round(alg / (nocache_ms / 1e3) / 1e9 / peak, 4)},
            "gpu_launches": 7 * args.steps,
            "clocks": clk,
        }
        print(json.dumps(out), flush=True)
    bpe.bpe_destroy(handle)
    if dist:
        dist.destroy_process_group()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cfg", type=int, default=5, help="workload 1..5 (5 = serving batch)")
    ap.add_argument("--n-docs", type=int, default=None, help="fewer documents (small profiling cases only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--reference-budget", type=float, default=60.0, help="total oracle seconds for --impl reference")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
