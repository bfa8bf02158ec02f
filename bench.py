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
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic_serving_batch.json")
KERNEL_SPAN = "k_prep_docs..k_giant_copy"
LAUNCHES_PER_CALL = 9
KERNEL_SRC = [os.path.join(ROOT, "byte_level_bpe_pretokenize_gb300", "csrc", f)
              for f in ("bpe_kernels.cu", "tiles.cuh", "memo.cuh", "decode.cuh", "train.cuh", "class_table.inc")]


def kernel_hash() -> str:
    """Hash of the kernel sources (the translation unit and what it includes),
    comments and blank space left out, so that a change to a comment keeps a
    profile taken on the same code."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SRC:
        text = open(f, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_from_profile():
    """DRAM bytes per full call of the timed kernels, from the committed ncu
    summary (profiles/traffic_serving_batch.json), when it was taken on the
    current kernel source; None otherwise."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    try:
        d = json.load(open(TRAFFIC_JSON))
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256_16") != kernel_hash():
        return None
    v = d.get("dram_bytes_per_full_call")
    return int(v) if v is not None else None


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
    """Time the single-threaded oracle on whole documents from the start of
    the batch until about budget_s of CPU time; optionally check those
    documents against the GPU output."""
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


def slice_docs(offsets: np.ndarray, max_bytes: int) -> int:
    """Number of whole documents from the start whose bytes fit in max_bytes."""
    return max(1, int(np.searchsorted(offsets, offsets[0] + max_bytes, side="right")) - 1)


def run_reference(args, world, rank):
    """The reference arm: the oracle on every host core (one pinned process
    per physical core over byte-balanced document shards), each step a
    bounded slice of the same workload."""
    if rank != 0:
        return
    from oracle import sharded
    cfg = args.cfg
    n = workloads.n_docs(cfg)
    lens = workloads.doc_lengths(cfg, 0, min(n, 600_000))
    offs = np.zeros(len(lens) + 1, dtype=np.int64)
    np.cumsum(lens, out=offs[1:])
    k = min(len(lens), slice_docs(offs, args.reference_slice_mib << 20))
    data, offsets = workloads.docs(cfg, 0, k)
    merges, vb, vo = workloads.table(cfg)
    for _ in range(args.warmup):
        sharded.encode(merges, vb, vo, data, offsets)
    walls, tok = [], 0
    r = None
    for _ in range(args.steps):
        r = sharded.encode(merges, vb, vo, data, offsets)
        walls.append(r["wall_s"])
        tok = len(r["ids"])
    wall = statistics.median(walls)
    v = data.size / wall / 1e6
    sample = (f"first {k} documents ({data.size} bytes) of the workload per step, on {r['procs']} pinned "
              f"single-threaded oracle processes ({r['cpu_model']})")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "MB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * wall, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "tokens_per_s": round(tok / wall, 1),
        "config": {"workload": workloads.NAMES[cfg], "n_docs_sampled": k, "bytes_sampled": int(data.size),
                   "merges": int(len(merges))},
        "cpu_baseline": {"value": round(v, 3), "unit": "MB/s", "cores": r["procs"], "kind": "oracle",
                         "sample": sample, "cpu_model": r["cpu_model"]},
        "e2e": {"value": round(v, 3), "unit": "MB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


class Encoder:
    """One workload resident on the GPU with its handle and output buffers."""

    def __init__(self, bpe, cfg, dev, local, rank=0, n_docs=None):
        import torch
        self.bpe, self.cfg = bpe, cfg
        self.data, self.offsets, self.merges, self.vb, self.vo = load_workload(cfg, rank, n_docs)
        self.n_bytes, self.n_docs = int(self.data.size), int(len(self.offsets) - 1)
        self.handle = bpe.bpe_build(self.merges, self.vb, self.vo, local)
        self.stream = torch.cuda.current_stream()
        self.d_data = torch.from_numpy(self.data).to(dev)
        self.d_off = torch.from_numpy(self.offsets).to(dev)
        self.d_ids = torch.empty(max(1, self.n_bytes), dtype=torch.int32, device=dev)
        self.d_out = torch.empty(self.n_docs + 1, dtype=torch.int64, device=dev)
        self.n_tokens = self.step(True)

    def step(self, want_total=False):
        return self.bpe.bpe_encode_batch(self.handle, self.d_data.data_ptr(), self.n_bytes, self.d_off.data_ptr(),
                                         self.n_docs, self.d_ids.data_ptr(), self.n_bytes, self.d_out.data_ptr(),
                                         want_total, self.stream.cuda_stream)

    def time_calls(self, steps, warmup):
        """CUDA-event time (ms) of each of `steps` calls after `warmup`."""
        import torch
        for _ in range(warmup):
            self.step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(self.stream)
            self.step()
            b.record(self.stream)
        torch.cuda.synchronize()
        self.bpe.bpe_sync_status(self.handle, self.stream.cuda_stream)
        return [a.elapsed_time(b) for a, b in ev]

    def kernel_ms(self, calls=3):
        """Per-kernel CUDA-event time of a call (median over `calls`), from
        events recorded before the first kernel and after each."""
        import torch
        bpe = self.bpe
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(bpe.ENCODE_LAUNCHES + 1)]
        for e in evs:  # materialise the CUDA events
            e.record(self.stream)
        pe = bpe.PhaseEvents([e.cuda_event for e in evs])
        per = []
        try:
            bpe.bpe_set_phase_events(self.handle, pe)
            for _ in range(calls):
                torch.cuda.synchronize()
                self.step()
                torch.cuda.synchronize()
                per.append([evs[i].elapsed_time(evs[i + 1]) for i in range(bpe.ENCODE_LAUNCHES)])
        finally:
            bpe.bpe_set_phase_events(self.handle, None)
        return {k: round(statistics.median(p[i] for p in per), 4) for i, k in enumerate(bpe.ENCODE_KERNELS)}

    def result(self):
        return self.d_ids[:self.n_tokens].cpu().numpy(), self.d_out.cpu().numpy()

    def close(self):
        self.bpe.bpe_destroy(self.handle)


def config_line(enc: "Encoder", ms: float, peak: float) -> dict:
    alg = algorithmic_bytes(enc.n_bytes, enc.n_docs, enc.n_tokens)
    return {"workload": workloads.NAMES[enc.cfg], "n_docs": enc.n_docs, "n_bytes": enc.n_bytes,
            "tokens": int(enc.n_tokens), "merges": int(len(enc.merges)), "ms_per_call": round(ms, 4),
            "input_mb_per_s": round(enc.n_bytes / (ms / 1e3) / 1e6, 3),
            "tokens_per_s": round(enc.n_tokens / (ms / 1e3), 1),
            "hbm_gbs_achieved": round(alg / (ms / 1e3) / 1e9, 2), "frac": round(alg / (ms / 1e3) / 1e9 / peak, 4),
            "algorithmic_bytes": alg}


def parity_line(enc: "Encoder", gpu_ids, gpu_off) -> tuple[dict, dict]:
    """The whole batch through the all-core oracle, compared id for id."""
    from oracle import sharded
    r = sharded.encode(enc.merges, enc.vb, enc.vo, enc.data, enc.offsets)
    same = bool(np.array_equal(gpu_ids, r["ids"]) and np.array_equal(gpu_off, r["offsets"]))
    line = {"fnv1a64_gpu": f"{workloads.fnv1a64(gpu_ids):016x}", "fnv1a64_oracle": f"{workloads.fnv1a64(r['ids']):016x}",
            "docs_compared": enc.n_docs, "identical": same}
    return line, r


def decode_line(bpe, enc: "Encoder", steps: int, peak: float) -> dict:
    """bpe_decode_batch on the encoded batch (ids resident in HBM): CUDA-event
    time per call (median after 3 warm-up calls), algorithmic bytes (ids and
    id offsets read, bytes and byte offsets written), and whether the bytes
    and offsets equal the input."""
    import torch
    dev = enc.d_ids.device
    n_tok = int(enc.n_tokens)
    out = torch.empty(enc.n_bytes + 64, dtype=torch.uint8, device=dev)
    out_off = torch.empty(enc.n_docs + 1, dtype=torch.int64, device=dev)
    s = enc.stream.cuda_stream

    def call(want=False):
        return bpe.bpe_decode_batch(enc.handle, enc.d_ids.data_ptr(), n_tok, enc.d_out.data_ptr(), enc.n_docs,
                                    out.data_ptr(), out.numel(), out_off.data_ptr(), want, s)

    total = call(True)
    same = bool(total == enc.n_bytes and torch.equal(out[:total], enc.d_data)
                and np.array_equal(out_off.cpu().numpy(), enc.offsets))
    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(enc.stream)
        call()
        b.record(enc.stream)
    torch.cuda.synchronize()
    bpe.bpe_sync_status(enc.handle, s)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    alg = 4 * n_tok + 8 * (enc.n_docs + 1) + enc.n_bytes + 8 * (enc.n_docs + 1)
    ach = alg / (ms / 1e3) / 1e9
    return {"ms_per_call": round(ms, 4), "output_mb_per_s": round(enc.n_bytes / (ms / 1e3) / 1e6, 3),
            "tokens_per_s": round(n_tok / (ms / 1e3), 1),
            "roofline": {"bound": "hbm", "achieved": round(ach, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(ach / peak, 4), "algorithmic_bytes_per_launch": alg,
                         "kernel": "k_dec_count..k_dec_write"},
            "round_trip_identical": same, "gpu_launches_per_call": 5}


def train_line(bpe, cfg: int, local: int) -> dict:
    """bpe_train on the trainer word list of a workload's corpus: wall time of
    the call (host arrays in, merge rows out), and whether its table equals
    the host trainer's."""
    import torch
    data, offsets, counts = workloads.train_words(workloads.corpus(cfg))
    want = workloads.table(cfg)[0]
    bpe.bpe_train(data[:64], np.array([0, min(64, data.size)], np.int64), np.ones(1, np.int64), 4, local)  # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    got = bpe.bpe_train(data, offsets, counts, workloads.n_merges(cfg), local)
    wall = time.perf_counter() - t0
    return {"workload": f"trainer word list of {workloads.NAMES[cfg]}'s corpus", "words": int(len(counts)),
            "word_bytes": int(data.size), "merges": int(len(got)), "seconds": round(wall, 3),
            "merges_per_s": round(len(got) / wall, 1),
            "identical_to_host_trainer": bool(got.shape == want.shape and np.array_equal(got, want))}


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
    enc = Encoder(bpe, cfg, dev, local, rank, args.n_docs)
    handle, stream, n_bytes, n_docs, n_tokens = enc.handle, enc.stream, enc.n_bytes, enc.n_docs, enc.n_tokens
    s_ptr = stream.cuda_stream
    data, offsets = enc.data, enc.offsets
    for _ in range(max(0, args.warmup - 1)):
        enc.step()
    bpe.bpe_sync_status(handle, s_ptr)

    # Timed region: K steps; the encode kernels are timed by their own event pair.
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
        enc.step()
    t_end.record(stream)
    bpe.bpe_set_timing_events(handle, None, None)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    bpe.bpe_sync_status(handle, s_ptr)
    step_ms = t_start.elapsed_time(t_end) / args.steps
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    if args.decode_only:
        if rank == 0:
            dec = decode_line(bpe, enc, args.steps, peaks()[0])
            print(json.dumps({"decode_only": True, "workload": workloads.NAMES[cfg], "n_docs": n_docs,
                              "n_bytes": n_bytes, "tokens": int(n_tokens), **dec}), flush=True)
        enc.close()
        if dist:
            dist.destroy_process_group()
        return None

    if args.kernels_only:
        if rank == 0:
            print(json.dumps({"kernels_only": True, "workload": workloads.NAMES[cfg], "n_docs": n_docs,
                              "n_bytes": n_bytes, "tokens": int(n_tokens), "ms_per_step": round(step_ms, 4),
                              "kernel_ms": round(kern_ms, 4), "gpu_launches": LAUNCHES_PER_CALL * args.steps}),
                  flush=True)
        enc.close()
        if dist:
            dist.destroy_process_group()
        return None

    # Secondary: the same calls with the word cache off (every pre-token runs
    # the merge loop), timed the same way, outside the headline region.
    # With the cache off the per-call memo of the misses is on by default;
    # the merge path alone is timed with the memo off too.
    bpe.bpe_set_word_cache(handle, False)
    nocache_ms = statistics.median(enc.time_calls(max(1, min(args.steps, 3)), 1))
    nocache_kernels = enc.kernel_ms()
    bpe.bpe_set_call_memo(handle, bpe.MEMO_OFF)
    nomemo_ms = statistics.median(enc.time_calls(max(1, min(args.steps, 3)), 1))
    nomemo_kernels = enc.kernel_ms()
    bpe.bpe_set_call_memo(handle, bpe.MEMO_AUTO)
    bpe.bpe_set_word_cache(handle, True)

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
    del h_data, h_off, h_ids, h_out
    dec = decode_line(bpe, enc, max(5, min(args.steps, 20)), peaks()[0]) if rank == 0 else None
    trn = train_line(bpe, 2, local) if rank == 0 and world == 1 and args.n_docs is None and not args.no_configs \
        else None
    (step_ms, kern_ms, e2e_s), (all_bytes, all_tokens, all_docs) = reduce_ranks(
        dist, dev, [step_ms, kern_ms, e2e_s], [n_bytes, n_tokens, n_docs])

    out = None
    if rank == 0:
        peak, peak_kind = peaks()
        alg = algorithmic_bytes(n_bytes, n_docs, n_tokens)
        achieved = alg / (kern_ms / 1e3) / 1e9
        value = all_bytes / (step_ms / 1e3) / 1e6
        cpu, configs = None, None
        if world == 1 and args.n_docs is None and not args.no_configs:
            # The other workloads, one at a time (median of >= 10 calls after
            # 3 warm-up calls), then every workload compared whole with the
            # oracle on all host cores.
            configs = {}
            head_ids, head_off = enc.result()
            for c in (1, 2, 3, 4):
                e = Encoder(bpe, c, dev, local)
                ms = statistics.median(e.time_calls(max(10, min(args.steps, 20)), 3))
                configs[f"C{c}"] = config_line(e, ms, peak)
                configs[f"C{c}"]["kernel_ms"] = e.kernel_ms()
                if c == 2:  # the per-call memo forced on where the misses are nearly all distinct
                    bpe.bpe_set_call_memo(e.handle, bpe.MEMO_ON)
                    configs["C2"]["memo_on_ms"] = round(statistics.median(e.time_calls(10, 3)), 4)
                    bpe.bpe_set_call_memo(e.handle, bpe.MEMO_AUTO)
                if not args.no_cpu_baseline:
                    ids_c, off_c = e.result()
                    configs[f"C{c}"]["parity"], _ = parity_line(e, ids_c, off_c)
                e.close()
                del e
                torch.cuda.empty_cache()
            configs[f"C{cfg}"] = config_line(enc, kern_ms, peak)
            configs[f"C{cfg}"]["kernel_ms"] = enc.kernel_ms()
            if not args.no_cpu_baseline:
                par, r = parity_line(enc, head_ids, head_off)
                configs[f"C{cfg}"]["parity"] = par
                cpu = {"value": round(n_bytes / r["wall_s"] / 1e6, 3), "unit": "MB/s", "cores": r["procs"],
                       "kind": "oracle",
                       "sample": f"the whole batch ({n_docs} documents, {n_bytes} bytes) on {r['procs']} pinned "
                                 f"single-threaded oracle processes over byte-balanced document shards "
                                 f"({r['cpu_s']:.0f} CPU-seconds)",
                       "cpu_model": r["cpu_model"], "physical_cores": r["cores"],
                       "tokens_per_s": round(len(r["ids"]) / r["wall_s"], 1),
                       "parity_vs_gpu": "identical" if par["identical"] else "differs"}
        elif world == 1 and not args.no_cpu_baseline:
            g_ids, g_off = enc.result()
            s = oracle_sample(cfg, data, offsets, enc.merges, enc.vb, enc.vo, args.cpu_budget, g_ids, g_off)
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
                       "tokens": int(n_tokens), "merges": int(len(enc.merges)), "n_vocab": int(len(enc.vo) - 1),
                       "l2": (f"inputs ({n_bytes / 2**20:.0f} MiB) larger than L2 (129 MB); no flush" if n_bytes > 129e6 else f"inputs ({n_bytes / 2**20:.0f} MiB) fit in L2: a profiling case, not a bench number"), "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                         "kernel": KERNEL_SPAN, "kernel_ms": round(kern_ms, 4),
                         "algorithmic_bytes_per_launch": alg, "traffic": traffic_from_profile()},
            "cpu_baseline": cpu,
            "e2e": {"value": round(all_bytes / e2e_s / 1e6, 3),
                    "unit": "MB/s", "h2d_bytes_per_step": n_bytes + 8 * (n_docs + 1),
                    "d2h_bytes_per_step": 4 * int(n_tokens) + 8 * (n_docs + 1)},
            "without_word_cache": {"value": round(n_bytes / (nocache_ms / 1e3) / 1e6, 3), "unit": "MB/s",
                                   "ms_per_step": round(nocache_ms, 4),
                                   "hbm_frac": round(alg / (nocache_ms / 1e3) / 1e9 / peak, 4),
                                   "per_call_memo": "on (the default with the cache off)",
                                   "kernel_ms": nocache_kernels,
                                   "memo_off": {"value": round(n_bytes / (nomemo_ms / 1e3) / 1e6, 3),
                                                "ms_per_step": round(nomemo_ms, 4), "kernel_ms": nomemo_kernels}},
            "decode": dec,
            "train": trn,
            "configs": configs,
            "gpu_launches": LAUNCHES_PER_CALL * args.steps,
            "clocks": clk,
        }
        print(json.dumps(out), flush=True)
    enc.close()
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
    ap.add_argument("--reference-slice-mib", type=int, default=64,
                    help="MiB of whole documents per --impl reference step")
    ap.add_argument("--no-configs", action="store_true", help="headline workload only (no C1-C4 lines, no full parity)")
    ap.add_argument("--decode-only", action="store_true",
                    help="profiling runs: after the encode steps, only bpe_decode_batch of the encoded batch "
                         "(3 warm-up calls, then --steps calls); prints a short line that is not a bench result")
    ap.add_argument("--kernels-only", action="store_true",
                    help="profiling runs: the warm-up and timed device calls only (no cache-off, e2e or oracle "
                         "legs); prints a short line that is not a bench result")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
