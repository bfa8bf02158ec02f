"""ORACLE — test infrastructure only: the oracle on every host core.

The same single-threaded oracle encoder (bpe_oracle.cpp), run as P separate
processes over byte-balanced contiguous document shards, each process pinned
to one core. Documents are independent, so the concatenated shard outputs are
the batch's encoding ("Hugging Face Tokenizers v1", section "performance
benchmarks": throughput is measured on physical cores pinned one worker each,
and the output ids are compared by their FNV-1a hash).

Processes are started with the ``spawn`` method, so the pool is safe to use
from a process that already holds a CUDA context. The input reaches the
workers through POSIX shared memory; each worker returns its shard's ids and
per-document token counts.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import platform
import subprocess
import time
from multiprocessing import shared_memory

import numpy as np

_W: dict = {}


def cpu_model() -> str:
    """The host CPU's model name as lscpu or /proc/cpuinfo reports it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def physical_cores() -> list[int]:
    """One logical CPU per physical core (the lowest-numbered SMT sibling),
    restricted to the CPUs this process may run on."""
    allowed = sorted(os.sched_getaffinity(0))
    seen, cores = set(), []
    for c in allowed:
        key = None
        try:
            base = f"/sys/devices/system/cpu/cpu{c}/topology"
            pkg = open(f"{base}/physical_package_id").read().strip()
            core = open(f"{base}/core_id").read().strip()
            key = (pkg, core)
        except OSError:
            key = ("cpu", c)
        if key not in seen:
            seen.add(key)
            cores.append(c)
    return cores


def _init(names, shapes, merges, vb, vo, core_q):
    import oracle
    try:
        core = core_q.get_nowait()
        os.sched_setaffinity(0, {core})
    except Exception:  # noqa: BLE001 - pinning is best effort
        pass
    shm_d = shared_memory.SharedMemory(name=names[0])
    shm_o = shared_memory.SharedMemory(name=names[1])
    _W["shm"] = (shm_d, shm_o)
    _W["data"] = np.ndarray((shapes[0],), dtype=np.uint8, buffer=shm_d.buf)
    _W["offsets"] = np.ndarray((shapes[1],), dtype=np.int64, buffer=shm_o.buf)
    _W["orc"] = oracle.Oracle(merges, vb, vo)


def _run(job):
    first, count = job
    if count < 0:  # start-up job: holds its worker so that every worker takes one
        time.sleep(0.2)
        return first, np.zeros(0, np.int32), np.zeros(0, np.int64), 0.0
    t0 = time.perf_counter()
    ids, off = _W["orc"].encode_batch(_W["data"], _W["offsets"], first, count)
    return first, ids, np.diff(off), time.perf_counter() - t0


def shards(offsets: np.ndarray, n: int) -> list[tuple[int, int]]:
    """n contiguous (first, count) document ranges of about equal bytes."""
    n_docs = len(offsets) - 1
    if n_docs == 0:
        return []
    lo, hi = int(offsets[0]), int(offsets[-1])
    cuts = [0]
    for k in range(1, n):
        cuts.append(int(np.searchsorted(offsets, lo + (hi - lo) * k / n, side="left")))
    cuts.append(n_docs)
    cuts = sorted(set(min(max(c, 0), n_docs) for c in cuts))
    return [(a, b - a) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def encode(merges, vb, vo, data: np.ndarray, offsets: np.ndarray, procs: int | None = None,
           shards_per_proc: int = 4) -> dict:
    """Encode a batch with the oracle on ``procs`` pinned processes.

    Returns ``{"ids", "offsets", "wall_s", "cpu_s", "procs", "cores",
    "cpu_model"}``: the whole batch's ids (int32) and document offsets (int64,
    starting at 0), the wall time of the parallel encode (pool start-up and
    input hand-over excluded), the summed per-shard encode time, and the
    number of processes.
    """
    data = np.ascontiguousarray(data, dtype=np.uint8)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    cores = physical_cores()
    procs = max(1, min(procs or len(cores), len(cores)))
    n_docs = len(offsets) - 1
    jobs = shards(offsets, procs * shards_per_proc)
    shm_d = shared_memory.SharedMemory(create=True, size=max(1, data.nbytes))
    shm_o = shared_memory.SharedMemory(create=True, size=max(8, offsets.nbytes))
    try:
        np.ndarray(data.shape, dtype=np.uint8, buffer=shm_d.buf)[:] = data
        np.ndarray(offsets.shape, dtype=np.int64, buffer=shm_o.buf)[:] = offsets
        ctx = mp.get_context("spawn")
        core_q = ctx.Queue()
        for c in cores[:procs]:
            core_q.put(c)
        args = ((shm_d.name, shm_o.name), (data.size, offsets.size), np.asarray(merges), np.asarray(vb),
                np.asarray(vo), core_q)
        with ctx.Pool(procs, initializer=_init, initargs=args) as pool:
            # the workers have attached and built their oracle once this returns
            pool.map(_run, [(0, -1)] * procs, chunksize=1)
            t0 = time.perf_counter()
            results = pool.map(_run, jobs, chunksize=1)
            wall = time.perf_counter() - t0
    finally:
        shm_d.close()
        shm_d.unlink()
        shm_o.close()
        shm_o.unlink()
    results.sort(key=lambda r: r[0])
    counts = np.zeros(n_docs, dtype=np.int64)
    parts = []
    for first, ids, cnt, _ in results:
        counts[first:first + len(cnt)] = cnt
        parts.append(ids)
    out_off = np.zeros(n_docs + 1, dtype=np.int64)
    np.cumsum(counts, out=out_off[1:])
    ids = np.concatenate(parts) if parts else np.zeros(0, dtype=np.int32)
    return {"ids": ids, "offsets": out_off, "wall_s": wall, "cpu_s": sum(r[3] for r in results),
            "procs": procs, "cores": len(cores), "cpu_model": cpu_model()}
