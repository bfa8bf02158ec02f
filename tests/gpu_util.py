"""Helpers for GPU tests: run the CUDA path through the C ABI and compare with
the oracle document by document."""
from __future__ import annotations

import numpy as np


def batch(docs: list[bytes]):
    data = np.frombuffer(b"".join(docs), dtype=np.uint8).copy()
    offsets = np.zeros(len(docs) + 1, dtype=np.int64)
    np.cumsum([len(d) for d in docs], out=offsets[1:])
    return data, offsets


def gpu_encode(handle: int, data: np.ndarray, offsets: np.ndarray, n_bytes: int | None = None):
    """Encode through bpe_encode_batch; returns (ids, out_offsets) as numpy."""
    import torch

    import byte_level_bpe_pretokenize_gb300 as bpe
    n = data.size if n_bytes is None else n_bytes
    d_data = torch.from_numpy(data if data.size else np.zeros(1, np.uint8)).cuda()
    d_off = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64)).cuda()
    d_ids = torch.full((max(1, n),), -7, dtype=torch.int32, device="cuda")
    d_out = torch.full((len(offsets),), -7, dtype=torch.int64, device="cuda")
    total = bpe.bpe_encode_batch(handle, d_data.data_ptr(), n, d_off.data_ptr(), len(offsets) - 1,
                                 d_ids.data_ptr(), d_ids.numel(), d_out.data_ptr(), True,
                                 torch.cuda.current_stream().cuda_stream)
    return d_ids[:total].cpu().numpy(), d_out.cpu().numpy()


def gpu_start_bits(data: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    import torch

    import byte_level_bpe_pretokenize_gb300 as bpe
    words = max(1, (data.size + 31) // 32)
    d_data = torch.from_numpy(data if data.size else np.zeros(1, np.uint8)).cuda()
    d_off = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64)).cuda()
    bits = torch.zeros(words, dtype=torch.int32, device="cuda")
    bpe.bpe_pretokenize_batch(d_data.data_ptr(), data.size, d_off.data_ptr(), len(offsets) - 1, bits.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return bits.cpu().numpy().view(np.uint32)


def assert_same_encoding(got, want, data, offsets, label=""):
    g_ids, g_off = got
    w_ids, w_off = want
    if np.array_equal(g_off, w_off) and np.array_equal(g_ids, w_ids):
        return
    for k in range(len(offsets) - 1):
        a = g_ids[g_off[k]:g_off[k + 1]] if g_off[k] <= g_off[k + 1] <= len(g_ids) else None
        b = w_ids[w_off[k]:w_off[k + 1]]
        if a is None or not np.array_equal(a, b):
            doc = bytes(data[offsets[k]:offsets[k + 1]])
            if a is not None:
                n = min(len(a), len(b))
                diff = np.nonzero(a[:n] != b[:n])[0]
                i = int(diff[0]) if len(diff) else n
                a, b = a[max(0, i - 5):i + 30], b[max(0, i - 5):i + 30]
                label = f"{label} (first difference at token {i}; showing from {max(0, i - 5)})"
            raise AssertionError(f"{label}: document {k} ({len(doc)} bytes, starts {doc[:60]!r}) differs:\n"
                                 f"gpu    {None if a is None else a[:40].tolist()}\noracle {b[:40].tolist()}\n"
                                 f"offsets gpu {g_off[k]}..{g_off[k + 1]} oracle {w_off[k]}..{w_off[k + 1]}")
    raise AssertionError(f"{label}: outputs differ (ids {len(g_ids)} vs {len(w_ids)})")
