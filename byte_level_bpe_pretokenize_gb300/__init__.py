"""Python binding of the GB300 batched byte-level BPE encoder.

Argument marshalling only: every step of the encoder runs in the CUDA kernels
of ``libbpe_gb300.so`` behind the C ABI in ``include/bpe_gb300.h``. There is
no CPU fallback; loading fails loudly when the library is missing.

Low level: ``bpe_build``, ``bpe_encode_batch``, ``bpe_encode_batch_noalloc``,
``bpe_pretokenize_batch``, ``bpe_decode_batch``, ``bpe_sync_status``,
``bpe_destroy`` take device pointers as integers, exactly like the C calls;
``bpe_encode_batch_host`` takes host pointers.
High level: ``Tokenizer`` takes torch CUDA tensors and the current stream.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libbpe_gb300.so")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared"]

BPE_OK = 0
ERRORS = {1: "INVALID_ARG", 2: "CAPACITY", 3: "CUDA", 4: "BAD_TABLE", 5: "TIMEOUT", 6: "INTERNAL", 7: "BAD_INPUT"}


class BpeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"BPE_ERR_{ERRORS.get(code, code)}: {msg}")
        self.code = code


def _sources():
    return [os.path.join(_CSRC, f) for f in ("bpe_kernels.cu", "tiles.cuh", "class_table.inc")] + \
        [os.path.join(_ROOT, "include", "bpe_gb300.h")]


def build(force: bool = False, nvcc: str = "nvcc") -> str:
    """Compile the CUDA library in-tree for sm_103a (cross-compiles without a GPU)."""
    if not force and os.path.exists(LIB_PATH) and \
            all(os.path.getmtime(LIB_PATH) >= os.path.getmtime(s) for s in _sources()):
        return LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *NVCC_FLAGS, "-o", tmp, os.path.join(_CSRC, "bpe_kernels.cu")])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lock = threading.Lock()
_lib = None

EXPORTS = ["bpe_build", "bpe_encode_batch", "bpe_encode_batch_host", "bpe_encode_batch_noalloc", "bpe_pretokenize_batch", "bpe_decode_batch", "bpe_set_word_cache",
           "bpe_set_timing_events", "bpe_set_phase_events", "bpe_set_call_memo", "bpe_sync_status", "bpe_table_info", "bpe_table_monotone", "bpe_merges_monotone",
           "bpe_workspace_bytes", "bpe_train", "bpe_destroy", "bpe_last_error"]


def lib():
    """The loaded C library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                                   "(the encoder has no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            L.bpe_build.restype = ctypes.c_int
            L.bpe_build.argtypes = [p, i64, p, p, i64, ctypes.c_int, ctypes.POINTER(p)]
            L.bpe_encode_batch.restype = ctypes.c_int
            L.bpe_encode_batch.argtypes = [p, p, i64, p, i64, p, i64, p, p, p]
            L.bpe_encode_batch_host.restype = ctypes.c_int
            L.bpe_encode_batch_host.argtypes = [p, p, i64, p, i64, p, i64, p, p, p]
            L.bpe_encode_batch_noalloc.restype = ctypes.c_int
            L.bpe_encode_batch_noalloc.argtypes = [p, p, i64, p, i64, p, i64, p, p, p]
            L.bpe_pretokenize_batch.restype = ctypes.c_int
            L.bpe_pretokenize_batch.argtypes = [p, i64, p, i64, p, p]
            L.bpe_decode_batch.restype = ctypes.c_int
            L.bpe_decode_batch.argtypes = [p, p, i64, p, i64, p, i64, p, p, p]
            L.bpe_set_word_cache.restype = ctypes.c_int
            L.bpe_set_word_cache.argtypes = [p, ctypes.c_int]
            L.bpe_set_timing_events.restype = ctypes.c_int
            L.bpe_set_timing_events.argtypes = [p, p, p]
            L.bpe_set_call_memo.restype = ctypes.c_int
            L.bpe_set_call_memo.argtypes = [p, ctypes.c_int]
            L.bpe_set_phase_events.restype = ctypes.c_int
            L.bpe_set_phase_events.argtypes = [p, p, ctypes.c_int]
            L.bpe_sync_status.restype = ctypes.c_int
            L.bpe_sync_status.argtypes = [p, p]
            L.bpe_table_info.restype = ctypes.c_int
            L.bpe_table_info.argtypes = [p, ctypes.POINTER(i64), ctypes.POINTER(i64)]
            L.bpe_table_monotone.restype = ctypes.c_int
            L.bpe_table_monotone.argtypes = [p, ctypes.POINTER(ctypes.c_int)]
            L.bpe_merges_monotone.restype = ctypes.c_int
            L.bpe_merges_monotone.argtypes = [p, i64, i64, ctypes.POINTER(ctypes.c_int)]
            L.bpe_train.restype = ctypes.c_int
            L.bpe_train.argtypes = [p, p, p, i64, i64, ctypes.c_int, p, ctypes.POINTER(i64)]
            L.bpe_workspace_bytes.restype = ctypes.c_int
            L.bpe_workspace_bytes.argtypes = [p, ctypes.POINTER(i64)]
            L.bpe_destroy.restype = ctypes.c_int
            L.bpe_destroy.argtypes = [p]
            L.bpe_last_error.restype = ctypes.c_char_p
            L.bpe_last_error.argtypes = []
            _ = i32
            _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != BPE_OK:
        raise BpeError(rc, lib().bpe_last_error().decode(errors="replace"))


# ------------------------------------------------------------ C-ABI mirror --

def bpe_build(merges, vocab_bytes, vocab_offsets, device: int = 0) -> int:
    """Host arrays in, opaque handle (int) out. See include/bpe_gb300.h."""
    m = np.ascontiguousarray(np.asarray(merges, dtype=np.int32).reshape(-1, 3))
    vb = np.ascontiguousarray(vocab_bytes, dtype=np.uint8)
    vo = np.ascontiguousarray(vocab_offsets, dtype=np.int64)
    h = ctypes.c_void_p()
    _check(lib().bpe_build(m.ctypes.data if m.size else None, len(m), vb.ctypes.data if vb.size else None,
                           vo.ctypes.data, len(vo) - 1, device, ctypes.byref(h)))
    return h.value


def bpe_encode_batch(handle: int, d_bytes: int, n_bytes: int, d_doc_offsets: int, n_docs: int, d_out_ids: int,
                     out_capacity: int, d_out_offsets: int, want_total: bool, stream: int) -> int | None:
    total = ctypes.c_int64(-1)
    _check(lib().bpe_encode_batch(handle, d_bytes, n_bytes, d_doc_offsets, n_docs, d_out_ids, out_capacity,
                                  d_out_offsets, ctypes.byref(total) if want_total else None, stream))
    return total.value if want_total else None


def bpe_encode_batch_host(handle: int, h_bytes: int, n_bytes: int, h_doc_offsets: int, n_docs: int,
                          h_out_ids: int, out_capacity: int, h_out_offsets: int, want_total: bool,
                          stream: int) -> int | None:
    """bpe_encode_batch on host buffers (pointers as integers; page-locked
    for overlap): copies in, encodes and copies out in a pipeline of slices."""
    total = ctypes.c_int64(-1)
    _check(lib().bpe_encode_batch_host(handle, h_bytes, n_bytes, h_doc_offsets, n_docs, h_out_ids, out_capacity,
                                       h_out_offsets, ctypes.byref(total) if want_total else None, stream))
    return total.value if want_total else None


NOALLOC_MAX_BYTES = 4 << 20  # batch limit of bpe_encode_batch_noalloc's fixed scratch


def bpe_encode_batch_noalloc(handle: int, d_bytes: int, n_bytes: int, d_doc_offsets: int, n_docs: int,
                             d_out_ids: int, out_capacity: int, d_out_offsets: int, want_total: bool,
                             stream: int) -> int | None:
    """bpe_encode_batch on fixed static scratch: allocates no device memory,
    n_bytes <= NOALLOC_MAX_BYTES, one call in flight per device."""
    total = ctypes.c_int64(-1)
    _check(lib().bpe_encode_batch_noalloc(handle, d_bytes, n_bytes, d_doc_offsets, n_docs, d_out_ids, out_capacity,
                                          d_out_offsets, ctypes.byref(total) if want_total else None, stream))
    return total.value if want_total else None


def bpe_pretokenize_batch(d_bytes: int, n_bytes: int, d_doc_offsets: int, n_docs: int, d_start_bits: int,
                          stream: int) -> None:
    _check(lib().bpe_pretokenize_batch(d_bytes, n_bytes, d_doc_offsets, n_docs, d_start_bits, stream))


def bpe_decode_batch(handle: int, d_ids: int, n_ids: int, d_id_offsets: int, n_docs: int, d_out_bytes: int,
                     out_capacity: int, d_out_byte_offsets: int, want_total: bool, stream: int) -> int | None:
    total = ctypes.c_int64(-1)
    _check(lib().bpe_decode_batch(handle, d_ids, n_ids, d_id_offsets, n_docs, d_out_bytes, out_capacity,
                                  d_out_byte_offsets, ctypes.byref(total) if want_total else None, stream))
    return total.value if want_total else None


def bpe_set_word_cache(handle: int, enable: bool) -> None:
    _check(lib().bpe_set_word_cache(handle, 1 if enable else 0))


def bpe_train(word_bytes, word_offsets, word_counts, n_merges: int, device: int = 0):
    """Merge rows int32[k, 3] (left, right, new_id) trained on the GPU from a
    word list (host arrays: bytes, offsets[n + 1], counts[n])."""
    wb = np.ascontiguousarray(word_bytes, dtype=np.uint8)
    wo = np.ascontiguousarray(word_offsets, dtype=np.int64)
    wc = np.ascontiguousarray(word_counts, dtype=np.int64)
    out = np.zeros((max(1, n_merges), 3), dtype=np.int32)
    made = ctypes.c_int64(0)
    _check(lib().bpe_train(wb.ctypes.data if wb.size else None, wo.ctypes.data, wc.ctypes.data if wc.size else None,
                           len(wo) - 1, n_merges, device, out.ctypes.data, ctypes.byref(made)))
    return out[:made.value].copy()


MEMO_OFF, MEMO_ON, MEMO_AUTO = 0, 1, 2


def bpe_set_call_memo(handle: int, mode: int) -> None:
    """Per-call memo of word-cache misses: MEMO_OFF, MEMO_ON or MEMO_AUTO (on
    exactly when the word cache is off)."""
    _check(lib().bpe_set_call_memo(handle, mode))


def bpe_set_timing_events(handle: int, ev_start: int | None, ev_stop: int | None) -> None:
    """cudaEvent_t handles (ints) recorded before the first and after the
    last kernel of each encode call."""
    _check(lib().bpe_set_timing_events(handle, ev_start, ev_stop))


ENCODE_LAUNCHES = 9
ENCODE_KERNELS = ("k_prep_docs", "k_prep_long", "k_tiles", "k_misses", "k_giants", "k_scan_tiles",
                  "k_scan_tile_sums", "k_compact", "k_giant_copy")


class PhaseEvents:
    """ENCODE_LAUNCHES + 1 cudaEvent_t handles (ints) held in a C array that
    lives as long as this object; bpe_set_phase_events records them around
    each kernel of the next encode calls."""

    def __init__(self, events: list[int]):
        if len(events) != ENCODE_LAUNCHES + 1:
            raise ValueError(f"need {ENCODE_LAUNCHES + 1} events")
        self.array = (ctypes.c_void_p * len(events))(*events)


def bpe_set_phase_events(handle: int, events: "PhaseEvents | None") -> None:
    if events is None:
        _check(lib().bpe_set_phase_events(handle, None, 0))
    else:
        _check(lib().bpe_set_phase_events(handle, ctypes.cast(events.array, ctypes.c_void_p), len(events.array)))


def bpe_sync_status(handle: int, stream: int) -> None:
    _check(lib().bpe_sync_status(handle, stream))


def bpe_table_info(handle: int) -> tuple[int, int]:
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().bpe_table_info(handle, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def bpe_table_monotone(handle: int) -> bool:
    m = ctypes.c_int()
    _check(lib().bpe_table_monotone(handle, ctypes.byref(m)))
    return bool(m.value)


def bpe_merges_monotone(merges, n_vocab: int) -> bool:
    """Host-only: whether every merge's operands are bytes or made by lower ranks."""
    mm = np.ascontiguousarray(np.asarray(merges, dtype=np.int32).reshape(-1, 3))
    out = ctypes.c_int()
    _check(lib().bpe_merges_monotone(mm.ctypes.data if mm.size else None, len(mm), n_vocab, ctypes.byref(out)))
    return bool(out.value)


def bpe_workspace_bytes(handle: int) -> int:
    """Device workspace the handle holds now (0 until a call needs it)."""
    b = ctypes.c_int64()
    _check(lib().bpe_workspace_bytes(handle, ctypes.byref(b)))
    return b.value


def bpe_destroy(handle: int) -> None:
    _check(lib().bpe_destroy(handle))


# --------------------------------------------------------------- torch API --

class Tokenizer:
    """A tokenizer on one GPU. Tensors are torch CUDA tensors on that GPU;
    calls run on the current torch stream."""

    def __init__(self, merges, vocab_bytes, vocab_offsets, device: int = 0):
        self.device = device
        self.handle = bpe_build(merges, vocab_bytes, vocab_offsets, device)

    def close(self):
        if getattr(self, "handle", None):
            bpe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _stream():
        import torch
        return torch.cuda.current_stream().cuda_stream

    def encode_into(self, data, offsets, out_ids, out_offsets, want_total: bool = True):
        """data uint8[N], offsets int64[D + 1] -> ids written into out_ids
        (int32, capacity >= N) and out_offsets (int64[D + 1]). Returns the
        token count when want_total (that waits for the stream)."""
        return bpe_encode_batch(self.handle, data.data_ptr(), data.numel(), offsets.data_ptr(), offsets.numel() - 1,
                                out_ids.data_ptr(), out_ids.numel(), out_offsets.data_ptr(), want_total,
                                self._stream())

    def encode(self, data, offsets):
        """Returns (ids int32[T], out_offsets int64[D + 1]) as CUDA tensors."""
        import torch
        out_ids = torch.empty(max(1, data.numel()), dtype=torch.int32, device=data.device)
        out_off = torch.empty(offsets.numel(), dtype=torch.int64, device=data.device)
        total = self.encode_into(data, offsets, out_ids, out_off, True)
        return out_ids[:total], out_off

    def decode(self, ids, id_offsets, capacity: int | None = None):
        """Returns (bytes uint8[B], byte_offsets int64[D + 1]) as CUDA tensors."""
        import torch
        if capacity is None:
            capacity = max(1, ids.numel() * 64)
        out = torch.empty(capacity, dtype=torch.uint8, device=ids.device)
        out_off = torch.empty(id_offsets.numel(), dtype=torch.int64, device=ids.device)
        total = bpe_decode_batch(self.handle, ids.data_ptr(), ids.numel(), id_offsets.data_ptr(),
                                 id_offsets.numel() - 1, out.data_ptr(), capacity, out_off.data_ptr(), True,
                                 self._stream())
        return out[:total], out_off


def pretokenize(data, offsets):
    """Start bits (uint32[(N + 31) / 32]) of the pre-tokens of a batch."""
    import torch
    words = max(1, (data.numel() + 31) // 32)
    bits = torch.zeros(words, dtype=torch.int32, device=data.device)
    bpe_pretokenize_batch(data.data_ptr(), data.numel(), offsets.data_ptr(), offsets.numel() - 1, bits.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    return bits
