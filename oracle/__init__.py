"""ORACLE — test infrastructure only.

A plain, slow, single-threaded CPU encoder for byte-level BPE (bpe_oracle.cpp)
and its ctypes binding. It shares no code with the CUDA encoder. Only the
tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import it; the product path never does.

Every step is pinned in tests/test_oracle_pins.py against the pages' worked
values, a brute-force encoder built on the ``regex`` module, closed forms and
invariants. No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile bpe_oracle.cpp into _build/liboracle.so with the host g++."""
    srcs = [os.path.join(_HERE, f) for f in ("bpe_oracle.cpp", "unicode_ranges.inc")]
    if not force and os.path.exists(_LIB) and all(os.path.getmtime(_LIB) >= os.path.getmtime(s) for s in srcs):
        return _LIB
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", tmp, srcs[0]])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.orc_new.restype = p
            lib.orc_new.argtypes = [p, i64, p, p, i64]
            lib.orc_free.argtypes = [p]
            lib.orc_pretokenize.restype = i64
            lib.orc_pretokenize.argtypes = [p, i64, p, i64]
            lib.orc_pretokenize_batch.restype = None
            lib.orc_pretokenize_batch.argtypes = [p, p, i64, p]
            lib.orc_units.restype = i64
            lib.orc_units.argtypes = [p, i64, p, i64]
            lib.orc_class.restype = i32
            lib.orc_class.argtypes = [i32]
            lib.orc_byte_to_unicode.restype = i32
            lib.orc_byte_to_unicode.argtypes = [i32]
            lib.orc_encode_piece.restype = i64
            lib.orc_encode_piece.argtypes = [p, p, i64, p, i64]
            lib.orc_encode_batch.restype = i64
            lib.orc_encode_batch.argtypes = [p, p, p, i64, i64, p, i64, p]
            lib.orc_decode.restype = i64
            lib.orc_decode.argtypes = [p, p, i64, p, i64]
            lib.orc_error.restype = ctypes.c_char_p
            lib.orc_error.argtypes = [p]
            _lib = lib
    return _lib


def _buf(x) -> np.ndarray:
    if isinstance(x, (bytes, bytearray)):
        return np.frombuffer(bytes(x), dtype=np.uint8)
    return np.ascontiguousarray(x, dtype=np.uint8)


def _p(a: np.ndarray):
    return a.ctypes.data if a.size else None


def pretokenize(text) -> list[int]:
    """Start offsets of the pre-tokens of one text."""
    lib = _load()
    b = _buf(text)
    cap = max(1, b.size)
    out = np.empty(cap, dtype=np.int64)
    n = lib.orc_pretokenize(_p(b), b.size, out.ctypes.data, cap)
    return out[:n].tolist()


def pretokenize_batch(data, offsets) -> np.ndarray:
    """Start bits (uint32[(N + 31) // 32]) of every piece of every document."""
    lib = _load()
    b = _buf(data)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    bits = np.zeros(max(1, (b.size + 31) // 32), dtype=np.uint32)
    d = b if b.size else np.zeros(1, np.uint8)
    lib.orc_pretokenize_batch(d.ctypes.data, offsets.ctypes.data, len(offsets) - 1, bits.ctypes.data)
    return bits


def pieces(text) -> list[bytes]:
    b = bytes(_buf(text))
    s = pretokenize(b) + [len(b)]
    return [b[s[i]:s[i + 1]] for i in range(len(s) - 1)]


def units(text) -> list[tuple[int, int, int]]:
    """(byte offset, codepoint or -1, class) per decoded unit; class 0 other,
    1 letter, 2 number, 3 whitespace."""
    lib = _load()
    b = _buf(text)
    cap = max(1, b.size)
    out = np.empty((cap, 3), dtype=np.int64)
    n = lib.orc_units(_p(b), b.size, out.ctypes.data, cap)
    return [tuple(r) for r in out[:n].tolist()]


def codepoint_class(cp: int) -> int:
    return int(_load().orc_class(cp))


def byte_to_unicode(b: int) -> int:
    return int(_load().orc_byte_to_unicode(b))


class Oracle:
    """The oracle encoder over one merge table and vocabulary.

    merges: int32[n, 3] rows (left_id, right_id, new_id), rank = row index.
    vocab: CSR (bytes uint8[], offsets int64[V + 1]) of each token's bytes.
    """

    def __init__(self, merges, vocab_bytes, vocab_offsets):
        self._lib = _load()
        self.merges = np.ascontiguousarray(np.asarray(merges, dtype=np.int32).reshape(-1, 3))
        self.vb = np.ascontiguousarray(vocab_bytes, dtype=np.uint8)
        self.vo = np.ascontiguousarray(vocab_offsets, dtype=np.int64)
        self.n_vocab = len(self.vo) - 1
        h = self._lib.orc_new(_p(self.merges), len(self.merges), _p(self.vb) or self.vb.ctypes.data,
                              self.vo.ctypes.data, self.n_vocab)
        if not h:
            raise ValueError("oracle rejected the table")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.orc_free(h)
            self._h = None

    def encode_piece(self, piece) -> list[int]:
        b = _buf(piece)
        out = np.empty(max(1, b.size), dtype=np.int32)
        n = self._lib.orc_encode_piece(self._h, _p(b), b.size, out.ctypes.data, out.size)
        if n < 0:
            raise RuntimeError(self._lib.orc_error(self._h).decode())
        return out[:n].tolist()

    def encode(self, text) -> list[int]:
        b = _buf(text)
        ids, _ = self.encode_batch(b, np.array([0, b.size], dtype=np.int64))
        return ids.tolist()

    def encode_batch(self, data, offsets, first: int = 0, count: int | None = None):
        """Encode documents [first, first + count); returns (ids int32, offsets int64)."""
        data = _buf(data)
        offsets = np.ascontiguousarray(offsets, dtype=np.int64)
        if count is None:
            count = len(offsets) - 1 - first
        nbytes = int(offsets[first + count] - offsets[first]) if count else 0
        cap = max(1, nbytes)
        ids = np.empty(cap, dtype=np.int32)
        out_off = np.empty(count + 1, dtype=np.int64)
        d = data if data.size else np.zeros(1, np.uint8)
        n = self._lib.orc_encode_batch(self._h, d.ctypes.data, offsets.ctypes.data, first, count,
                                       ids.ctypes.data, cap, out_off.ctypes.data)
        if n < 0:
            raise RuntimeError(self._lib.orc_error(self._h).decode())
        return ids[:n].copy(), out_off

    def decode(self, ids) -> bytes:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        cap = int(sum(int(self.vo[i + 1] - self.vo[i]) for i in ids.tolist() if 0 <= i < self.n_vocab)) + 1
        out = np.empty(cap, dtype=np.uint8)
        n = self._lib.orc_decode(self._h, _p(ids) or out.ctypes.data, ids.size, out.ctypes.data, cap)
        if n < 0:
            raise RuntimeError("oracle decode failed")
        return bytes(out[:n])
