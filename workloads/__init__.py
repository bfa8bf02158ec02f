"""Seeded synthetic inputs for batched byte-level BPE encoding.

Input generation only: corpora, documents and the BPE trainer that turns a
corpus into a ranked merge table. The CUDA encoder and the CPU oracle both
consume these arrays as data; nothing here computes an encoding.

Five workloads, each named by what it is:

====  =========================================================================
cfg   workload
====  =========================================================================
1     tiny: 512 merges trained on a 256 KiB ASCII corpus; 256 ASCII documents
      of 1-4 KiB (about 640 KiB)
2     mixed-script: 32,000 merges trained on a 16 MiB mixed-script corpus;
      16,384 mixed-script documents, log-normal lengths (median 4 KiB,
      sigma 1.0)
3     long context: 150,000 merges trained on a 64 MiB ASCII corpus; 16
      mixed-script documents of 8 MiB with a newline every 40-120 bytes
4     adversarial long pre-tokens: the tiny table; 4,096 documents, each a
      1-64 KiB run of one letter, digit or CJK ideograph, 10% normal text
      around it and a whitespace run of up to 4 KiB
5     serving batch: 100,000 merges trained on a 32 MiB ASCII corpus;
      4,194,304 ASCII documents of 64-448 bytes (about 1 GiB)
====  =========================================================================

Seeds: corpus ``0xB9E00000 + cfg``, documents ``0xB9E10000 + cfg``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libworkloads.so")
_lock = threading.Lock()
_lib = None

NAMES = {
    1: "tiny-512m-256docs",
    2: "mixed-script-32k-16384docs",
    3: "long-context-150k-16x8MiB",
    4: "adversarial-long-pretokens-4096docs",
    5: "serving-batch-100k-4Mdocs-1GiB",
}


def build(force: bool = False) -> str:
    """Compile gen.cpp into _build/libworkloads.so (host code, any arch)."""
    src = os.path.join(_HERE, "gen.cpp")
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(src):
        return _LIB
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", "-o", tmp, src])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.wl_corpus.restype = i64
            lib.wl_corpus.argtypes = [ctypes.c_int, ctypes.c_uint64, p, i64]
            lib.wl_docs.restype = i64
            lib.wl_docs.argtypes = [ctypes.c_int, ctypes.c_uint64, i64, i64, p, p]
            lib.wl_train.restype = i64
            lib.wl_train.argtypes = [p, i64, i64, p]
            lib.wl_train_words.restype = i64
            lib.wl_train_words.argtypes = [p, i64, ctypes.POINTER(i64), p, p, p]
            for f in ("wl_cfg_corpus_bytes", "wl_cfg_n_merges", "wl_cfg_n_docs"):
                getattr(lib, f).restype = i64
                getattr(lib, f).argtypes = [ctypes.c_int]
            lib.wl_word.restype = ctypes.c_int
            lib.wl_word.argtypes = [ctypes.c_int, ctypes.c_char_p]
            lib.wl_fnv1a64.restype = ctypes.c_uint64
            lib.wl_fnv1a64.argtypes = [p, i64, ctypes.c_uint64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def corpus_seed(cfg: int) -> int:
    return 0xB9E00000 + cfg


def docs_seed(cfg: int) -> int:
    return 0xB9E10000 + cfg


def n_docs(cfg: int) -> int:
    return int(_load().wl_cfg_n_docs(cfg))


def n_merges(cfg: int) -> int:
    return int(_load().wl_cfg_n_merges(cfg))


def word_list() -> list[str]:
    lib = _load()
    buf = ctypes.create_string_buffer(32)
    out = []
    for i in range(2000):
        lib.wl_word(i, buf)
        out.append(buf.value.decode())
    return out


def corpus(cfg: int) -> np.ndarray:
    """The trainer corpus of a workload as uint8."""
    lib = _load()
    cap = int(lib.wl_cfg_corpus_bytes(cfg)) + 8
    out = np.empty(cap, dtype=np.uint8)
    n = lib.wl_corpus(cfg, corpus_seed(cfg), _ptr(out), cap)
    if n < 0:
        raise RuntimeError(f"corpus generation failed for cfg {cfg}")
    return out[:n].copy()


def doc_lengths(cfg: int, first: int = 0, count: int | None = None, seed: int | None = None) -> np.ndarray:
    lib = _load()
    if count is None:
        count = n_docs(cfg) - first
    lens = np.empty(count, dtype=np.int64)
    r = lib.wl_docs(cfg, docs_seed(cfg) if seed is None else seed, first, count, _ptr(lens), None)
    if r < 0:
        raise RuntimeError("document generation failed")
    return lens


def docs(cfg: int, first: int = 0, count: int | None = None, seed: int | None = None):
    """Documents [first, first + count) of a workload.

    Returns ``(data uint8[N], offsets int64[count + 1])``; document k is
    ``data[offsets[k]:offsets[k + 1]]``. Every document comes from its own
    random stream, so a subset equals the same slice of the full batch.
    """
    lib = _load()
    seed = docs_seed(cfg) if seed is None else seed
    lens = doc_lengths(cfg, first, count, seed)
    offsets = np.zeros(len(lens) + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    data = np.empty(int(offsets[-1]), dtype=np.uint8)
    r = lib.wl_docs(cfg, seed, first, len(lens), _ptr(lens), _ptr(data) if data.size else _ptr(np.empty(1, np.uint8)))
    if r < 0:
        raise RuntimeError("document generation failed")
    return data, offsets


def train_words(text: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The trainer's word list of a corpus: (bytes uint8, offsets int64[n+1],
    counts int64[n]) of its distinct pre-tokens, first-seen order."""
    lib = _load()
    text = np.ascontiguousarray(text, dtype=np.uint8)
    total = ctypes.c_int64(0)
    n = lib.wl_train_words(_ptr(text) if text.size else 0, text.size, ctypes.byref(total), None, None, None)
    data = np.zeros(max(1, total.value), np.uint8)
    offsets = np.zeros(n + 1, np.int64)
    counts = np.zeros(max(1, n), np.int64)
    lib.wl_train_words(_ptr(text) if text.size else 0, text.size, ctypes.byref(total), _ptr(data), _ptr(offsets),
                       _ptr(counts))
    return data[:total.value], offsets, counts[:n]


def train(text: np.ndarray, merges: int) -> np.ndarray:
    """BPE trainer: int32[k, 3] rows (left_id, right_id, new_id); rank = row.

    Byte b has ID b; merge k gets ID 256 + k. k < ``merges`` when the corpus
    runs out of pairs first.
    """
    lib = _load()
    text = np.ascontiguousarray(text, dtype=np.uint8)
    out = np.empty((max(merges, 1), 3), dtype=np.int32)
    k = lib.wl_train(_ptr(text) if text.size else 0, text.size, merges, _ptr(out))
    return out[:k].copy()


FNV64_BASIS = 0xCBF29CE484222325


def fnv1a64(a: np.ndarray, h: int = FNV64_BASIS) -> int:
    """FNV-1a 64 digest of an array's bytes (little-endian), continuing from h.

    A checksum to compare id streams between implementations; it is not part
    of any encoding.
    """
    a = np.ascontiguousarray(a)
    if a.size == 0:
        return h
    return int(_load().wl_fnv1a64(a.ctypes.data, a.nbytes, h))


def vocab_from_merges(merges: np.ndarray):
    """Byte strings of every token as CSR ``(bytes uint8[], offsets int64[V+1])``.

    Token b < 256 is the single byte b; token new_id of a merge row is the
    concatenation of its left and right tokens.
    """
    merges = np.asarray(merges, dtype=np.int64).reshape(-1, 3)
    n_vocab = 256 + len(merges)
    if len(merges):
        n_vocab = max(n_vocab, int(merges[:, 2].max()) + 1)
    toks: list[bytes | None] = [None] * n_vocab
    for b in range(256):
        toks[b] = bytes([b])
    for left, right, new in merges.tolist():
        toks[new] = toks[left] + toks[right]
    lens = np.array([len(t) if t is not None else 0 for t in toks], dtype=np.int64)
    offsets = np.zeros(n_vocab + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    data = np.frombuffer(b"".join(t for t in toks if t is not None), dtype=np.uint8).copy()
    return data, offsets


_table_cache: dict[int, tuple] = {}


def table(cfg: int):
    """(merges, vocab_bytes, vocab_offsets) of a workload; cfg 4 reuses cfg 1.

    Trained tables are cached in _build/ keyed by configuration so repeated
    runs on one machine train once.
    """
    src = 1 if cfg == 4 else cfg
    if src in _table_cache:
        return _table_cache[src]
    path = os.path.join(_BUILD, f"table_cfg{src}.npy")
    merges = None
    if os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(os.path.join(_HERE, "gen.cpp")):
        merges = np.load(path)
    if merges is None:
        merges = train(corpus(src), n_merges(src))
        os.makedirs(_BUILD, exist_ok=True)
        tmp = path + f".tmp{os.getpid()}.npy"
        np.save(tmp, merges)
        os.replace(tmp, path)
    vb, vo = vocab_from_merges(merges)
    _table_cache[src] = (merges, vb, vo)
    return _table_cache[src]
