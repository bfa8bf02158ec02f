"""Brute-force byte-level BPE for tiny inputs, used to pin the oracle.

Independent of the oracle's C++ code: the split is the ``regex`` module
running the GPT-2-style pattern, symbols are Python ``bytes`` objects, a pair's
rank is found by scanning the merge list from the top, and ids by scanning the
vocabulary list. Every merge step rescans all pairs.
"""
from __future__ import annotations

GPT2_PATTERN = r"""'s|'t|'re|'ve|'m|'ll|'d| ?\p{L}+| ?\p{N}+| ?[^\s\p{L}\p{N}]+|\s+(?!\S)|\s+"""

_compiled = None


def split(text: bytes) -> list[bytes]:
    """Pre-tokens of a text. Invalid UTF-8 bytes become lone surrogates
    (surrogateescape), which the pattern treats as neither letter, number nor
    whitespace — one unit per byte."""
    global _compiled
    import regex
    if _compiled is None:
        _compiled = regex.compile(GPT2_PATTERN)
    s = text.decode("utf-8", errors="surrogateescape")
    return [m.encode("utf-8", errors="surrogateescape") for m in _compiled.findall(s)]


def merge_piece(piece: bytes, merges: list[tuple[bytes, bytes]]) -> list[bytes]:
    syms = [bytes([b]) for b in piece]
    while True:
        best = None
        for i in range(len(syms) - 1):
            for r, (a, b) in enumerate(merges):
                if best is not None and r >= best:
                    break
                if syms[i] == a and syms[i + 1] == b:
                    best = r
                    break
        if best is None:
            return syms
        a, b = merges[best]
        out, i = [], 0
        while i < len(syms):
            if i + 1 < len(syms) and syms[i] == a and syms[i + 1] == b:
                out.append(a + b)
                i += 2
            else:
                out.append(syms[i])
                i += 1
        syms = out


def encode(text: bytes, merges_ids, vocab: list[bytes]) -> list[int]:
    """merges_ids: rows (left_id, right_id, new_id); vocab[id] = token bytes."""
    merges = [(vocab[a], vocab[b]) for a, b, _ in merges_ids]
    ids = []
    for piece in split(text):
        for sym in merge_piece(piece, merges):
            ids.append(vocab.index(sym))
    return ids
