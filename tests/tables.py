"""Small merge tables for tests, built from byte strings."""
from __future__ import annotations

import random

import numpy as np


def table_from_pairs(pairs, ids=None, n_vocab=None):
    """merges (int32[k, 3]), vocab bytes, vocab offsets for merge rows given as
    (left_bytes, right_bytes) in rank order.

    Tokens are the 256 single bytes plus one token per row; row k gets id
    ``ids[k]`` (default 256 + k). Left and right must already be tokens when
    the whole table is built, in any row order (tables need not be monotone).
    """
    pairs = [(bytes(a), bytes(b)) for a, b in pairs]
    if ids is None:
        ids = [256 + k for k in range(len(pairs))]
    if n_vocab is None:
        n_vocab = max([255] + list(ids)) + 1
    tok: list[bytes] = [b""] * n_vocab
    for b in range(256):
        tok[b] = bytes([b])
    index = {tok[b]: b for b in range(256)}
    for (a, b), i in zip(pairs, ids):
        tok[i] = a + b
        index[a + b] = i
    rows = []
    for (a, b), i in zip(pairs, ids):
        rows.append((index[a], index[b], i))
    merges = np.array(rows, dtype=np.int32).reshape(-1, 3)
    lens = np.array([len(t) for t in tok], dtype=np.int64)
    offsets = np.zeros(n_vocab + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    data = np.frombuffer(b"".join(tok), dtype=np.uint8).copy()
    return merges, data, offsets


def vocab_list(vb, vo) -> list[bytes]:
    return [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]


def random_table(rng: random.Random, alphabet: bytes, n_merges: int, monotone: bool):
    """A random table over an alphabet: each new token joins two existing
    tokens. With monotone=False the rows are shuffled, so a merge may use a
    token that a lower-priority row creates."""
    tokens = [bytes([c]) for c in alphabet]
    seen = set(tokens)
    pairs = []
    tries = 0
    while len(pairs) < n_merges and tries < 50 * n_merges:
        tries += 1
        a, b = rng.choice(tokens), rng.choice(tokens)
        if a + b in seen or len(a + b) > 8:
            continue
        seen.add(a + b)
        tokens.append(a + b)
        pairs.append((a, b))
    if not monotone:
        rng.shuffle(pairs)
    return table_from_pairs(pairs)
