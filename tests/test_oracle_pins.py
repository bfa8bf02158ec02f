"""Pins for the oracle: each step checked against something other than itself.

- values the pages print (tests/golden/pages_worked_examples.json);
- the ``regex`` module running the GPT-2-style pattern (pre-tokenizer and
  codepoint classes) and Python's UTF-8 codec;
- brute force on tiny inputs (tests/brute_force.py);
- closed forms (empty table, chains of doubling merges);
- invariants (round trip, no ranked pair left, per-document independence).
"""
import itertools
import json
import os
import random
import unicodedata

import numpy as np
import pytest

import oracle
import workloads
from tests import brute_force
from tests.tables import random_table, table_from_pairs, vocab_list

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


def _oracle_for(pairs, **kw):
    m, vb, vo = table_from_pairs(pairs, **kw)
    return oracle.Oracle(m, vb, vo), vocab_list(vb, vo)


# ------------------------------------------------------------ worked values --

def test_worked_pretokenize():
    for case in GOLDEN["pretokenize"]:
        got = [p.decode() for p in oracle.pieces(case["text"].encode())]
        assert got == case["pieces"], case["cite"]


def test_worked_utf8():
    for case in GOLDEN["utf8"]:
        raw = case["text"].encode("utf-8")
        assert raw == bytes.fromhex(case["bytes"].replace(" ", ""))
        u = oracle.units(raw)
        assert [cp for _, cp, _ in u] == case["codepoints"]
        assert [pos for pos, _, _ in u] == [0, 3]


def test_worked_byte_to_unicode():
    for case in GOLDEN["byte_to_unicode"]:
        assert oracle.byte_to_unicode(case["byte"]) == case["codepoint"], case["cite"]


def test_byte_to_unicode_properties():
    image = [oracle.byte_to_unicode(b) for b in range(256)]
    assert len(set(image)) == 256  # a bijection onto its image
    for b, cp in enumerate(image):
        ch = chr(cp)
        assert ch.isprintable() and not ch.isspace(), (b, cp)
        if chr(b).isprintable() and not chr(b).isspace() and b != 0xAD:
            assert cp == b  # printable Latin-1 stands for itself
        else:
            assert 256 <= cp < 256 + 68


def test_worked_leftmost_non_overlapping():
    case = GOLDEN["leftmost_non_overlapping"][0]
    o, vocab = _oracle_for([(b"a", b"a")])
    ids = o.encode_piece(b"aaa")
    assert [vocab[i].decode() for i in ids] == case["result"], case["cite"]


def test_worked_toy_ranks():
    case = GOLDEN["toy_ranks"][0]
    # Ranks are row indices: fill the unused rows with pairs that never occur.
    rows = [(b"q", bytes([0x30 + k])) for k in range(11)]
    for a, b, r in case["ranks"]:
        rows[r] = (a.encode(), b.encode())
    o, vocab = _oracle_for(rows)
    ids = o.encode(case["word"].encode())
    assert [vocab[i].decode() for i in ids] == case["result"], case["cite"]


def test_worked_vocabulary_lookup():
    case = GOLDEN["vocabulary_lookup"][0]
    words = [b"hello", b" world"]
    pairs, ids, next_id = [], [], 300
    for w in words:
        for k in range(2, len(w) + 1):
            pairs.append((w[:k - 1], w[k - 1:k]))
            ids.append(next_id)
            next_id += 1
    ids[len(b"hello") - 2] = case["ids"][0]
    ids[-1] = case["ids"][1]
    o, vocab = _oracle_for(pairs, ids=ids)
    assert o.encode(case["text"].encode()) == case["ids"], case["cite"]
    # The page's symbol string for " world" uses the byte-to-unicode space.
    assert "".join(chr(oracle.byte_to_unicode(b)) for b in b" world") == case["symbols"][1]


@pytest.mark.parametrize("cfg", [1, 2])
def test_round_trip_page_list(cfg):
    m, vb, vo = workloads.table(cfg)
    o = oracle.Oracle(m, vb, vo)
    for t in GOLDEN["round_trip"]["texts"]:
        raw = t.encode()
        assert o.decode(o.encode(raw)) == raw


# ------------------------------------------- library special cases (regex) --

regex = pytest.importorskip("regex")

from tests.fuzz import fuzz_text as _fuzz_text  # noqa: E402


def test_pretokenize_vs_regex_fuzz():
    rng = random.Random(1234)
    for trial in range(4000):
        t = _fuzz_text(rng, rng.randint(0, 24))
        assert oracle.pieces(t) == brute_force.split(t), t


def test_pretokenize_vs_regex_contractions():
    # Every string of length <= 5 over an alphabet rich in contraction parts.
    alpha = ["'", "s", "r", "e", "l", " ", "\n", "x", "1", "!"]
    for n in range(0, 6):
        for tup in itertools.product(alpha, repeat=n):
            t = "".join(tup).encode()
            assert oracle.pieces(t) == brute_force.split(t), t


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_pretokenize_vs_regex_workloads(cfg):
    data, off = workloads.docs(cfg, 0, 3)
    for k in range(3):
        d = bytes(data[off[k]:off[k + 1]])[:300_000]
        assert oracle.pieces(d) == brute_force.split(d)


def test_codepoint_classes_vs_regex():
    is_l, is_n, is_s = regex.compile(r"\p{L}"), regex.compile(r"\p{N}"), regex.compile(r"\s")
    checked = 0
    for cp in range(0x110000):
        if 0xD800 <= cp <= 0xDFFF:
            continue
        c = chr(cp)
        if unicodedata.category(c) == "Cn":
            continue  # unassigned in the oracle's Unicode version; regex may be newer
        want = 3 if is_s.match(c) else 1 if is_l.match(c) else 2 if is_n.match(c) else 0
        assert oracle.codepoint_class(cp) == want, hex(cp)
        checked += 1
    assert checked > 280_000


def test_utf8_units_vs_codec():
    rng = random.Random(7)
    for _ in range(2000):
        t = _fuzz_text(rng, rng.randint(0, 12))
        s = t.decode("utf-8", errors="surrogateescape")
        want = [(-1 if 0xDC80 <= ord(ch) <= 0xDCFF else ord(ch)) for ch in s]
        assert [cp for _, cp, _ in oracle.units(t)] == want, t


# ------------------------------------------------------------- brute force --

def test_brute_force_exhaustive_small():
    rng = random.Random(99)
    alphabet = b"ab "
    tables = [random_table(rng, alphabet, k, mono) for k in (3, 6, 10) for mono in (True, False)]
    texts = [bytes(t) for n in range(0, 8) for t in itertools.product(alphabet, repeat=n)]
    for m, vb, vo in tables:
        o = oracle.Oracle(m, vb, vo)
        vocab = vocab_list(vb, vo)
        for t in texts:
            assert o.encode(t) == brute_force.encode(t, m.tolist(), vocab), (t, m.tolist())


def test_brute_force_random_up_to_12_bytes():
    rng = random.Random(2024)
    for trial in range(300):
        alphabet = bytes(rng.sample(b"abcx1 '\n", rng.randint(2, 5)))
        m, vb, vo = random_table(rng, alphabet, rng.randint(1, 25), monotone=rng.random() < 0.5)
        o = oracle.Oracle(m, vb, vo)
        vocab = vocab_list(vb, vo)
        for _ in range(20):
            t = bytes(rng.choice(alphabet) for _ in range(rng.randint(0, 12)))
            assert o.encode(t) == brute_force.encode(t, m.tolist(), vocab), (t, m.tolist())


def test_non_monotone_table_reading():
    # (ab, a) outranks (a, b): one step merges every (a, b), so "abab" gives
    # [ab, ab] and not [aba, b].
    o, vocab = _oracle_for([(b"ab", b"a"), (b"a", b"b")])
    assert [vocab[i] for i in o.encode(b"abab")] == [b"ab", b"ab"]


# ------------------------------------------------------------- closed forms --

def test_empty_table_gives_bytes():
    m, vb, vo = table_from_pairs([])
    o = oracle.Oracle(m, vb, vo)
    rng = random.Random(5)
    for _ in range(50):
        t = bytes(rng.randrange(256) for _ in range(rng.randint(0, 40)))
        assert o.encode(t) == list(t)


@pytest.mark.parametrize("levels", [1, 2, 3, 5])
def test_doubling_chain_closed_form(levels):
    pairs = [(b"a" * (1 << j), b"a" * (1 << j)) for j in range(levels)]
    o, vocab = _oracle_for(pairs)
    for n in range(1, 200):
        toks = [vocab[i] for i in o.encode(b"a" * n)]
        q, r = divmod(n, 1 << levels)
        want = [b"a" * (1 << levels)] * q + [b"a" * (1 << j) for j in reversed(range(levels)) if r >> j & 1]
        assert toks == want, n
        assert len(toks) == q + bin(r).count("1")


# --------------------------------------------------------------- invariants --

def test_invariants_on_tiny_workload():
    m, vb, vo = workloads.table(1)
    o = oracle.Oracle(m, vb, vo)
    ranked = {(int(a), int(b)) for a, b, _ in m}
    data, off = workloads.docs(1, 0, 24)
    ids, ioff = o.encode_batch(data, off)
    for k in range(24):
        d = bytes(data[off[k]:off[k + 1]])
        doc_ids = ids[ioff[k]:ioff[k + 1]].tolist()
        assert doc_ids == o.encode(d)  # per-document independence
        assert len(doc_ids) <= len(d)
        assert o.decode(doc_ids) == d
        pieces = oracle.pieces(d)
        assert b"".join(pieces) == d  # pieces tile the document
        flat = []
        for p in pieces:
            pid = o.encode_piece(p)
            flat += pid
            assert not any((pid[i], pid[i + 1]) in ranked for i in range(len(pid) - 1))
        assert flat == doc_ids
