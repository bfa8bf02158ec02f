"""CUDA path vs the oracle, element by element, through the C ABI.

Sizes the oracle finishes in seconds that still span many 4 KiB chunks and a
ragged tail, plus the edge cases: empty batch and documents, bytes outside
every document, invalid UTF-8, pre-tokens at the thread / CTA / window size
limits, long runs that cross many chunks, contractions, every codepoint class.
"""
import random
import unicodedata

import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_util import assert_same_encoding, batch, gpu_encode, gpu_start_bits
from tests.tables import random_table, table_from_pairs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bpe():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import byte_level_bpe_pretokenize_gb300 as m
    return m


def _pair(bpe, table):
    m, vb, vo = table
    return bpe.bpe_build(m, vb, vo, 0), oracle.Oracle(m, vb, vo)


@pytest.fixture(scope="module")
def tiny(bpe):
    h, o = _pair(bpe, workloads.table(1))
    yield h, o
    bpe.bpe_destroy(h)


def check(handle, orc, data, offsets, label="", n_bytes=None):
    """GPU ids with the word cache on and off, and the per-call memo of the
    misses on and off (by default it is on exactly when the cache is off),
    each equal to the oracle's."""
    import byte_level_bpe_pretokenize_gb300 as bpe
    want = orc.encode_batch(data, offsets)
    for cache, memo in ((True, bpe.MEMO_AUTO), (False, bpe.MEMO_AUTO), (True, bpe.MEMO_ON), (False, bpe.MEMO_OFF)):
        bpe.bpe_set_word_cache(handle, cache)
        bpe.bpe_set_call_memo(handle, memo)
        got = gpu_encode(handle, data, offsets, n_bytes)
        assert_same_encoding(got, want, data, offsets,
                             f"{label} (word cache {'on' if cache else 'off'}, memo mode {memo})")
    bpe.bpe_set_word_cache(handle, True)
    bpe.bpe_set_call_memo(handle, bpe.MEMO_AUTO)
    return got


EDGE_DOCS = [
    b"", b"Hello world!", b"a", b" ", b"  ", b"\n", b"it's", b" 's", b"x''s", b"'sam", b"'s's'll", b"I'M 'RE 'll've",
    b"  \nfoo", b"a  b", b"a\t b", b"a \tb", b"   \n\n  x  ", b"tail   ", "Grüße 🐈".encode(), "你好 世界".encode(),
    b"\xff\xfe abc \x80\x80", b"\xe4\xbd", b"\xe4\xbd a", b"\xf0\x9f\x90", b"\xed\xa0\x80x", b"12345 678,9!!",
    " a  b 　c\u0085d".encode(), "é́ x".encode(), b"A" * 64, b"B" * 65, b"c" * 255,
    b"d" * 256, b"e" * 257, b" " * 300, b"7" * 5000, "中".encode() * 1500, b"\t\n " * 700,
]


def test_edge_documents(bpe, tiny):
    h, o = tiny
    data, off = batch(EDGE_DOCS)
    check(h, o, data, off, "edge docs")


def test_empty_batches(bpe, tiny):
    h, o = tiny
    check(h, o, np.zeros(0, np.uint8), np.zeros(1, np.int64), "no docs")
    check(h, o, np.zeros(0, np.uint8), np.zeros(6, np.int64), "empty docs")


def test_bytes_outside_documents(bpe, tiny):
    h, o = tiny
    docs = [b"junk  before ", b"alpha beta", b"", b" gamma's  ", b"junk after"]
    data, off = batch(docs)
    inner = off[1:4].copy()  # documents 1..2 only
    got = gpu_encode(h, data, inner)
    want_ids, want_off = o.encode_batch(data, inner)
    assert np.array_equal(got[1] - 0, want_off) and np.array_equal(got[0], want_ids)


def test_tiny_workload_full(bpe, tiny):
    h, o = tiny
    data, off = workloads.docs(1)
    check(h, o, data, off, "tiny workload")


def test_documents_straddling_chunks(bpe, tiny):
    # Multi-byte characters, contractions and whitespace placed across every
    # offset around the 4 KiB chunk edges.
    h, o = tiny
    rng = random.Random(3)
    pieces = ["中", "é", "🌀", " 's", "'ll", "  ", "\n", "x", "9", "!", " a", " "]
    docs = []
    for shift in range(0, 48):
        body = "".join(rng.choice(pieces) for _ in range(rng.randint(1, 40)))
        docs.append(b"q" * (4096 - 24 + shift) + body.encode())
    data, off = batch(docs)
    check(h, o, data, off, "straddling")


def test_many_tiny_documents(bpe, tiny):
    h, o = tiny
    rng = random.Random(11)
    alpha = [b"a", b" ", b"'", b"s", b"1", b"\n", "é".encode(), b"\xff"]
    docs = [b"".join(rng.choice(alpha) for _ in range(rng.randint(0, 3))) for _ in range(30000)]
    data, off = batch(docs)
    check(h, o, data, off, "tiny docs")


def test_fuzz_documents(bpe, tiny):
    from tests.fuzz import fuzz_text as _fuzz_text
    h, o = tiny
    rng = random.Random(17)
    docs = [_fuzz_text(rng, rng.randint(0, 200)) for _ in range(3000)]
    data, off = batch(docs)
    check(h, o, data, off, "fuzz")


def test_pretokenizer_bits_match(bpe):
    from tests.fuzz import fuzz_text as _fuzz_text
    rng = random.Random(23)
    docs = [_fuzz_text(rng, rng.randint(0, 300)) for _ in range(4000)]
    docs += [bytes(workloads.docs(c, 0, 2)[0][:200_000]) for c in (2, 3, 4)]
    data, off = batch(docs)
    got = gpu_start_bits(data, off)
    want = oracle.pretokenize_batch(data, off)
    assert np.array_equal(got[:len(want)], want)


def test_codepoint_classes_via_split(bpe):
    # For each assigned codepoint X, "aXa", "1X1" and "!X!" are one piece iff
    # X is a letter, a number or other, respectively.
    docs = []
    cps = [cp for cp in range(0x80, 0x110000) if not 0xD800 <= cp <= 0xDFFF
           and unicodedata.category(chr(cp)) != "Cn"]
    for cp in cps:
        x = chr(cp).encode()
        docs += [b"a" + x + b"a", b"1" + x + b"1", b"!" + x + b"!"]
    data, off = batch(docs)
    got = gpu_start_bits(data, off)
    want = oracle.pretokenize_batch(data, off)
    assert np.array_equal(got[:len(want)], want)


@pytest.mark.parametrize("levels", [1, 3, 6])
def test_long_runs_doubling_chain(bpe, levels):
    pairs = [(b"a" * (1 << j), b"a" * (1 << j)) for j in range(levels)]
    h, o = _pair(bpe, table_from_pairs(pairs))
    docs = [b"a" * n for n in (1, 2, 3, 63, 64, 65, 255, 256, 257, 4095, 4096, 4097, 5000, 70001)]
    docs += [b"x " + b"a" * 9000 + b" y", b"a" * 3000 + b"\n" * 5000]
    data, off = batch(docs)
    got = check(h, o, data, off, f"chain {levels}")
    for k, d in enumerate(docs):
        if set(d) == {ord("a")}:
            q, r = divmod(len(d), 1 << levels)
            assert got[1][k + 1] - got[1][k] == q + bin(r).count("1")
    bpe.bpe_destroy(h)


@pytest.mark.parametrize("seed", range(6))
def test_random_tables_including_non_monotone(bpe, seed):
    rng = random.Random(seed)
    alphabet = bytes(rng.sample(b"abcxy1 '\n", rng.randint(2, 6)))
    table = random_table(rng, alphabet, rng.randint(1, 60), monotone=seed % 2 == 0)
    h, o = _pair(bpe, table)
    docs = [bytes(rng.choice(alphabet) for _ in range(rng.randint(0, rng.choice([12, 80, 600, 9000]))))
            for _ in range(400)]
    data, off = batch(docs)
    check(h, o, data, off, f"random table {seed}")
    bpe.bpe_destroy(h)


def test_token_made_by_two_rules(bpe):
    # "abc" is made both by (ab, c) and by (a, bc): the miss path must not
    # assume one rule per token. Ranks put either split first.
    for order in ([(b"a", b"b"), (b"b", b"c"), (b"ab", b"c"), (b"a", b"bc")],
                  [(b"b", b"c"), (b"a", b"b"), (b"a", b"bc"), (b"ab", b"c"), (b"abc", b"abc")]):
        ids = [256, 257, 258, 258] + ([259] if len(order) > 4 else [])
        m, vb, vo = table_from_pairs(order, ids=ids)
        h, o = bpe.bpe_build(m, vb, vo, 0), oracle.Oracle(m, vb, vo)
        rng = random.Random(len(order))
        docs = [bytes(rng.choice(b"abc  x") for _ in range(rng.randint(0, 40))) for _ in range(400)]
        docs += [b"abc" * 30, b" abcabc", b"aabbcc", b"abcabcabc"]
        data, off = batch(docs)
        check(h, o, data, off, f"two rules for one token ({len(order)} rows)")
        bpe.bpe_destroy(h)


def test_non_identity_ids(bpe):
    # Byte tokens and merged tokens at arbitrary ids (not b and 256 + k).
    pairs = [(b"h", b"e"), (b"he", b"l"), (b"hel", b"l"), (b" ", b"w"), (b"l", b"o")]
    m, vb, vo = table_from_pairs(pairs, ids=[15339, 1917, 700, 3001, 42000])
    perm = np.random.default_rng(0).permutation(256)
    # move byte tokens to ids 50000 + perm[b]
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    n_vocab = 50256 + 1
    new = [b""] * n_vocab
    remap = {}
    for b in range(256):
        remap[b] = 50000 + int(perm[b])
    for i, t in enumerate(toks):
        if len(t) > 1:
            remap[i] = i
    for i, t in enumerate(toks):
        if t:
            new[remap[i]] = t
    m2 = np.array([[remap[a], remap[b], remap[c]] for a, b, c in m.tolist()], dtype=np.int32)
    lens = np.array([len(t) for t in new], dtype=np.int64)
    vo2 = np.zeros(n_vocab + 1, dtype=np.int64)
    np.cumsum(lens, out=vo2[1:])
    vb2 = np.frombuffer(b"".join(new), dtype=np.uint8).copy()
    h, o = _pair(bpe, (m2, vb2, vo2))
    data, off = batch([b"hello world", b"hell", b"lol low", "ü".encode()])
    check(h, o, data, off, "remapped ids")
    bpe.bpe_destroy(h)


@pytest.mark.parametrize("p_miss", [0.12, 0.15, 0.17, 0.19, 0.25])
def test_miss_density_around_deferral_limit(bpe, p_miss):
    # Common words (word-cache hits) mixed with random letter strings (misses)
    # so that 4 KiB chunks hold from about 120 to about 200 misses: chunks
    # on both sides of the 160 a chunk hands to the GPU-wide miss merge.
    h, o = _pair(bpe, workloads.table(5))
    rng = random.Random(int(p_miss * 1000))
    common = [b" the", b" of", b" and", b" to", b" in", b" is", b" that", b" for", b" it", b" was"]
    letters = b"bcdfghjklmnpqrstvwxz"
    docs = []
    for _ in range(16):
        words = []
        while sum(len(w) for w in words) < 4000:
            if rng.random() < p_miss:
                words.append(b" " + bytes(rng.choice(letters) for _ in range(rng.randint(4, 12))))
            else:
                words.append(rng.choice(common))
        docs.append(b"".join(words))
    data, off = batch(docs)
    check(h, o, data, off, f"miss density {p_miss}")
    bpe.bpe_destroy(h)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_workload_slices(bpe, cfg):
    h, o = _pair(bpe, workloads.table(cfg))
    count = {2: 60, 3: 1, 4: 12, 5: 3000}[cfg]
    data, off = workloads.docs(cfg, 0, count)
    if cfg == 3:
        data, off = data[:3_000_000].copy(), np.array([0, 3_000_000], dtype=np.int64)
    check(h, o, data, off, f"workload {cfg} slice")
    bpe.bpe_destroy(h)


def test_decode_round_trip(bpe, tiny):
    import torch
    h, o = tiny
    docs = EDGE_DOCS + [bytes(workloads.docs(2, 0, 5)[0])]
    data, off = batch(docs)
    ids, ioff = gpu_encode(h, data, off)
    d_ids = torch.from_numpy(ids if ids.size else np.zeros(1, np.int32)).cuda()
    d_ioff = torch.from_numpy(ioff).cuda()
    out = torch.zeros(data.size + 8, dtype=torch.uint8, device="cuda")
    out_off = torch.zeros(len(off), dtype=torch.int64, device="cuda")
    total = bpe.bpe_decode_batch(h, d_ids.data_ptr(), ids.size, d_ioff.data_ptr(), len(off) - 1, out.data_ptr(),
                                 out.numel(), out_off.data_ptr(), True, torch.cuda.current_stream().cuda_stream)
    assert total == data.size
    assert bytes(out[:total].cpu().numpy()) == bytes(data)
    assert np.array_equal(out_off.cpu().numpy(), off)


def test_error_paths(bpe, tiny):
    import torch
    h, o = tiny
    data, off = batch([b"hello", b"world"])
    d = torch.from_numpy(data).cuda()
    ids = torch.zeros(16, dtype=torch.int32, device="cuda")
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # capacity below the token count: nothing past it is written
    ids[1:] = -5
    with pytest.raises(bpe.BpeError) as e:
        bpe.bpe_encode_batch(h, d.data_ptr(), data.size, torch.from_numpy(off).cuda().data_ptr(), 2, ids.data_ptr(),
                             1, out.data_ptr(), True, s)
    assert e.value.code == 2
    assert (ids[1:] == -5).all()
    # offsets that go backwards are reported, not trusted
    bad = torch.tensor([0, 8, 3], dtype=torch.int64, device="cuda")
    with pytest.raises(bpe.BpeError) as e:
        bpe.bpe_encode_batch(h, d.data_ptr(), data.size, bad.data_ptr(), 2, ids.data_ptr(), 16, out.data_ptr(),
                             True, s)
    assert e.value.code == 7
    # the handle works normally afterwards
    check(h, o, data, off, "after errors")
    # an id out of range in decode
    bad_ids = torch.tensor([1, 999999], dtype=torch.int32, device="cuda")
    bo = torch.tensor([0, 2], dtype=torch.int64, device="cuda")
    outb = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(bpe.BpeError) as e:
        bpe.bpe_decode_batch(h, bad_ids.data_ptr(), 2, bo.data_ptr(), 1, outb.data_ptr(), 16, out.data_ptr(), True, s)
    assert e.value.code == 7
