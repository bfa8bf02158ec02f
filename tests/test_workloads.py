"""The seeded generators and the BPE trainer that make the inputs."""
from collections import Counter

import numpy as np
import pytest

import workloads


def naive_train(pieces: list[bytes], n_merges: int):
    """Recount every step: most frequent adjacent pair, ties to the smallest
    (left_id, right_id), replace left to right without overlap ("Tokenisierung",
    section "Byte Pair Encoding schrittweise")."""
    words = Counter(pieces)
    seqs = {w: list(w) for w in words}
    merges = []
    for k in range(n_merges):
        counts = Counter()
        for w, f in words.items():
            s = seqs[w]
            for i in range(len(s) - 1):
                counts[(s[i], s[i + 1])] += f
        if not counts:
            break
        best = max(counts.items(), key=lambda kv: (kv[1], -kv[0][0], -kv[0][1]))[0]
        new = 256 + k
        merges.append((best[0], best[1], new))
        for w in words:
            s, out, i = seqs[w], [], 0
            while i < len(s):
                if i + 1 < len(s) and (s[i], s[i + 1]) == best:
                    out.append(new)
                    i += 2
                else:
                    out.append(s[i])
                    i += 1
            seqs[w] = out
    return np.array(merges, dtype=np.int32).reshape(-1, 3)


def test_trainer_tie_break_smallest_ids():
    # (a, b) and (c, d) both occur once: the smaller ids win.
    m = workloads.train(np.frombuffer(b"cd!ab", np.uint8), 1)
    assert m.tolist() == [[ord("a"), ord("b"), 256]]
    # Equal left id: the smaller right id wins.
    m = workloads.train(np.frombuffer(b"az!ay", np.uint8), 1)
    assert m.tolist() == [[ord("a"), ord("y"), 256]]


def test_trainer_counts_pairs_within_pretokens_only():
    # "a b" never forms the pair (a, space) or (space, b) inside one piece
    # except as the leading space of " b".
    m = workloads.train(np.frombuffer(b"a b", np.uint8), 10)
    assert m.tolist() == [[ord(" "), ord("b"), 256]]


@pytest.mark.parametrize("cfg,nbytes", [(1, 16 << 10), (2, 8 << 10)])
def test_trainer_equals_naive_recount(cfg, nbytes):
    regex = pytest.importorskip("regex")  # noqa: F841
    from tests import brute_force
    text = bytes(workloads.corpus(cfg)[:nbytes])
    text = text.decode("utf-8", errors="ignore").encode()
    want = naive_train(brute_force.split(text), 120)
    got = workloads.train(np.frombuffer(text, np.uint8), 120)
    assert got.tolist() == want.tolist()


def test_docs_subset_is_slice_of_batch():
    data, off = workloads.docs(5, 0, 40)
    d2, o2 = workloads.docs(5, 10, 5)
    assert bytes(d2) == bytes(data[off[10]:off[15]])
    d3, _ = workloads.docs(5, 0, 40)
    assert bytes(d3) == bytes(data)


def test_doc_shapes():
    lens = workloads.doc_lengths(5, 0, 20000)
    assert lens.min() >= 60 and lens.max() <= 448
    lens = workloads.doc_lengths(1)
    assert len(lens) == 256 and lens.min() >= 1020 and lens.max() <= 4096
    data, off = workloads.docs(4, 0, 4)
    for k in range(4):
        d = bytes(data[off[k]:off[k + 1]])
        d.decode("utf-8")  # valid UTF-8
        assert 1024 <= len(d) <= 65536 * 10 // 9 + 4096 + 64
    data, off = workloads.docs(2, 0, 50)
    bytes(data).decode("utf-8")


def test_table_vocab_is_consistent():
    m, vb, vo = workloads.table(1)
    assert len(m) == 512
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    assert len(set(toks)) == len(toks)
    for a, b, c in m.tolist():
        assert toks[c] == toks[a] + toks[b]
        assert c == 256 + m.tolist().index([a, b, c])


def test_train_words_tile_the_corpus():
    text = workloads.corpus(2)[:200_000]
    data, offsets, counts = workloads.train_words(text)
    words = [bytes(data[offsets[i]:offsets[i + 1]]) for i in range(len(counts))]
    assert len(set(words)) == len(words) and all(words)
    assert int((np.diff(offsets) * counts).sum()) == text.size
    # the host trainer on the corpus equals the naive recount on the word list
    pieces = [w for w, c in zip(words, counts) for _ in range(int(c))]
    assert workloads.train(text, 40).tolist() == naive_train(pieces, 40).tolist()
