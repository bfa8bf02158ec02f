"""bpe_train (the merge table trained on the GPU) against the host trainer
and the naive recount ("Tokenisierung", section "Byte Pair Encoding
schrittweise": count adjacent pairs, take the most frequent, ties to the
smallest ids, replace, count again)."""
from collections import Counter

import numpy as np
import pytest

import workloads
from tests.test_workloads import naive_train

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


def word_list(pieces):
    c = Counter(pieces)
    words = list(c)
    data = np.frombuffer(b"".join(words), np.uint8) if words else np.zeros(0, np.uint8)
    offsets = np.concatenate([[0], np.cumsum([len(w) for w in words])]).astype(np.int64)
    return data, offsets, np.array([c[w] for w in words], np.int64)


def test_ties_overlaps_and_stop(bpe):
    # ties: (a, b) and (c, d) once each -> the smaller ids first
    assert bpe.bpe_train(*word_list([b"cd", b"ab"]), 1).tolist() == [[ord("a"), ord("b"), 256]]
    assert bpe.bpe_train(*word_list([b"az", b"ay"]), 1).tolist() == [[ord("a"), ord("y"), 256]]
    # counts are weighted by word count; runs of equal symbols count every pair
    pieces = [b"aaaa"] * 3 + [b"ab"] * 5 + [b"x"]
    want = naive_train(pieces, 50)
    got = bpe.bpe_train(*word_list(pieces), 50)
    assert got.tolist() == want.tolist()
    assert len(got) < 50  # stops when no pair is left
    # empty input and zero merges
    assert bpe.bpe_train(np.zeros(0, np.uint8), np.zeros(1, np.int64), np.zeros(0, np.int64), 5).shape == (0, 3)
    assert bpe.bpe_train(*word_list([b"ab"]), 0).shape == (0, 3)


@pytest.mark.parametrize("seed", range(4))
def test_random_word_lists_equal_naive_recount(bpe, seed):
    rng = np.random.default_rng(seed)
    alphabet = rng.choice(np.frombuffer(b"abcdexyz 1'", np.uint8), size=rng.integers(2, 6), replace=False)
    pieces = [bytes(rng.choice(alphabet, size=int(rng.integers(1, 30)))) for _ in range(400)]
    want = naive_train(pieces, 200)
    got = bpe.bpe_train(*word_list(pieces), 200)
    assert got.tolist() == want.tolist()


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_workload_tables_equal_host_trainer(bpe, cfg):
    """The whole merge table of each workload: the GPU trainer on the host
    trainer's word list equals the host trainer's table row for row."""
    data, offsets, counts = workloads.train_words(workloads.corpus(cfg))
    want = workloads.table(cfg)[0]
    got = bpe.bpe_train(data, offsets, counts, workloads.n_merges(cfg))
    assert got.shape == want.shape, (got.shape, want.shape)
    if not np.array_equal(got, want):
        k = int(np.nonzero((got != want).any(axis=1))[0][0])
        raise AssertionError(f"config {cfg}: merge {k} differs: gpu {got[k].tolist()} host {want[k].tolist()}")
