"""The all-core oracle (oracle.sharded) equals the single-process oracle.

Documents are independent, so encoding byte-balanced shards in separate
processes and concatenating must give the single-process encoding exactly.
Also pins the FNV-1a 64 digest used to compare id streams to the published
test vectors of FNV-1a 64.
"""
import numpy as np

import oracle
import workloads
from oracle import sharded


def test_fnv1a64_published_vectors():
    assert workloads.fnv1a64(np.frombuffer(b"", np.uint8)) == 0xCBF29CE484222325
    assert workloads.fnv1a64(np.frombuffer(b"a", np.uint8)) == 0xAF63DC4C8601EC8C
    assert workloads.fnv1a64(np.frombuffer(b"foobar", np.uint8)) == 0x85944171F73967E8
    # chaining over parts equals one pass over the whole
    h = workloads.fnv1a64(np.frombuffer(b"foo", np.uint8))
    assert workloads.fnv1a64(np.frombuffer(b"bar", np.uint8), h) == 0x85944171F73967E8


def test_shards_cover_documents_in_order():
    offsets = np.array([0, 5, 5, 90, 100, 400, 401, 1000], dtype=np.int64)
    for n in (1, 2, 3, 7, 20):
        s = sharded.shards(offsets, n)
        assert s[0][0] == 0 and sum(c for _, c in s) == len(offsets) - 1
        assert all(a + c == b for (a, c), (b, _) in zip(s[:-1], s[1:]))
    assert sharded.shards(np.zeros(1, np.int64), 4) == []


def test_sharded_equals_single_process():
    merges, vb, vo = workloads.table(1)
    data, offsets = workloads.docs(1, 0, 96)
    # empty documents at the start, middle and end
    data = np.concatenate([data, np.frombuffer(b"it's  \n\tx", np.uint8)])
    offsets = np.concatenate([[0, 0], offsets, offsets[-1:], [offsets[-1] + 9, offsets[-1] + 9]]).astype(np.int64)
    want_ids, want_off = oracle.Oracle(merges, vb, vo).encode_batch(data, offsets)
    got = sharded.encode(merges, vb, vo, data, offsets, procs=3)
    assert np.array_equal(got["offsets"], want_off)
    assert np.array_equal(got["ids"], want_ids)
    assert got["procs"] >= 1 and got["wall_s"] >= 0
