"""bpe_encode_batch_host (host buffers, pipelined slices) against
bpe_encode_batch (device buffers), through the C ABI."""
import numpy as np
import pytest

import workloads
from tests.gpu_util import assert_same_encoding, batch, gpu_encode

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


@pytest.fixture(scope="module")
def handle(bpe):
    m, vb, vo = workloads.table(1)
    h = bpe.bpe_build(m, vb, vo, 0)
    yield h
    bpe.bpe_destroy(h)


def host_encode(bpe, h, data, offsets, capacity=None, pinned=True):
    import torch
    cap = data.size if capacity is None else capacity
    t_data = torch.from_numpy(data if data.size else np.zeros(1, np.uint8))
    t_off = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64))
    t_ids = torch.full((max(1, cap),), -7, dtype=torch.int32)
    t_out = torch.full((len(offsets),), -7, dtype=torch.int64)
    if pinned:
        t_data, t_off, t_ids, t_out = (t.pin_memory() for t in (t_data, t_off, t_ids, t_out))
    total = bpe.bpe_encode_batch_host(h, t_data.data_ptr(), data.size, t_off.data_ptr(), len(offsets) - 1,
                                      t_ids.data_ptr(), cap, t_out.data_ptr(), True,
                                      torch.cuda.current_stream().cuda_stream)
    return t_ids.numpy(), t_out.numpy(), total


@pytest.mark.parametrize("pinned", [True, False])
def test_many_slices_match_device_path(bpe, handle, pinned):
    # ~48 MB of serving-batch documents: 8 slices of ~6 MB
    data, off = workloads.docs(5, 0, 180_000)
    want = gpu_encode(handle, data, off)
    ids, out, total = host_encode(bpe, handle, data, off, pinned=pinned)
    assert total == len(want[0])
    assert_same_encoding((ids[:total], out), want, data, off, "host path")


def test_edges_long_documents_and_gaps(bpe, handle):
    # a document longer than a slice, empty documents, bytes outside documents
    docs = [b"junk", b"", b"x" * (9 << 20), b"it's  \n\tx", b"", "Grüße 🐈 你好".encode() * 1000, b"q" * 70_001]
    data, off = batch(docs)
    off = off.copy()
    off[0] = 4  # the first 4 bytes lie outside every document
    want = gpu_encode(handle, data, off)
    ids, out, total = host_encode(bpe, handle, data, off)
    assert total == len(want[0])
    assert_same_encoding((ids[:total], out), want, data, off, "host path edges")


def test_empty_and_capacity(bpe, handle):
    for n_docs in (0, 3):
        ids, out, total = host_encode(bpe, handle, np.zeros(0, np.uint8), np.zeros(n_docs + 1, np.int64))
        assert total == 0 and (out == 0).all()
    data, off = workloads.docs(5, 0, 2000)
    full = gpu_encode(handle, data, off)[0]
    with pytest.raises(bpe.BpeError) as err:
        host_encode(bpe, handle, data, off, capacity=100)
    assert err.value.code == 2
    # the ids that fit are written, nothing past them
    ids, out, total = None, None, None
    import torch
    t_data = torch.from_numpy(data).pin_memory()
    t_off = torch.from_numpy(off).pin_memory()
    t_ids = torch.full((160,), -7, dtype=torch.int32).pin_memory()
    t_out = torch.full((len(off),), -7, dtype=torch.int64).pin_memory()
    with pytest.raises(bpe.BpeError):
        bpe.bpe_encode_batch_host(handle, t_data.data_ptr(), data.size, t_off.data_ptr(), len(off) - 1,
                                  t_ids.data_ptr(), 100, t_out.data_ptr(), True,
                                  torch.cuda.current_stream().cuda_stream)
    got = t_ids.numpy()
    assert (got[:100] == full[:100]).all() and (got[100:] == -7).all()
