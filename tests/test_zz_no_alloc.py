"""bpe_encode_batch_noalloc (fixed static scratch, no device allocation)
against bpe_encode_batch, through the C ABI.

Collected last so that it also runs after every other GPU test has used the
library in the same process; it passes on its own too.
"""
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


def _device(data, offsets):
    import torch
    d_data = torch.from_numpy(data if data.size else np.zeros(1, np.uint8)).cuda()
    d_off = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64)).cuda()
    d_ids = torch.full((max(1, data.size),), -7, dtype=torch.int32, device="cuda")
    d_out = torch.full((len(offsets),), -7, dtype=torch.int64, device="cuda")
    return d_data, d_off, d_ids, d_out


def _noalloc(bpe, h, dev, n_bytes, want_total=True):
    import torch
    d_data, d_off, d_ids, d_out = dev
    return bpe.bpe_encode_batch_noalloc(h, d_data.data_ptr(), n_bytes, d_off.data_ptr(), d_off.numel() - 1,
                                        d_ids.data_ptr(), d_ids.numel(), d_out.data_ptr(), want_total,
                                        torch.cuda.current_stream().cuda_stream)


def _batches():
    """Two different batches: serving-sized ASCII documents, and mixed UTF-8
    with pre-tokens longer than shared memory (they use the scratch pool)."""
    a = workloads.docs(5, 0, 4000)
    b_docs = [bytes(workloads.docs(2, 0, 120)[0][:700_000]), b"7" * 5000, b"q" * 70_001, "中".encode() * 1500,
              b"", b"it's  \n\tx", b"\xff\xfe abc \x80"]
    b = batch(b_docs)
    assert a[0].size > 1_000_000 and b[0].size > 600_000
    return [a, b]


def test_two_calls_in_a_row_match_bpe_encode_batch(bpe, handle):
    import torch
    batches = _batches()
    want = [gpu_encode(handle, d, o) for d, o in batches]
    devs = [_device(d, o) for d, o in batches]
    # Two calls queued back to back on one stream, no wait between them.
    _noalloc(bpe, handle, devs[0], batches[0][0].size, want_total=False)
    total = _noalloc(bpe, handle, devs[1], batches[1][0].size)
    torch.cuda.synchronize()
    assert total == len(want[1][0])
    for k, ((d, o), dev, w) in enumerate(zip(batches, devs, want)):
        got = (dev[2][:len(w[0])].cpu().numpy(), dev[3].cpu().numpy())
        assert_same_encoding(got, w, d, o, f"no-alloc call {k}")
    # Two more calls in a row, each waited for, in the other order.
    for k in (1, 0):
        d, o = batches[k]
        dev = _device(d, o)
        total = _noalloc(bpe, handle, dev, d.size)
        got = (dev[2][:total].cpu().numpy(), dev[3].cpu().numpy())
        assert_same_encoding(got, want[k], d, o, f"no-alloc repeat {k}")


def test_limit_and_empty_batch(bpe, handle):
    import torch
    limit = bpe.NOALLOC_MAX_BYTES
    lens = workloads.doc_lengths(5, 0, limit // 200)
    n = int(np.searchsorted(np.cumsum(lens), limit))
    d, o = workloads.docs(5, 0, n)
    d = np.concatenate([d, np.frombuffer(b"x" * (limit - d.size), np.uint8)])
    o = np.append(o, limit)
    assert d.size == limit
    dev = _device(d, o)
    total = _noalloc(bpe, handle, dev, limit)
    got = (dev[2][:total].cpu().numpy(), dev[3].cpu().numpy())
    assert_same_encoding(got, gpu_encode(handle, d, o), d, o, "batch at the limit")
    # One byte more is rejected before anything is queued.
    big = _device(np.zeros(limit + 1, np.uint8), np.array([0, limit + 1], np.int64))
    with pytest.raises(bpe.BpeError) as err:
        _noalloc(bpe, handle, big, limit + 1)
    assert err.value.code == 1 and "4 MiB" in str(err.value)
    # the limit in the message is the binding's constant
    assert f"limit of {limit} bytes" in str(err.value)
    torch.cuda.synchronize()
    assert (big[2].cpu().numpy() == -7).all() and (big[3].cpu().numpy() == -7).all()
    # Empty batches.
    for n_docs in (0, 5):
        dev = _device(np.zeros(0, np.uint8), np.zeros(n_docs + 1, np.int64))
        assert _noalloc(bpe, handle, dev, 0) == 0
        assert (dev[3].cpu().numpy() == 0).all()


def test_calls_allocate_no_device_memory(bpe):
    """A fresh handle, used only through the no-alloc call: after the first
    call (which looks up the scratch address once per device), further calls
    leave the device's free memory unchanged, and the handle's own workspace
    is never created."""
    import torch
    m, vb, vo = workloads.table(1)
    h = bpe.bpe_build(m, vb, vo, 0)
    try:
        d, o = workloads.docs(5, 0, 3000)
        dev = _device(d, o)
        want = None
        _noalloc(bpe, h, dev, d.size)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(3):
            total = _noalloc(bpe, h, dev, d.size)
            got = (dev[2][:total].cpu().numpy(), dev[3].cpu().numpy())
            if want is None:
                want = got
            assert_same_encoding(got, want, d, o, "repeat")
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert bpe.bpe_workspace_bytes(h) == 0
    finally:
        bpe.bpe_destroy(h)
