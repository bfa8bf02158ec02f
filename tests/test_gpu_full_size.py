"""Full-size workloads through bpe_encode_batch, compared whole with the oracle.

Every configuration is encoded whole on the GPU, in one call, as the bench
launches it, and the oracle encodes the same batch on every host core
(oracle.sharded: byte-balanced document shards, one pinned process each).
The two id streams and document offset arrays must be equal element for
element; the FNV-1a 64 digests of both id streams are printed ("Hugging Face
Tokenizers v1", section "performance benchmarks": the output ids are checked
by their FNV-1a hash). Properties that hold at any size are checked as well.
"""
import numpy as np
import pytest

import workloads
from oracle import sharded

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


def gpu_encode_whole(bpe, cfg):
    import torch
    data, offsets = workloads.docs(cfg)
    merges, vb, vo = workloads.table(cfg)
    h = bpe.bpe_build(merges, vb, vo, 0)
    try:
        d_data = torch.from_numpy(data).cuda()
        d_off = torch.from_numpy(offsets).cuda()
        d_ids = torch.empty(data.size, dtype=torch.int32, device="cuda")
        d_out = torch.empty(len(offsets), dtype=torch.int64, device="cuda")
        def call():
            return bpe.bpe_encode_batch(h, d_data.data_ptr(), data.size, d_off.data_ptr(), len(offsets) - 1,
                                        d_ids.data_ptr(), d_ids.numel(), d_out.data_ptr(), True,
                                        torch.cuda.current_stream().cuda_stream)
        total = call()
        ids = d_ids[:total].cpu().numpy()
        out_off = d_out.cpu().numpy()
        # the same handle again, twice (nothing of a call may leak into the next)
        for _ in range(2):
            d_ids.fill_(-7)
            d_out.fill_(-7)
            assert call() == total
            assert np.array_equal(d_ids[:total].cpu().numpy(), ids), f"config {cfg}: a repeated call differs"
            assert np.array_equal(d_out.cpu().numpy(), out_off), f"config {cfg}: a repeated call's offsets differ"
    finally:
        bpe.bpe_destroy(h)
    return data, offsets, (merges, vb, vo), ids, out_off


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_workload_equals_oracle(bpe, cfg):
    data, offsets, (merges, vb, vo), ids, out_off = gpu_encode_whole(bpe, cfg)
    n_vocab = len(vo) - 1
    total = len(ids)
    assert 0 < total <= data.size
    assert ids.min() >= 0 and ids.max() < n_vocab
    assert out_off[0] == 0 and out_off[-1] == total
    n_tok, n_byte = np.diff(out_off), np.diff(offsets)
    assert (n_tok <= n_byte).all() and ((n_byte == 0) == (n_tok == 0)).all()

    ref = sharded.encode(merges, vb, vo, data, offsets)
    g_digest, o_digest = workloads.fnv1a64(ids), workloads.fnv1a64(ref["ids"])
    print(f"\nconfig {cfg} ({workloads.NAMES[cfg]}): {len(offsets) - 1} documents, {data.size} bytes, "
          f"{total} tokens; FNV-1a 64 gpu {g_digest:016x} oracle {o_digest:016x}; oracle on "
          f"{ref['procs']} processes ({ref['cpu_model']}) {ref['wall_s']:.1f} s")
    assert np.array_equal(out_off, ref["offsets"]), f"config {cfg}: document offsets differ from the oracle"
    if not np.array_equal(ids, ref["ids"]):
        k = int(np.nonzero(ids[:min(len(ids), len(ref['ids']))] != ref["ids"][:min(len(ids), len(ref['ids']))])[0][0])
        doc = int(np.searchsorted(out_off, k, side="right")) - 1
        raise AssertionError(f"config {cfg}: ids differ from the oracle first at token {k} (document {doc})")
    assert g_digest == o_digest


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_workload_decodes_back(bpe, cfg):
    """decode(encode(x)) == x on every whole workload ("Tokenisierung",
    section "Prüfe zuerst den Roundtrip"), byte for byte, with the document
    offsets; the ids come from the GPU encoder (equal to the oracle's by the
    test above)."""
    import torch
    data, offsets = workloads.docs(cfg)
    merges, vb, vo = workloads.table(cfg)
    h = bpe.bpe_build(merges, vb, vo, 0)
    try:
        s = torch.cuda.current_stream().cuda_stream
        d_data = torch.from_numpy(data).cuda()
        d_off = torch.from_numpy(offsets).cuda()
        d_ids = torch.empty(data.size, dtype=torch.int32, device="cuda")
        d_ioff = torch.empty(len(offsets), dtype=torch.int64, device="cuda")
        total = bpe.bpe_encode_batch(h, d_data.data_ptr(), data.size, d_off.data_ptr(), len(offsets) - 1,
                                     d_ids.data_ptr(), d_ids.numel(), d_ioff.data_ptr(), True, s)
        del d_data
        out = torch.full((data.size + 64,), 0xAB, dtype=torch.uint8, device="cuda")
        out_off = torch.full((len(offsets),), -7, dtype=torch.int64, device="cuda")
        for _ in range(2):  # twice on one handle
            n = bpe.bpe_decode_batch(h, d_ids.data_ptr(), total, d_ioff.data_ptr(), len(offsets) - 1, out.data_ptr(),
                                     out.numel(), out_off.data_ptr(), True, s)
            assert n == data.size
            assert np.array_equal(out[:n].cpu().numpy(), data), f"config {cfg}: decoded bytes differ"
            assert (out[n:].cpu().numpy() == 0xAB).all()
            assert np.array_equal(out_off.cpu().numpy(), offsets), f"config {cfg}: decoded offsets differ"
    finally:
        bpe.bpe_destroy(h)
