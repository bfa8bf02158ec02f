"""Full-size workloads through bpe_encode_batch, as the bench launches it.

Every configuration is encoded whole on the GPU. Properties that hold at any
size are checked over the whole output: offsets start at 0, never decrease
and end at the token count; every id is in the vocabulary; tokens never
outnumber bytes. A seeded sample of documents is also compared id for id
with the oracle, which encodes each sampled document on its own (documents
are independent). The sample includes the first and last documents, documents
that straddle 4 KiB chunk edges and ones that straddle the 1024-chunk tiles
of the chunk scan.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

# sampled documents per configuration (C3's documents are 8 MiB each, which
# the oracle encodes in seconds apiece)
SAMPLES = {2: 240, 3: 2, 4: 40, 5: 400}


@pytest.fixture(scope="module")
def bpe():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import byte_level_bpe_pretokenize_gb300 as m
    return m


def _sample(offsets: np.ndarray, count: int, seed: int) -> list[int]:
    n_docs = len(offsets) - 1
    rng = np.random.default_rng(seed)
    picks = {0, n_docs - 1}
    # documents holding a chunk edge (multiple of 4096) and a tile edge
    # (multiple of 4096 * 1024)
    for edge_unit in (4096, 4096 * 1024):
        n_edges = int(offsets[-1] // edge_unit)
        if n_edges:
            for e in rng.integers(1, n_edges + 1, size=max(1, count // 4)):
                k = int(np.searchsorted(offsets, e * edge_unit, side="right")) - 1
                picks.add(min(max(k, 0), n_docs - 1))
    while len(picks) < min(count, n_docs):
        picks.add(int(rng.integers(0, n_docs)))
    return sorted(picks)


@pytest.mark.parametrize("cfg", [5, 2, 4, 3])
def test_full_workload(bpe, cfg):
    import torch
    data, offsets = workloads.docs(cfg)
    merges, vb, vo = workloads.table(cfg)
    n_vocab = len(vo) - 1
    h = bpe.bpe_build(merges, vb, vo, 0)
    try:
        d_data = torch.from_numpy(data).cuda()
        d_off = torch.from_numpy(offsets).cuda()
        d_ids = torch.empty(data.size, dtype=torch.int32, device="cuda")
        d_out = torch.empty(len(offsets), dtype=torch.int64, device="cuda")
        total = bpe.bpe_encode_batch(h, d_data.data_ptr(), data.size, d_off.data_ptr(), len(offsets) - 1,
                                     d_ids.data_ptr(), d_ids.numel(), d_out.data_ptr(), True,
                                     torch.cuda.current_stream().cuda_stream)
        out_off = d_out.cpu().numpy()
        ids_dev = d_ids[:total]
        assert 0 < total <= data.size
        assert ids_dev.min().item() >= 0 and ids_dev.max().item() < n_vocab
        assert out_off[0] == 0 and out_off[-1] == total
        assert (np.diff(out_off) >= 0).all()
        # no document has more tokens than bytes, and non-empty ones have some
        n_tok, n_byte = np.diff(out_off), np.diff(offsets)
        assert (n_tok <= n_byte).all() and ((n_byte == 0) == (n_tok == 0)).all()
        orc = oracle.Oracle(merges, vb, vo)
        for k in _sample(offsets, SAMPLES[cfg], 0xF0115 + cfg):
            want = orc.encode(bytes(data[offsets[k]:offsets[k + 1]]))
            got = ids_dev[out_off[k]:out_off[k + 1]].cpu().numpy().tolist()
            assert got == want, f"config {cfg}, document {k} ({offsets[k + 1] - offsets[k]} bytes) differs"
    finally:
        bpe.bpe_destroy(h)
