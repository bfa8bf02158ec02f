"""The C ABI: the library loads, exports every call the header declares, and
bpe_build's host-side table checks reject bad tables (no GPU needed)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import workloads
from tests.tables import table_from_pairs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bpe():
    import __graft_entry__
    __graft_entry__.build()
    import byte_level_bpe_pretokenize_gb300 as m
    return m


def declared_calls():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(bpe_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_call(bpe):
    names = declared_calls()
    assert len(names) >= 8
    lib = ctypes.CDLL(bpe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(bpe.EXPORTS)


def test_binding_has_same_names(bpe):
    for n in declared_calls():
        if n != "bpe_last_error":
            assert callable(getattr(bpe, n)), n


def _build_code(bpe, m, vb, vo):
    h = ctypes.c_void_p()
    m = np.ascontiguousarray(np.asarray(m, dtype=np.int32).reshape(-1, 3))
    vb = np.ascontiguousarray(vb, dtype=np.uint8)
    vo = np.ascontiguousarray(vo, dtype=np.int64)
    return bpe.lib().bpe_build(m.ctypes.data if m.size else None, len(m), vb.ctypes.data, vo.ctypes.data,
                               len(vo) - 1, 0, ctypes.byref(h))


BAD_TABLE = 4


def test_build_rejects_missing_byte(bpe):
    m, vb, vo = table_from_pairs([(b"a", b"b")])
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    toks[7] = b""  # byte 7 has no token
    lens = np.array([len(t) for t in toks])
    vo2 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    vb2 = np.frombuffer(b"".join(toks), np.uint8)
    assert _build_code(bpe, m, vb2, vo2) == BAD_TABLE


def test_build_rejects_inconsistent_merge(bpe):
    m, vb, vo = table_from_pairs([(b"a", b"b"), (b"ab", b"c")])
    m = m.copy()
    m[1, 1] = ord("d")  # (ab, d) cannot make "abc"
    assert _build_code(bpe, m, vb, vo) == BAD_TABLE


def test_build_rejects_duplicate_pair(bpe):
    m, vb, vo = table_from_pairs([(b"a", b"b")])
    m2 = np.concatenate([m, m])
    assert _build_code(bpe, m2, vb, vo) == BAD_TABLE


def test_build_rejects_duplicate_token_bytes(bpe):
    m, vb, vo = table_from_pairs([(b"a", b"b")], n_vocab=258)
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    toks[257] = b"ab"
    lens = np.array([len(t) for t in toks])
    vo2 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    vb2 = np.frombuffer(b"".join(toks), np.uint8)
    assert _build_code(bpe, m, vb2, vo2) == BAD_TABLE


def test_build_rejects_id_out_of_range(bpe):
    m, vb, vo = table_from_pairs([(b"a", b"b")])
    m = m.copy()
    m[0, 0] = 10 ** 6
    assert _build_code(bpe, m, vb, vo) == BAD_TABLE


def test_null_handle_is_invalid_arg(bpe):
    rc = bpe.lib().bpe_encode_batch(None, None, 0, None, 0, None, 0, None, None, None)
    assert rc == 1
    assert bpe.lib().bpe_destroy(None) == 1


def test_workload_tables_pass_host_checks(bpe):
    # Valid tables get past the table checks (the call then needs a device).
    for cfg in (1,):
        m, vb, vo = workloads.table(cfg)
        rc = _build_code(bpe, m, vb, vo)
        assert rc in (0, 3)  # OK on a GPU machine, CUDA error without a device


def test_merges_monotone_host_only(bpe):
    # "Tokenisierung", section "Byte Pair Encoding schrittweise": a trainer
    # merges pairs of the symbols that exist, so its tables are monotone.
    m, vb, vo = table_from_pairs([(b"a", b"b"), (b"ab", b"a")])
    assert bpe.bpe_merges_monotone(m, len(vo) - 1)
    # the abab example: (ab, a) at rank 0 uses "ab", which rank 1 makes
    m, vb, vo = table_from_pairs([(b"ab", b"a"), (b"a", b"b")], ids=[257, 256])
    assert not bpe.bpe_merges_monotone(m, len(vo) - 1)
    assert bpe.bpe_merges_monotone(np.zeros((0, 3), np.int32), 256)
    merges, _, vo5 = workloads.table(5)
    assert bpe.bpe_merges_monotone(merges, len(vo5) - 1)
    # a token made by two rules counts from its lowest rank
    m, vb, vo = table_from_pairs([(b"a", b"b"), (b"b", b"c"), (b"ab", b"c"), (b"a", b"bc"), (b"abc", b"a")],
                                 ids=[256, 257, 258, 258, 259])
    assert bpe.bpe_merges_monotone(m, len(vo) - 1)
    with pytest.raises(bpe.BpeError):
        bpe.bpe_merges_monotone(np.array([[1, 2, 999]], np.int32), 300)


def test_measurement_hooks_check_their_arguments(bpe):
    L = bpe.lib()
    # a null handle, and a wrong event count, are rejected before anything is kept
    assert L.bpe_set_phase_events(None, None, 0) == 1
    assert L.bpe_set_timing_events(None, None, None) == 1
    assert bpe.ENCODE_LAUNCHES == len(bpe.ENCODE_KERNELS)
    hdr = open(os.path.join(ROOT, "include", "bpe_gb300.h")).read()
    assert f"#define BPE_ENCODE_LAUNCHES {bpe.ENCODE_LAUNCHES}" in hdr
    # the kernel order the header states is the binding's
    assert ", ".join(bpe.ENCODE_KERNELS) in " ".join(hdr.replace("*", " ").split())
    with pytest.raises(ValueError):
        bpe.PhaseEvents([0] * 3)


def test_call_memo_modes_checked(bpe):
    L = bpe.lib()
    assert L.bpe_set_call_memo(None, bpe.MEMO_AUTO) == 1
    hdr = open(os.path.join(ROOT, "include", "bpe_gb300.h")).read()
    for name, v in (("BPE_MEMO_OFF", bpe.MEMO_OFF), ("BPE_MEMO_ON", bpe.MEMO_ON), ("BPE_MEMO_AUTO", bpe.MEMO_AUTO)):
        assert f"#define {name} {v}" in hdr
