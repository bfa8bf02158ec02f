"""Host-side helpers of bench.py (no GPU): the algorithmic-bytes formula of
the roofline, the kernel-source hash that keys the committed DRAM-traffic
profile, and the lookup of that profile."""
import json

import bench


def test_algorithmic_bytes_formula():
    # input bytes + document offsets read, ids (4 B) + document offsets written
    n_bytes, n_docs, n_tok = 1_073_661_860, 4_194_304, 188_698_661
    want = n_bytes + 8 * (n_docs + 1) + 4 * n_tok + 8 * (n_docs + 1)
    assert bench.algorithmic_bytes(n_bytes, n_docs, n_tok) == want == 1_895_565_384


def test_kernel_hash_ignores_comments_only(tmp_path, monkeypatch):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {  // twice\n  return 2 * x; /* plain */\n}\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", [str(a)])
    h0 = bench.kernel_hash()
    a.write_text("// a header comment\nint f(int x) {\n  return 2 * x;  // other words\n}\n")
    assert bench.kernel_hash() == h0
    a.write_text("int f(int x) {\n  return 3 * x;\n}\n")
    assert bench.kernel_hash() != h0


def test_traffic_profile_keyed_by_hash(tmp_path, monkeypatch):
    a = tmp_path / "k.cu"
    a.write_text("int g;\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", [str(a)])
    prof = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(prof))
    assert bench.traffic_from_profile() is None  # no file
    prof.write_text(json.dumps({"kernel_source_sha256_16": bench.kernel_hash(), "dram_bytes_per_full_call": 123}))
    assert bench.traffic_from_profile() == 123
    a.write_text("int g2;\n")  # the kernels changed since the capture
    assert bench.traffic_from_profile() is None
