"""Host-side pieces of bench.py that decide what the JSON line reports, checked without
a GPU: the roofline's algorithmic bytes for the headline scan (every visible MXFP4
indexer row once: 68 bytes an entry, CSA2 page «890 字节是怎么来的»; plus the bf16
queries and the head weights), the headline workload's shape, and the rule that a
committed ncu traffic figure is used only while the kernel sources it was taken on are
unchanged."""
import os

import pytest

import bench


def test_headline_scan_bytes_per_launch():
    w = bench.FP4Decode()
    assert (w.B, w.N, w.H_I, w.k, w.window, w.n_keep, w.block) == (8, 1 << 20, 64, 512, 128, 2048, 8)
    # decode at context L = 2^20: the query sits at t = L - 1 and sees V = t entries (m = 1)
    assert w.V == (1 << 20) - 1
    keys = 8 * ((1 << 20) - 1) * 68
    queries = 8 * 64 * (128 * 2 + 4)          # bf16 query rows and fp32 head weights
    assert w.main_amount() == keys + queries == 570_557_920
    # about 71.3 MB of indexer keys per query at 1M
    assert abs(((1 << 20) - 1) * 68 / 1e6 - 71.3) < 0.05


def test_v4pro_variant_keeps_the_scan_and_changes_the_selection():
    v = bench.V4ProDecode()
    assert (v.H, v.k) == (128, 1024)
    assert v.main_amount() == bench.FP4Decode().main_amount()


def _profile(tmp_path, text):
    d = tmp_path / "profiles"
    d.mkdir(exist_ok=True)
    (d / "p.txt").write_text(text)


def test_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _profile(tmp_path, "# comment: ignored\nkernel_source_sha256_16: abc123\ndram_bytes_per_launch: 12345\n")
    assert bench._profile_traffic("p.txt", "abc123") == 12345.0
    assert bench._profile_traffic("p.txt", "other") is None
    assert bench._profile_traffic("missing.txt", "abc123") is None
    _profile(tmp_path, "kernel_source_sha256_16: abc123\ndram_bytes_per_launch: not a number\n")
    assert bench._profile_traffic("p.txt", "abc123") is None


def test_kernel_hash_covers_every_listed_source(tmp_path, monkeypatch):
    src = tmp_path / "compressed_sparse_attention_06_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "a.cu").write_text("one")
    (src / "b.cuh").write_text("two")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench._kernel_hash(("a.cu", "b.cuh"))
    (src / "b.cuh").write_text("two, changed")
    assert bench._kernel_hash(("a.cu", "b.cuh")) != h
    assert len(h) == 16


def test_committed_headline_profile_is_parsable():
    w = bench.FP4Decode
    path = os.path.join(bench.ROOT, "profiles", w.profile)
    assert os.path.exists(path)
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    assert len(kv["kernel_source_sha256_16"]) == 16
    # DRAM traffic of one 1M launch: at least the algorithmic bytes, and within 10 % of them
    t = float(kv["dram_bytes_per_launch"])
    assert w().main_amount() <= t <= 1.1 * w().main_amount()
