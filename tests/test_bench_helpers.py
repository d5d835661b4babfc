"""bench.py's roofline bookkeeping on the CPU: DRAM traffic from a committed
ncu summary is reported only while the kernel sources still hash to the
ones that summary was taken on."""
import os

import bench


def _doc(tmp_path, digest, traffic=123456):
    p = tmp_path / "profile.md"
    p.write_text(f"# a summary\n\nsource_sha256: {digest}\ndram_bytes_per_launch: {traffic}\n")
    return str(p)


def test_traffic_is_reported_for_the_profiled_sources(tmp_path):
    for sources in (bench.KERNEL_SOURCES, bench.KERNEL_SOURCES_CHUNK):
        doc = _doc(tmp_path, bench.kernel_source_hash(sources))
        assert bench.profiled_traffic(doc, sources) == 123456.0


def test_traffic_is_dropped_once_the_sources_change(tmp_path):
    doc = _doc(tmp_path, "0" * 64)
    assert bench.profiled_traffic(doc, bench.KERNEL_SOURCES) is None
    # a summary without the fields, or none at all
    empty = tmp_path / "empty.md"
    empty.write_text("no figures here\n")
    assert bench.profiled_traffic(str(empty), bench.KERNEL_SOURCES) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md"), bench.KERNEL_SOURCES) is None


def test_the_hash_covers_every_listed_source():
    # each source file named for a profile exists in the package
    for name in set(bench.KERNEL_SOURCES) | set(bench.KERNEL_SOURCES_CHUNK):
        assert os.path.exists(os.path.join(bench.REPO, "paged_attention_kv_gb300", "csrc", name)), name
    assert bench.kernel_source_hash(bench.KERNEL_SOURCES) != bench.kernel_source_hash(bench.KERNEL_SOURCES_CHUNK)
