"""Host-side rules of bench.py (no GPU): the captured DRAM traffic of the split-KV kernel
is reported only for the kernel sources it was taken on, judged by a hash of their code
that leaves comments and blank lines out."""

import os
import shutil

import bench


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "paged_latent_attention_mla_gb300", "csrc")
    dst = tmp_path / "paged_latent_attention_mla_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    return dst


def test_hash_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.kernel_sources_sha256()
    p = dst / bench.KERNEL_SOURCES[0]
    text = p.read_text()
    p.write_text("// a new comment line\n\n" + text.replace("\n", "  // trailing note\n", 1))
    assert bench.kernel_sources_sha256() == before


def test_hash_changes_with_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.kernel_sources_sha256()
    p = dst / bench.KERNEL_SOURCES[0]
    p.write_text(p.read_text() + "\nstatic int probe_extra_symbol = 1;\n")
    assert bench.kernel_sources_sha256() != before


def test_traffic_withheld_for_other_sources(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = dst / bench.KERNEL_SOURCES[0]
    p.write_text(p.read_text() + "\nstatic int probe_extra_symbol = 1;\n")
    for workload in bench.NCU_TRAFFIC:
        assert bench.measured_traffic(workload) is None
    assert bench.measured_traffic("no such workload") is None
