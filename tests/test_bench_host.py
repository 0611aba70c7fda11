"""Host-side logic of bench.py (CPU): the source digest that ties committed ncu counters to a kernel
version, and the oracle-sample extrapolation over a workload's units."""
import os
import shutil

import pytest

import bench


@pytest.fixture()
def sources_copy(tmp_path, monkeypatch):
    """A copy of the decode kernel's sources under a temporary root, which bench reads instead."""
    src = os.path.join(bench.ROOT, "kv_cache_quantization_quantize_gb300", "csrc")
    dst = tmp_path / "kv_cache_quantization_quantize_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in bench.DECODE_SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return dst


def test_digest_ignores_comments_and_whitespace(sources_copy):
    base = bench.decode_source_digest()
    p = sources_copy / "tq_decode.cu"
    text = p.read_text(encoding="utf-8")
    p.write_text("// a comment line\n/* a block\n   comment */\n" + text.replace("\n", "\n  ", 3), encoding="utf-8")
    assert bench.decode_source_digest() == base


def test_digest_changes_with_code(sources_copy):
    base = bench.decode_source_digest()
    p = sources_copy / "tq_decode.cu"
    p.write_text(p.read_text(encoding="utf-8") + "\nstatic const int tq_digest_probe = 1;\n", encoding="utf-8")
    assert bench.decode_source_digest() != base


def test_profiled_traffic_follows_the_digest(sources_copy, tmp_path, monkeypatch):
    prof = tmp_path / "k_decode.md"
    digest = bench.decode_source_digest()
    prof.write_text(f"- source_digest: `{digest}`\n- traffic_bytes_per_launch: 12345\n", encoding="utf-8")
    assert bench.profiled_traffic(str(prof)) == 12345
    prof.write_text("- source_digest: `0000`\n- traffic_bytes_per_launch: 12345\n", encoding="utf-8")
    assert bench.profiled_traffic(str(prof)) is None


def test_oracle_units_and_sample_size(monkeypatch):
    monkeypatch.setattr(bench, "WL", dict(bench.WORKLOADS["long"]))
    assert bench.oracle_units() == 32 * 8 * 32
    assert 10 <= bench.oracle_sample_reps() < 150
    monkeypatch.setattr(bench, "WL", dict(bench.WORKLOADS["llama8b"]))
    assert bench.oracle_units() == 32 * 8
    assert bench.oracle_sample_reps() == 150
