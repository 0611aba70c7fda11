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


def test_config_depends_on_the_workload_only(monkeypatch):
    """Both arms print bench_config(): it must not depend on anything measured."""
    monkeypatch.setattr(bench, "WL", dict(bench.WORKLOADS["llama8b"]))
    a = bench.bench_config(1)
    b = bench.bench_config(1, "hybrid", "contiguous")
    assert a == b
    # 32 layers x (8 KV heads x (32640 packed x 92 B + 128 ring x 512 B) + 32 q heads x 128 x 6 B)
    assert bench.nominal_step_bytes(bench.WL) == 32 * (8 * (32640 * 92 + 128 * 512) + 32 * 128 * 6)
    assert "786 MB" in a["l2"]
    assert bench.bench_config(1, layout="paged")["layout"].startswith("paged")


def test_record_bytes_of_the_workloads():
    assert bench.record_bytes(bench.WORKLOADS["llama8b"]) == 52 + 40
    assert bench.record_bytes(bench.WORKLOADS["batched"]) == 52 + 72
    assert bench.record_bytes(bench.WORKLOADS["d256"]) == 100 + 80
    assert bench.record_bytes(dict(bench.WORKLOADS["llama8b"], kb=4, vb=4)) == 68 + 72
