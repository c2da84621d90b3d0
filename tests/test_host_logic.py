"""Host-side logic that needs no GPU: the binding's refusal to run without the
compiled library, and the source hash that ties committed DRAM counters to the
kernel code they were taken on."""
import os
import shutil

import pytest

import bench
import block_scaled_mxfp4_activation_gb300 as mx


def test_missing_library_raises(monkeypatch, tmp_path):
    # No library and building disabled: loading fails loudly (no fallback path).
    monkeypatch.setattr(mx, "_lib", None)
    monkeypatch.setattr(mx._build, "LIB", str(tmp_path / "libmxfp4.so"))
    with pytest.raises(RuntimeError, match="not found"):
        mx.load_library(build_if_missing=False)


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "block_scaled_mxfp4_activation_gb300", "csrc")
    dst = tmp_path / "block_scaled_mxfp4_activation_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o", "*.so"))
    return dst


def test_source_hash_follows_code_not_comments(monkeypatch, tmp_path):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash()
    assert h0 == bench.source_hash()  # deterministic
    gemm = dst / "gemm.cu"
    text = gemm.read_text()
    # comment-only edits (line and block comments, spacing) keep the hash
    gemm.write_text("// a new line comment\n/* a block\n   comment */\n" + text.replace("\n", "\n  ", 3))
    assert bench.source_hash() == h0
    # a code edit changes it
    gemm.write_text(text + "\nstatic int mxfp4_probe_symbol = 1;\n")
    assert bench.source_hash() != h0
