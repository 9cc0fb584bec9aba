"""The traffic record's freshness hash (bench.source_hash): it follows the
attention's code, not its comments or layout, and not the other kernels."""
import os
import shutil

import bench


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "mla_decode_attention_absorbed_gb300", "csrc")
    dst = tmp_path / "mla_decode_attention_absorbed_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in os.listdir(src):
        shutil.copy(os.path.join(src, name), dst / name)
    return dst


def _hash_at(root, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(root))
    return bench.source_hash()


def test_hash_ignores_comments_and_other_kernels(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    h0 = _hash_at(tmp_path, monkeypatch)
    attn = dst / "attn_tc.cu"
    attn.write_text("// a new comment line\n/* and a block\n   comment */\n\n" + attn.read_text())
    assert _hash_at(tmp_path, monkeypatch) == h0
    proj = dst / "proj_tc.cu"  # not one of the attention's sources
    proj.write_text(proj.read_text() + "\nstatic int unused_symbol = 1;\n")
    assert _hash_at(tmp_path, monkeypatch) == h0


def test_hash_follows_the_attention_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    h0 = _hash_at(tmp_path, monkeypatch)
    for name in bench.ATTN_SOURCES:
        f = dst / name
        text = f.read_text()
        f.write_text(text + "\nstatic int changed_code = 1;\n")
        assert _hash_at(tmp_path, monkeypatch) != h0, name
        f.write_text(text)
    assert _hash_at(tmp_path, monkeypatch) == h0
