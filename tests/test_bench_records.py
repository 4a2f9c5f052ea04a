"""bench.py's use of the committed capture record on the CPU: the kernel
source hash ignores comments and blank lines but follows every code edit,
and a record is used only for the workload, kernel mode and source it was
taken on (otherwise the bench line's traffic figure is null)."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_records_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _with_sources(bench, tmp_path, texts):
    names = []
    for i, t in enumerate(texts):
        p = tmp_path / f"k{i}.cu"
        p.write_text(t)
        names.append(str(p))
    bench.KERNEL_SOURCES = names
    return bench.kernel_source_sha()


def test_source_hash_ignores_comments_only(tmp_path):
    b = _bench()
    base = _with_sources(b, tmp_path, ["int a = 1;  // one\n/* block\n comment */\nint b = 2;\n", "float c;\n"])
    same = _with_sources(b, tmp_path, ["\n\nint a = 1;  // another word\nint b = 2;  /* x */\n", "float c;  // c\n"])
    assert base == same
    assert _with_sources(b, tmp_path, ["int a = 2;\nint b = 2;\n", "float c;\n"]) != base
    assert _with_sources(b, tmp_path, ["int a = 1;\nint b = 2;\n", "double c;\n"]) != base


def test_capture_record_matches_workload_mode_and_source(tmp_path, monkeypatch):
    b = _bench()
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("int kernel_body;\n")
    b.KERNEL_SOURCES = [str(src)]
    rec = {"workload": "qwen3_8b", "mode": "default", "source_sha": b.kernel_source_sha(),
           "dram_bytes_read": 1.0, "dram_bytes_write": 2.0}
    (tmp_path / "profiles" / "lamp_fwd_traffic.json").write_text(json.dumps(rec))
    assert b._capture("qwen3_8b") is not None
    assert b._capture("gemma3_12b") is None
    assert b._capture("qwen3_8b", "pv8") is None
    src.write_text("int kernel_body_changed;\n")
    assert b._capture("qwen3_8b") is None
