"""The bench's traffic record is keyed to the project kernel's code: a
comment edit keeps it, a code change drops it (the line then reports null)."""
import importlib.util
import json
import os
import shutil

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def copy_sources(b, dst):
    for src in b.KERNEL_SOURCES:
        os.makedirs(os.path.join(dst, os.path.dirname(src)), exist_ok=True)
        shutil.copy(os.path.join(ROOT, src), os.path.join(dst, src))


def test_hash_ignores_comments_not_code(tmp_path):
    b = load_bench()
    copy_sources(b, str(tmp_path))
    b.ROOT = str(tmp_path)
    base = b.kernel_source_hash()
    first = os.path.join(str(tmp_path), b.KERNEL_SOURCES[0])
    with open(first, "a") as f:
        f.write("\n// a comment\n/* another\n   one */\n")
    assert b.kernel_source_hash() == base
    with open(first, "a") as f:
        f.write("static int unused_symbol_for_the_test = 1;\n")
    assert b.kernel_source_hash() != base


def test_record_is_used_only_for_its_shape_and_source(tmp_path):
    b = load_bench()
    copy_sources(b, str(tmp_path))
    os.makedirs(os.path.join(str(tmp_path), "profiles"))
    b.ROOT = str(tmp_path)
    rec = {"source_sha256_16": b.kernel_source_hash(), "workload_base": "llama2-7b",
           "dram_bytes_read": 300, "dram_bytes_write": 100, "captured_layers": 4}
    with open(os.path.join(str(tmp_path), "profiles", "project_kernel_traffic.json"), "w") as f:
        json.dump(rec, f)
    assert b.profiled_traffic("llama2-7b", 32) == 400 * 32 / 4
    assert b.profiled_traffic("llama2-13b", 40) is None
    with open(os.path.join(str(tmp_path), b.KERNEL_SOURCES[0]), "a") as f:
        f.write("static int changed = 2;\n")
    assert b.profiled_traffic("llama2-7b", 32) is None
