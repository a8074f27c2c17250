"""bench.py keys recorded DRAM traffic to the code of the kernel sources: comment edits keep the
key, code edits change it."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_lines_ignore_comments_and_blank_lines():
    b = _bench()
    a = "int x = 1;  // one\n\n// a comment line\nint y = 2;\n"
    c = "int x = 1;  // the first\n// another comment\n\n\nint y = 2;   \n"
    assert b._code_lines(a) == b._code_lines(c) == "int x = 1;\nint y = 2;"


def test_code_lines_see_code_changes_and_keep_strings():
    b = _bench()
    assert b._code_lines("int x = 1;\n") != b._code_lines("int x = 2;\n")
    s = 'const char* u = "a//b";  // note\n'
    assert b._code_lines(s) == s.rstrip()


def test_recorded_traffic_entries_name_both_kernel_families():
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for key, ent in rec.items():
        assert ent["dram_bytes_per_launch"] > 0 and len(ent["source_hash"]) == 16, key
