"""Host-side pieces of bench.py that need no GPU: the source hash that decides
whether a stored ncu traffic figure still describes the kernel."""
import os

import bench


def _hash_of(tmp_path, text, name="k.cu"):
    p = tmp_path / name
    p.write_text(text, encoding="utf-8")
    return bench.code_hash(str(p))


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    base = _hash_of(tmp_path, "int f(int x) {\n  return x + 1;  // one more\n}\n")
    assert _hash_of(tmp_path, "// header\nint f(int x) { /* body */ return x + 1; }\n") == base
    assert _hash_of(tmp_path, "int  f(int x)\n{\n\treturn x+1;\n}\n") == base


def test_code_hash_sees_code_and_string_literals(tmp_path):
    base = _hash_of(tmp_path, 'asm("add.u32 %0, %1, 1; // x" : "=r"(y) : "r"(x));\n')
    # a change inside a string literal (even after "//" in it) is a code change
    assert _hash_of(tmp_path, 'asm("add.u32 %0, %1, 2; // x" : "=r"(y) : "r"(x));\n') != base
    assert _hash_of(tmp_path, 'asm("add.u32 %0, %1, 1; // y" : "=r"(y) : "r"(x));\n') != base
    assert _hash_of(tmp_path, 'asm("add.u32 %0, %1, 1; // x" : "=r"(z) : "r"(x));\n') != base
    # an escaped quote does not end the literal
    assert _hash_of(tmp_path, 'const char* s = "a\\"//b";\n') != _hash_of(tmp_path, 'const char* s = "a\\"//c";\n')


def test_traffic_record_only_for_its_workload_and_hash(tmp_path, monkeypatch):
    root = tmp_path
    (root / "profiles").mkdir()
    csrc = root / "sparse_retrieval_host_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int f() { return 1; } // v1\n", encoding="utf-8")
    h = bench.code_hash(str(csrc / "k.cu"))
    (root / "profiles" / "traffic.json").write_text(
        '{"attend": {"source": "k.cu", "source_code_hash": "%s", "dram_bytes_per_launch": 7, "workload": "w"}}' % h)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.traffic_record("attend", "w")["dram_bytes_per_launch"] == 7
    assert bench.traffic_record("attend", "other") is None
    (csrc / "k.cu").write_text("int f() { return 1; } // v2, comments only\n", encoding="utf-8")
    assert bench.traffic_record("attend", "w") is not None
    (csrc / "k.cu").write_text("int f() { return 2; }\n", encoding="utf-8")
    assert bench.traffic_record("attend", "w") is None
    assert os.path.exists(root / "profiles" / "traffic.json")
