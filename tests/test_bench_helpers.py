"""CPU checks of bench.py's bookkeeping: committed ncu counters are matched to
the kernel sources by a hash that ignores comments but not code."""
import bench


def _sha_of(tmp_path, text):
    p = tmp_path / "k.cu"
    p.write_text(text)
    old = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        return bench.file_sha(["k.cu"])
    finally:
        bench.ROOT = old


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    base = "int f(int x) {\n    return x + 1;\n}\n"
    commented = ("// header comment\n/* block\n   comment */\nint f(int x) {  // trailing\n\n"
                 "    return x + 1;   \n}\n")
    assert _sha_of(tmp_path, base) == _sha_of(tmp_path, commented)


def test_code_hash_changes_with_code(tmp_path):
    assert _sha_of(tmp_path, "int f() { return 1; }\n") != _sha_of(tmp_path, "int f() { return 2; }\n")

