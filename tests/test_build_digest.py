"""The build digest that ties a committed ncu summary to the kernel it measured: it
follows the code (a changed instruction gives a new digest) and ignores comments,
blank lines and trailing blanks (editing a comment keeps the summary valid)."""
from block_sparse_kv_bsr_gb300 import _build


def test_code_of_ignores_comments_and_blank_space():
    a = b"int x = 1;  // one\n\n/* block\n comment */\nint y = 2;\n"
    b = b"int x = 1;\n// a comment line\nint y = 2;   \n\n"
    assert _build._code_of(a) == _build._code_of(b) == b"int x = 1;\nint y = 2;"


def test_code_changes_change_the_digest(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_bytes(b"__global__ void k() { }  // c\n")
    monkeypatch.setattr(_build, "CSRC", str(tmp_path))
    d0 = _build.kernel_digest(("k.cu",))
    src.write_bytes(b"// a new comment\n__global__ void k() { }\n")
    assert _build.kernel_digest(("k.cu",)) == d0
    src.write_bytes(b"__global__ void k() { int z = 0; }\n")
    assert _build.kernel_digest(("k.cu",)) != d0


def test_sources_hold_no_comment_markers_inside_strings():
    # inline PTX strings must not contain "//" or "/*", which the digest would cut
    import os
    import re
    for name in os.listdir(_build.CSRC):
        if not name.endswith((".cu", ".cuh", ".h", ".cpp")):
            continue
        text = open(os.path.join(_build.CSRC, name), encoding="utf-8").read()
        for lit in re.findall(r'"(?:[^"\\\n]|\\.)*"', text):
            assert "//" not in lit and "/*" not in lit, (name, lit)
