"""Host-side build helpers (no GPU)."""

from attention_dv_predict_gb300 import build


def test_source_hash_ignores_comments_and_layout():
    a = "int f() { return 1; } // one\n/* a block\n   comment */\n"
    b = "int f()  {\n    return 1;\n}\n"
    assert build._code_only(a) == build._code_only(b)
    assert build._code_only("int f() { return 2; }") != build._code_only(b)


def test_source_hash_is_stable():
    assert build.source_hash() == build.source_hash()
    assert len(build.source_hash()) == 16
