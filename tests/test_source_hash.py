"""The kernel-source hash that ties the committed DRAM-traffic figure to the kernels it
was measured on: comments do not enter it, code does."""
import bench


def test_comments_do_not_change_the_code():
    a = 'int f(int x) {  // doubles\n  /* a block\n     comment */\n  return 2 * x;\n}\n'
    b = 'int f(int x) {\n  return 2 * x;  // still doubles\n}\n'
    assert bench._code_only(a) == bench._code_only(b)


def test_code_and_literals_are_kept():
    a = 'const char* s = "a // not a comment";\nint y = 1;\n'
    assert '"a // not a comment"' in bench._code_only(a)
    assert bench._code_only(a) != bench._code_only(a.replace("int y = 1", "int y = 2"))
    c = "char q = '\\'';  // quote\nint z;\n"
    assert bench._code_only(c) == "char q = '\\'';\nint z;"

