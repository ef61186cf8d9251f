"""The kernel-source hash that keys the stored ncu traffic figures: comments and layout do not change it, code does."""
import bench


def test_comments_and_layout_do_not_count():
    a = 'int a = 1; // one\n/* a block\n comment */ const char* s = "x // kept";\n'
    b = 'int a = 1;\n\n  // another comment\nconst char* s = "x // kept";'
    assert bench._code_only(a) == bench._code_only(b)


def test_code_and_string_literals_count():
    assert bench._code_only("int a = 1;") != bench._code_only("int a = 2;")
    assert bench._code_only('f("x // y");') != bench._code_only('f("x");')
