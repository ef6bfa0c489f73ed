"""The build digest that keys recorded ncu traffic figures to kernel code
(bench.py): comments do not count, code does."""
import bench


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // line comment\n'
           'const char *s = "x // not a comment /* nor this */";\n'
           '/* block\n   comment */ int b = \'/\';   \n'
           'int c = 2 / 3;\n')
    assert bench.strip_comments(src) == (
        'int a = 1;\n'
        'const char *s = "x // not a comment /* nor this */";\n'
        " int b = '/';\n"
        'int c = 2 / 3;')


def test_digest_ignores_comments_but_not_code():
    files = {name: "" for name in bench.KERNEL_SOURCES["quant"]}
    files["quant.cu"] = "__global__ void k() { int x = 1; }\n"
    base = bench.source_digest("quant", files.__getitem__)
    commented = dict(files, **{"quant.cu": "// header\n__global__ void k() { int x = 1;/* why */ }  // end\n"})
    assert bench.source_digest("quant", commented.__getitem__) == base
    changed = dict(files, **{"quant.cu": "__global__ void k() { int x = 2; }\n"})
    assert bench.source_digest("quant", changed.__getitem__) != base


def test_digest_of_the_tree_is_stable():
    assert bench.source_digest("matmul") == bench.source_digest("matmul")
    assert len(bench.source_digest("quant")) == 16
