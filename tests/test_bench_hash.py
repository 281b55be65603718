"""The source hash that keeps a committed ncu profile valid (bench.py): it
follows the code of a kernel's sources, not their comments or layout."""
import bench


def test_code_only_strips_comments_and_layout():
    src = 'int a;  // note\n/* block\n comment */ int   b;\nconst char *s = "x // y /* z */";\n'
    assert bench.code_only(src) == 'int a; int b; const char *s = "x // y /* z */";'


def test_hash_ignores_comments_but_not_code():
    base = {"fa_tc.cuh": "template <int D> void f() { g(D); }  // one\n"}
    texts = dict(base)

    def read(name):
        return texts.get(name, "")

    h0 = bench.kernel_source_hash("fa_tc_fwd_kernel<bf16>", read)
    texts["fa_tc.cuh"] = "// a new header comment\ntemplate <int D>\nvoid f() {\n  g(D);\n}\n"
    assert bench.kernel_source_hash("fa_tc_fwd_kernel<bf16>", read) == h0
    texts["fa_tc.cuh"] = "template <int D> void f() { g(D + 1); }\n"
    assert bench.kernel_source_hash("fa_tc_fwd_kernel<bf16>", read) != h0


def test_hash_covers_the_shared_sources():
    texts = {}

    def read(name):
        return texts.get(name, "")

    h0 = bench.kernel_source_hash("fa_bwd_kernel<bf16>", read)
    texts["fa_api.cu"] = "int launch() { return 1; }"
    assert bench.kernel_source_hash("fa_bwd_kernel<bf16>", read) != h0
