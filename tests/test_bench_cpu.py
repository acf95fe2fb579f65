"""Host-side logic of bench.py that decides what it reports: the GEMM code hash
that gates the profiled DRAM traffic (comments do not count, code does) and
the parsing of the committed ncu summary."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_strip_comments_keeps_code_only():
    b = load_bench()
    src = "int a = 1; // one\n/* block\n comment */\nint b = 2;\n\n   // only a comment\nint c;  \n"
    assert b.strip_comments(src) == "int a = 1;\nint b = 2;\nint c;"
    assert b.strip_comments(src.replace("// one", "// uno")) == b.strip_comments(src)
    assert b.strip_comments(src.replace("int b = 2;", "int b = 3;")) != b.strip_comments(src)


def test_profiled_traffic_follows_the_code_hash():
    b = load_bench()
    text = open(os.path.join(ROOT, "profiles", "gemm_mxf4_llama8b_down_train_step.md")).read()
    for mode, low in (("separate", 1e8), ("grouped", 3e8)):
        t = b.profiled_traffic(mode)
        if b.gemm_source_hash() in text and f"dram bytes per {'grouped launch' if mode == 'grouped' else 'launch'}" in text:
            # DRAM bytes per gemm_fp4 launch, ~2e8 at the 8B shapes; per grouped launch ~6e8
            assert t is not None and t > low
        else:
            assert t is None
