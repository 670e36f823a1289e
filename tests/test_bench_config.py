"""bench.py's timing hygiene on CPU: which workloads are timed with an L2
flush before every step (a step that moves less than twice the 129 MB L2)
and what the JSON line's config says about it."""
import bench
from fsdp_sharded_mixed_shard_gb300 import workloads as W


def test_small_workloads_are_timed_cold():
    assert bench.needs_flush(W.TINY_FLAT, "fused")          # 34 MB per step
    cfg = bench.config_of(W.TINY_FLAT, "fused")
    assert cfg["l2"].startswith("L2 flushed before every timed step")
    assert "256 MB" in cfg["l2"]
    assert bench.FLUSH_BYTES > bench.L2_BYTES


def test_large_workloads_exceed_l2():
    for wl, path in ((W.GPT2_SMALL, "fused"), (W.STAGE3_SLICE, "fused"),
                     (W.LLAMA_2B, "two_pass"), (W.FLAT_1P5B, "two_pass")):
        assert not bench.needs_flush(wl, path), wl.name
        assert bench.config_of(wl, path)["l2"].startswith("inputs larger than L2")
    # GPT-2 list at N = 8: (2N + 26) bytes per parameter
    assert bench.step_bytes(W.GPT2_SMALL, "fused") == 42 * 124_439_808


def test_flat_shape_option():
    import sys
    old = sys.argv
    try:
        sys.argv = ["bench.py", "--flat", "40000064", "--ranks", "64", "--clip", "1.0"]
        a = bench.parse_args()
    finally:
        sys.argv = old
    wl = bench.selected_workload(a)
    assert wl.numels == [40_000_064] and wl.n_ranks == 64 and wl.max_grad_norm == 1.0
    assert wl.name == "flat_40000064_n64_bf16_clip"
    assert bench.config_of(wl, "two_pass")["shard_elems"] == 625_001


def test_traffic_figures_survive_comment_edits_only():
    a = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    b = "/* f: successor */\nint f(int x) {\n    return x + 1;\n}\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_sha(a) == bench.code_sha(b)
    assert bench.code_sha(a) != bench.code_sha(c)


def test_both_arms_report_the_same_config():
    """The libzero arm and the reference (checker) arm build their `config`
    through one function, so the driver can match the two lines."""
    import inspect
    cfg = bench.run_config(W.FLAT_1P5B, "two_pass", 1)
    assert cfg == dict(bench.config_of(W.FLAT_1P5B, "two_pass"),
                       parallelism="8 simulated ranks per GPU x 1 GPUs")
    assert "run_config(" in inspect.getsource(bench.run_reference)
    assert "run_config(" in inspect.getsource(bench.run_libzero)
