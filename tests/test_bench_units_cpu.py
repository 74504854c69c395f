"""The roofline units the benchmark reports, checked against the shapes they
come from: per-launch algorithmic bytes of each kernel kind (weights once,
activations, every cached K/V byte once) and their sum over a step."""
import pytest

import bench
from synth import WORKLOADS, make_state_np

MB = 1e6


def test_weight_bytes_of_the_qwen3_8b_shaped_layer():
    wl = WORKLOADS["full_stack"]
    s = wl.shape
    B, W = wl.batch, wl.window
    M = B * W
    b = bench.algorithmic_bytes(s, B, W, prefix_total=0)
    # the weight term of each projection, from the layer's shape alone
    weights = {"gemm_qkv": (32 + 2 * 8) * 128 * 4096 * 2, "gemm_o": 4096 * 4096 * 2,
               "gemm_gateup": 2 * 12288 * 4096 * 2, "gemm_down": 12288 * 4096 * 2,
               "lmhead": 151936 * 4096 * 2}
    for kind, wbytes in weights.items():
        act = b[kind] - wbytes
        # what is left is activations: a few MB at 128 rows, never weights
        assert 0 < act < 8 * MB, (kind, act)
    assert weights["gemm_qkv"] == pytest.approx(50.3 * MB, rel=1e-3)
    assert weights["lmhead"] == pytest.approx(1245.2 * MB, rel=1e-3)
    # attention without a prefix moves only the window (q, o, window K/V)
    assert b["attn"] == 2 * (M * 2 * 8 * 128 + 2 * M * 32 * 128)


def test_attention_bytes_grow_by_4_kib_per_cached_token():
    wl = WORKLOADS["full_stack"]
    s = wl.shape
    a0 = bench.algorithmic_bytes(s, 8, 16, 0)["attn"]
    a1 = bench.algorithmic_bytes(s, 8, 16, 1000)["attn"]
    assert a1 - a0 == 1000 * 4096  # K + V, 8 kv heads x 128 dims, bf16


def test_step_bytes_of_the_benchmark_workload():
    """36 layers of weights + the LM head + every cached K/V byte once: the
    ~20 GB per step the whole-step roofline divides by the copy bandwidth."""
    wl = WORKLOADS["full_stack"]
    s = wl.shape
    st = make_state_np(wl)
    prefix_total = int(st["seq_len"].sum())
    b = bench.algorithmic_bytes(s, wl.batch, wl.window, prefix_total)
    per_layer = sum(b[k] for k in ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down", "attn"))
    step = s.n_layers * per_layer + b["lmhead"]
    weights = s.n_layers * 2 * (48 * 128 * 4096 + 4096 * 4096 + 3 * 12288 * 4096) \
        + 2 * 151936 * 4096
    kv = s.n_layers * prefix_total * 4096
    assert step >= weights + kv
    # activations (inputs, outputs, residual reads) are ~18 MB a layer
    assert step - (weights + kv) == pytest.approx(s.n_layers * 17.7e6, rel=0.05)
    assert 19e9 < step < 21.5e9


def test_flops_per_kind_from_the_shape_and_by_brute_force():
    """Projections: two FLOPs per weight per row; LM head: over the masked
    rows only; attention: 4*hd per q head and visible (query, key) pair,
    counted here pair by pair for a small ragged case."""
    wl = WORKLOADS["full_stack"]
    s = wl.shape
    B, W = 3, 5
    lens = [7, 0, 19]
    f = bench.algorithmic_flops(s, B, W, sum(lens), masked_rows=4)
    M = B * W
    params = {"gemm_qkv": 4096 * 48 * 128, "gemm_o": 32 * 128 * 4096,
              "gemm_gateup": 4096 * 2 * 12288, "gemm_down": 12288 * 4096}
    for kind, p in params.items():
        assert f[kind] == 2 * M * p, kind
    assert f["lmhead"] == 2 * 4 * 151936 * 4096
    pairs = sum(L + p + 1 for L in lens for p in range(W))
    assert f["attn"] == 4 * 32 * 128 * pairs


def test_kernel_bound_is_the_larger_of_hbm_and_tensor_time():
    # one kind at 1 GB and 1 GFLOP (HBM-bound), one at 1 MB and 1 TFLOP
    byts = {"a": 10 ** 9, "b": 10 ** 6}
    flops = {"a": 10 ** 9, "b": 10 ** 12}
    tim = {"a": (2.0, 2), "b": (4.0, 2)}  # ms total, launches
    k = bench.kernel_rates(tim, byts, 1000.0, 1, flops, 1000.0)
    assert k["a"]["bound"] == "hbm" and k["b"]["bound"] == "tensor"
    assert k["a"]["gbs"] == pytest.approx(1000.0)   # 1 GB in 1 ms
    assert k["b"]["tflops"] == pytest.approx(500.0)  # 1 TFLOP in 2 ms
    assert k["b"]["frac_tensor"] == pytest.approx(0.5)
