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
