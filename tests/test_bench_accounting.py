"""The measurement arithmetic of bench.py, on CPU: the algorithmic bytes and
flops each call is credited with, and the roofline figures derived from a
CUDA-event time."""

import types

import pytest

import bench

MB = 1 << 20


def test_layer_call_bytes_and_flops_at_the_benchmark_shape():
    """T=4096 H=2048 E=128 K=8 I=768, bf16, every expert with rows: N = 32768
    routed rows.  Tensor sizes: X [N,H] 128 MiB, tokens [T,H] 16 MiB, act [N,I]
    48 MiB, (g,u) and dgu [N,2I] 96 MiB, W_gate + W_up 768 MiB, W_down 384 MiB,
    int32 index arrays 128 KiB each; probs and their grads fp32 [T,K] 128 KiB."""
    by, fl = bench._gemm_bytes(T=4096, H=2048, E_active=128, E=128, K=8, I=768)
    X, tok, act, gu, wgu, wd, idx = 128 * MB, 16 * MB, 48 * MB, 96 * MB, 768 * MB, 384 * MB, MB // 8
    assert by["permute"] == tok + X + 4 * idx             # tokens read, K copies written, indices
    assert by["gate_up_swiglu"] == X + wgu + act + gu     # X and both weights read; act, (g,u) written
    assert by["down_proj"] == act + wd + X                # act and W_down read; expanded written
    assert by["unpermute"] == X + tok + idx + idx         # expanded, row_map, probs read; out written
    assert by["unpermute_grad"] == tok + 2 * X + idx + 2 * idx
    assert by["down_dgrad_swiglu"] == X + wd + 2 * gu     # dY, W_down, (g,u) read; dgu written
    assert by["gate_up_dgrad"] == gu + wgu + X            # dgu and both weights read; dX written
    assert by["down_wgrad"] == X + act + wd               # dY, act read; dW_down written
    assert by["gate_up_wgrad"] == gu + X + wgu            # dgu, X read; dW_gate, dW_up written
    assert by["permute_grad"] == X + tok + idx
    N, H, I = 32768, 2048, 768
    for name in ("gate_up_swiglu", "gate_up_dgrad", "gate_up_wgrad"):
        assert fl[name] == 2 * N * H * (2 * I)               # two [N,H] x [H,I] products
    for name in ("down_proj", "down_dgrad_swiglu", "down_wgrad"):
        assert fl[name] == 2 * N * H * I


def test_fused_permute_moves_only_the_token_operand():
    plain, _ = bench._gemm_bytes(T=4096, H=2048, E_active=128, E=128, K=8, I=768)
    fused, _ = bench._gemm_bytes(T=4096, H=2048, E_active=128, E=128, K=8, I=768, fused=True)
    X, tok = 128 * MB, 16 * MB
    assert plain["permute"] - fused["permute"] == tok + X   # no row copy
    assert plain["gate_up_swiglu"] - fused["gate_up_swiglu"] == X - tok
    assert plain["gate_up_wgrad"] - fused["gate_up_wgrad"] == X - tok
    assert plain["down_proj"] == fused["down_proj"]


def test_weights_of_experts_without_rows_are_not_read_but_their_grads_are_written():
    full, _ = bench._gemm_bytes(T=64, H=128, E_active=8, E=8, K=2, I=64)
    part, _ = bench._gemm_bytes(T=64, H=128, E_active=3, E=8, K=2, I=64)
    w_gu, w_d = 2 * 64 * 128 * 2, 128 * 64 * 2            # per expert
    assert full["gate_up_swiglu"] - part["gate_up_swiglu"] == 5 * w_gu
    assert full["down_proj"] - part["down_proj"] == 5 * w_d
    assert full["gate_up_wgrad"] == part["gate_up_wgrad"]
    assert full["down_wgrad"] == part["down_wgrad"]


def test_roofline_figures_from_an_event_time():
    """A call moving 1 GB and 100 GFLOP in 200 us: 5000 GB/s and 500 TFLOP/s;
    against 6783.8 GB/s and 1707.9 TFLOP/s the bytes take longer, so the call
    is HBM-bound and its roofline fraction is the bandwidth fraction."""
    work = types.SimpleNamespace(bytes={"k": 1e9, "m": 1e9}, flops={"k": 1e11})
    per = {"k": {"launches": 10, "avg_ms": 0.2, "total_ms": 2.0},
           "m": {"launches": 10, "avg_ms": 0.2, "total_ms": 2.0}}
    peaks = {"hbm_gbs": 6783.8, "bf16_tflops_sustained": 1707.9}
    t = bench.kernel_table(per, work, peaks)
    assert t["k"]["gbs"] == pytest.approx(5000.0)
    assert t["k"]["tflops"] == pytest.approx(500.0)
    assert t["k"]["bound"] == "hbm"
    assert t["k"]["roofline_frac"] == pytest.approx(5000.0 / 6783.8)
    assert t["k"]["share"] == pytest.approx(0.5)
    assert t["m"]["bound"] == "hbm" and t["m"]["roofline_frac"] == pytest.approx(5000.0 / 6783.8)
    # 1 GB for 1000 TFLOP is tensor-bound
    work.flops["k"] = 1e15
    t = bench.kernel_table(per, work, peaks)
    assert t["k"]["bound"] == "tensor"
    assert t["k"]["roofline_frac"] == pytest.approx((1e15 / 1707.9e12) / 2e-4)
