"""The bench's byte models (host logic, no GPU): the per-kernel figures that
the roofline fractions divide by must account for the whole call's bytes
the way the kernels split the work."""
import dataclasses

import pytest

import bench
from mixture_experts_ffn_gate_gb300 import synth

pytestmark = pytest.mark.cpu

WL = synth.WORKLOADS["fwd_t2048_h6144_i2048_e256_k8_bias"]


@pytest.mark.parametrize("U", [1, 61, 195, 256])
def test_weight_gradients_written_once_across_kernels(U):
    # zeros for the untouched experts plus the two weight-gradient GEMMs'
    # outputs make every expert's FP32 gradient exactly once
    H, I, E, k, T = WL.H, WL.I, WL.E, WL.k, 2048
    n = T * k
    zeros = bench.backward_kernel_bytes("zero_grads", WL, T, U, k)
    dwd = bench.backward_kernel_bytes("wgrad_down", WL, T, U, k) - (2 * n * H * 2 + 2 * n * I * 2)
    dwgu = bench.backward_kernel_bytes("wgrad_gate_up", WL, T, U, k) - (2 * n * 2 * I * 2 + n * H * 2)
    assert zeros + dwd + dwgu == E * 3 * H * I * 4


def test_training_step_bytes_drop_only_the_recomputation():
    T, U = 2048, 195
    fwd = bench.algorithmic_bytes(WL, T, U)
    bwd = bench.backward_bytes(WL, T, U)
    step = bench.train_bytes(WL, T, U)
    recompute_read = U * 2 * WL.I * WL.H * 2
    kept_gu = 2 * T * WL.k * WL.I * 4
    assert step == fwd + bwd - recompute_read + kept_gu
    assert fwd + bwd - step > 0.8 * recompute_read   # the pair saves most of a W_gate_up read


def test_training_step_kernel_names_map_to_their_calls():
    T, U, k = 2048, 195, WL.k
    assert bench.train_kernel_bytes("bwd:wgrad_gate_up", WL, T, U, k) == \
        bench.backward_kernel_bytes("wgrad_gate_up", WL, T, U, k)
    assert bench.train_kernel_bytes("fwd:gemm_down", WL, T, U, k) == bench.kernel_bytes("gemm_down", WL, T, U, k)
    # the training forward's gate_up also writes g and u
    assert bench.train_kernel_bytes("fwd:gemm_gate_up", WL, T, U, k) == \
        bench.kernel_bytes("gemm_gate_up", WL, T, U, k) + 2 * T * k * WL.I * 4
    assert bench.train_kernel_bytes("fwd:router", WL, T, U, k) is None


def test_decode_kernel_bytes_cover_the_call():
    # the fused decode kernel moves the call's bytes plus its act rows out and back
    wl = synth.WORKLOADS["decode_h2048_i768_e128_k8"]
    for T, U in ((1, 8), (2, 15), (4, 30)):
        call = bench.algorithmic_bytes(wl, T, U)
        assert bench.kernel_bytes("decode_fused", wl, T, U, wl.k) == call + 2 * T * wl.k * wl.I * 4
    # MXFP8 weights: 1 + 1/32 bytes per weight
    mx = bench.algorithmic_bytes(wl, 1, 8, bench.BPE["mxfp8"]) - (1 * wl.H * 2 + wl.E * 4 + wl.H * 4)
    assert mx == pytest.approx(8 * 3 * wl.H * wl.I * (1 + 1 / 32))


def test_smaller_expert_variant_scales_the_weight_bytes():
    small = dataclasses.replace(WL, E=16)
    assert bench.backward_kernel_bytes("zero_grads", small, 128, 16, WL.k) == 0
    assert bench.kernel_bytes("gemm_gate_up", small, 256, 16, WL.k) < bench.kernel_bytes("gemm_gate_up", WL, 256, 30, WL.k)
