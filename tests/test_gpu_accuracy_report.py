"""The warp-decode article's accuracy claim as a measured report (its section
핵심 내용: the output lands 1.4x closer to a full FP32 reference than the
expert-centric kernels it replaces).  Those kernels round the intermediate
activation to BF16 (the article's section 경쟁 구도 / 비교 names dropping that
quantisation); here they are stood in for by the plain emulation of that
one step -- FP32 dot products, act = silu(g) * u rounded to BF16, FP32 down
projection and combine -- on the same bytes.  Both outputs are measured
against the FP64 oracle; the test prints the two normwise errors and their
ratio and requires the library's output to be at least 1.4x closer."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bf16_round(a: np.ndarray) -> np.ndarray:
    """float32 -> nearest BF16 (ties to even), returned as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _prior_style(x, L, wgu, wd, k):
    """FP32 layer whose intermediate activation is rounded to BF16."""
    idx, w = gu.oracle_ref(x, L, wgu, wd, k)[1:]
    xf = x.float().cpu().numpy()
    T, H = xf.shape
    I = wd.shape[2]
    out = np.zeros((T, H), np.float32)
    for e in np.unique(idx):
        ge = wgu[int(e)].float().cpu().numpy()
        de = wd[int(e)].float().cpu().numpy()
        rows, slots = np.nonzero(idx == e)
        g = xf[rows] @ ge[:I].T
        u = xf[rows] @ ge[I:].T
        act = _bf16_round((g / (1.0 + np.exp(-g))) * u)
        y = act @ de.T
        out[rows] += w[rows, slots].astype(np.float32)[:, None] * y
    return out


@pytest.mark.parametrize("name,T", [("decode_h2048_i768_e128_k8", 4), ("decode_h4096_i1536_e128_k8_bias", 16)])
def test_output_closer_to_the_exact_layer_than_a_bf16_intermediate(name, T):
    wl = synth.WORKLOADS[name]
    wgu, wd = synth.make_weights(wl, device="cuda")
    bias = synth.make_bias(wl)
    x, L = synth.make_tokens(wl, T, call=11, device="cuda", bias=bias)
    ours = m.moe_ffn_forward_ex(x, L, wgu, wd, wl.k).cpu().double().numpy()
    ref = gu.oracle_ref(x, L, wgu, wd, wl.k)[0]
    prior = _prior_style(x, L, wgu, wd, wl.k).astype(np.float64)
    err_ours = np.linalg.norm(ours - ref) / np.linalg.norm(ref)
    err_prior = np.linalg.norm(prior - ref) / np.linalg.norm(ref)
    print(f"\n{name} T={T}: normwise error vs FP64 -- library {err_ours:.3e}, "
          f"BF16-intermediate emulation {err_prior:.3e}, ratio {err_prior / err_ours:.1f}")
    assert err_prior / err_ours >= 1.4
