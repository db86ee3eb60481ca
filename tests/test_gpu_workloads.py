"""The five layer shapes at full size, in the launch configuration the
benchmark times (default options, AUTO path): outputs of the tokens the
oracle can afford (all of them for small T, a sample that includes the most
loaded expert's tokens and the last token otherwise) against the FP64 oracle,
plus run-to-run bit identity.  Weights are drawn on the GPU; the oracle reads
back the exact BF16 bytes of the experts its tokens select."""
import gc

import numpy as np
import pytest
import torch

from mixture_experts_ffn_gate_gb300 import moe_ffn as m
from mixture_experts_ffn_gate_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = [
    ("decode_h2048_i768_e128_k8", 1, None),
    ("decode_h2048_i768_e128_k8", 2, None),
    ("decode_h4096_i1536_e128_k8_bias", 1, None),
    ("decode_h4096_i1536_e128_k8_bias", 4, None),
    ("decode_h4096_i1536_e128_k8_bias", 16, None),
    ("decode_h4096_i1536_e128_k8_bias", 64, 24),
    ("decode_h7168_i2048_e384_k8_bias", 1, None),
    ("decode_h7168_i2048_e384_k8_bias", 8, None),
    ("decode_h7168_i2048_e384_k8_bias", 32, 8),
    ("fwd_t2048_h6144_i2048_e256_k8_bias", 2048, 12),
]

_weights = {}


def weights(name):
    if name not in _weights:
        _weights.clear()
        gc.collect()
        torch.cuda.empty_cache()
        _weights[name] = synth.make_weights(synth.WORKLOADS[name], device="cuda")
    return _weights[name]


def sample_tokens(idx, T, n):
    """n tokens: the first, the last, and tokens of the most loaded expert,
    topped up with a seeded random choice."""
    if n is None or n >= T:
        return np.arange(T)
    counts = np.bincount(idx.ravel(), minlength=idx.max() + 1)
    heavy = np.nonzero((idx == counts.argmax()).any(axis=1))[0]
    pick = {0, T - 1, *heavy[: n // 3].tolist()}
    rng = np.random.default_rng(T)
    while len(pick) < n:
        pick.add(int(rng.integers(T)))
    return np.array(sorted(pick))


@pytest.mark.parametrize("name,T,n_sample", CASES, ids=lambda v: str(v))
def test_workload_against_oracle(name, T, n_sample):
    wl = synth.WORKLOADS[name]
    wgu, wd = weights(name)
    x, L = synth.make_tokens(wl, T, call=7, device="cuda")
    out, idx, w = gu.run_gpu(x, L, wgu, wd, wl.k, m.MOE_PATH_AUTO)
    toks = sample_tokens(idx.numpy(), T, n_sample)
    r_out, r_idx, r_w = gu.oracle_ref(x, L, wgu, wd, wl.k, tokens=toks)
    gu.assert_accepted(out[toks], idx[toks], w[toks], r_out, r_idx, r_w, what=f"{name} T={T}")
    assert m.moe_ffn_device_faults(clear=True) == 0


@pytest.mark.parametrize("name,T,runs", [("decode_h2048_i768_e128_k8", 1, 100),
                                          ("decode_h2048_i768_e128_k8", 2, 100),
                                          ("decode_h4096_i1536_e128_k8_bias", 4, 100),
                                          ("decode_h7168_i2048_e384_k8_bias", 32, 100),
                                          ("fwd_t2048_h6144_i2048_e256_k8_bias", 2048, 100)],
                         ids=lambda v: str(v))
def test_workload_bit_identical_runs(name, T, runs):
    wl = synth.WORKLOADS[name]
    wgu, wd = weights(name)
    x, L = synth.make_tokens(wl, T, call=11, device="cuda")
    ws = m.new_workspace(T, wl.H, wl.I, wl.E, wl.k)
    first = m.moe_ffn_forward_ex(x, L, wgu, wd, wl.k, workspace=ws).clone()
    same = torch.ones((), dtype=torch.bool, device="cuda")
    for _ in range(runs - 1):
        o = m.moe_ffn_forward_ex(x, L, wgu, wd, wl.k, workspace=ws)
        same &= (o.view(torch.int32) == first.view(torch.int32)).all()
    torch.cuda.synchronize()
    assert bool(same)
    assert m.moe_ffn_device_faults(clear=True) == 0
