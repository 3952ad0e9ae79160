"""The FMA-pipe exp2 the prefill softmax uses for one exponential pair in four.

Method: 2^x = 2^j * 2^f, j = round(x), f in [-1/2, 1/2], with a degree-4
minimax polynomial for 2^f fitted by csrc/fit_exp2.py.  Stated bound: relative
error <= 2.7e-6 against exact 2^x for x in [-125, 127] (about 23 ulp at 1.0;
the bf16 rounding P receives afterwards is 2^-9 = 2e-3).
"""
import ctypes
import importlib.util
import os

import numpy as np
import pytest
import torch

BOUND = 2.7e-6
CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "gqa_softmax_attention_gb300",
                    "csrc")
COEF = [9.999992847e-01, 6.931217909e-01, 2.402474433e-01, 5.591785908e-02, 9.570102207e-03]


def _fma32(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def emulate(x):
    """The kernel's steps in float32 (one rounding per fused multiply-add)."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126))
    sh = np.float32(12582912.0)
    t = (x + sh).astype(np.float32)
    j = (t - sh).astype(np.float32)
    f = _fma32(j, np.float32(-1), x)
    c = [np.float32(v) for v in COEF]
    p = _fma32(np.full_like(f, c[4]), f, np.full_like(f, c[3]))
    p = _fma32(p, f, np.full_like(f, c[2]))
    p = _fma32(p, f, np.full_like(f, c[1]))
    p = _fma32(p, f, np.full_like(f, c[0]))
    bits = (p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))).astype(np.uint32)
    return bits.view(np.float32)


def test_coefficients_match_the_fit_script():
    spec = importlib.util.spec_from_file_location("fit_exp2", os.path.join(CSRC, "fit_exp2.py"))
    fit = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit)
    c32 = np.array([float(c) for c in fit.remez(4)], dtype=np.float32)
    assert np.allclose(c32, np.array(COEF, dtype=np.float32), rtol=2e-7, atol=0)


def test_algorithm_error_bound_on_cpu():
    x = np.concatenate([np.linspace(-125, 127, 2_000_001), np.arange(-125, 128, 0.5)]).astype(np.float32)
    y = emulate(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() <= BOUND
    # arguments far below the range give a tiny non-negative value, never garbage
    z = emulate(np.array([-126.0, -200.0, -1e30], dtype=np.float32))
    assert np.all(z >= 0) and np.all(z < 2.0 ** -124)


@pytest.mark.gpu
def test_kernel_exp2_matches_exp2f():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gqa_softmax_attention_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    x = torch.cat([torch.linspace(-125, 127, 1_000_001), torch.arange(-125, 127, 0.25),
                   torch.rand(100_000, generator=torch.Generator().manual_seed(0)) * -30]).cuda()
    y = torch.empty_like(x)
    st = lib.gqa_exp2_poly(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.numel(),
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    ref = torch.exp2(x)                     # CUDA exp2f
    rel = ((y.double() - ref.double()).abs() / ref.double()).max().item()
    assert rel <= BOUND + 2.0 ** -23        # exp2f itself is within ~1 ulp
    # bit-exact agreement with the float32 emulation of the same steps
    assert np.array_equal(y.cpu().numpy().view(np.uint32), emulate(x.cpu().numpy()).view(np.uint32))
