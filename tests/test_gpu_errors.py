"""Argument validation and error codes of the C ABI (host-side checks, GPU present)."""
import numpy as np
import pytest

from seismic_wave_propagation_gb300 import StencilError, StencilPlan, synth
from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu

ARG, ALIGN, ALIAS = -1, -2, -3


def code_of(fn):
    with pytest.raises(StencilError) as ei:
        fn()
    return ei.value.code


def test_apply_argument_errors():
    torch = torch_cuda()
    n = 32
    plan = StencilPlan(n, n, n, 4, synth.laplacian8_coeffs())
    a = torch.zeros(n ** 3 + 64, device="cuda")
    b = torch.zeros(n ** 3 + 64, device="cuda")
    assert code_of(lambda: plan.apply(0, b.data_ptr())) == ARG
    assert code_of(lambda: plan.apply(a.data_ptr() + 4, b.data_ptr())) == ALIGN
    assert code_of(lambda: plan.apply(a.data_ptr(), a.data_ptr())) == ALIAS
    assert code_of(lambda: plan.apply(a.data_ptr(), a.data_ptr() + 256)) == ALIAS
    host = np.zeros(n ** 3, np.float32)
    assert code_of(lambda: plan.apply(host.ctypes.data, b.data_ptr())) == ARG
    plan.apply(a.data_ptr(), b.data_ptr())
    plan.status()
    plan.close()


def test_wave_aliasing_rules():
    torch = torch_cuda()
    n = 32
    plan = StencilPlan(n, n, n, 4, synth.laplacian8_coeffs())
    f = [torch.zeros(n ** 3, device="cuda") for _ in range(5)]
    up, u, un, s, e = [t.data_ptr() for t in f]
    plan.wave_step(up, u, up, s, e)  # u_next == u_prev exactly: allowed
    plan.status()
    assert code_of(lambda: plan.wave_step(up, u, u, s, e)) == ALIAS
    assert code_of(lambda: plan.wave_step(up, u, s, s, e)) == ALIAS
    assert code_of(lambda: plan.wave_step(up, u, e, s, e)) == ALIAS
    assert code_of(lambda: plan.wave_step(up, u, up + 16, s, e)) == ALIAS
    assert code_of(lambda: plan.wave_step(up, u, un + 8, s, e)) == ALIGN
    plan.close()


def test_plan_creation_errors():
    torch_cuda()
    c = synth.laplacian8_coeffs()
    with pytest.raises(StencilError):
        StencilPlan(30, 32, 32, 4, c)  # nx not a multiple of 4
    with pytest.raises(StencilError):
        StencilPlan(32, 32, 32, 5, list(c) + [0.0])
    with pytest.raises(StencilError):
        StencilPlan(0, 32, 32, 4, c)
