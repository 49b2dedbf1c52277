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


def test_eta_stencil_and_band_step_argument_errors():
    torch = torch_cuda()
    n = 32
    plan = StencilPlan(n, n, n, 4, synth.laplacian8_coeffs())
    e = torch.zeros(n ** 3, device="cuda")
    out = torch.zeros(n ** 3, device="cuda")
    assert code_of(lambda: plan.eta_stencil(0, out.data_ptr(), 0.5, 1 / 12)) == ARG
    assert code_of(lambda: plan.eta_stencil(e.data_ptr(), e.data_ptr(), 0.5, 1 / 12)) == ALIAS
    assert code_of(lambda: plan.eta_stencil(e.data_ptr(), out.data_ptr() + 4, 0.5, 1 / 12)) == ALIGN
    plan.eta_stencil(e, out, 0.5, 1 / 12)
    plan.status()
    f = [torch.zeros(n ** 3, device="cuda") for _ in range(5)]
    up, u, un, s, et = [t.data_ptr() for t in f]
    assert code_of(lambda: plan.wave_step_pml(up, u, un, s, et, -1)) == ARG
    assert code_of(lambda: plan.wave_step_pml(up, u, u, s, et, 4)) == ALIAS
    plan.close()


def test_host_phases_need_a_pipelined_call():
    torch_cuda()
    n = 64
    plan = StencilPlan(n, n, n, 4, synth.laplacian8_coeffs())
    assert code_of(lambda: plan.host_phases()) == ARG
    u = synth.uniform_field(n, n, n)
    out = np.empty_like(u)
    plan.apply_host(u, out, 1)
    ph = plan.host_phases()
    assert ph["slabs"] >= 1 and ph["total_ms"] > 0
    plan.close()


def test_slab_calls_reject_arrays_of_another_device_kind():
    torch = torch_cuda()
    from seismic_wave_propagation_gb300 import StencilSlabs
    slabs = StencilSlabs(64, 32, 40, 4, synth.laplacian8_coeffs(), 2)
    sizes = [(slabs.extent(k)["end"] - slabs.extent(k)["begin"]) * 64 * 32 for k in range(2)]
    dev = [torch.zeros(sz, device="cuda") for sz in sizes]
    host = [np.zeros(sz, np.float32) for sz in sizes]
    assert code_of(lambda: slabs.apply([dev[0].data_ptr(), host[1].ctypes.data], [x.clone() for x in dev])) == ARG
    assert code_of(lambda: slabs.exchange([dev[0].data_ptr(), dev[0].data_ptr()])) == ALIAS
    slabs.close()
