"""The gradient gate of the GPU parity tests, checked on the CPU against oracle gradients.

At the training-step workload's input scale (N(0,1)/8) the largest |dq| and |dk| of a slice
are a few 1e-3, under the bf16 path's absolute bound of 2e-2: that bound alone would accept
an all-zero gradient. These tests pin the gate (the absolute bound and a bound relative to
the tensor's own magnitude) to what it must reject and accept, on the oracle's gradients of
real slices of that workload (the analytic gradient of softmax attention over S_i).
"""
import numpy as np
import pytest
import torch

import fibattn_inputs as fi
import oracle
from gpu_common import TOL, f64, grad_gate, oracle_bwd_slices


@pytest.fixture(scope="module")
def c5_grads():
    spec = fi.WORKLOADS["c5"]
    inp = fi.workload_inputs("c5", layers=[0])
    # layer 0 and layer 15 of the coprime schedule (different tables), first and last slices
    ref = oracle_bwd_slices(inp, spec["sched"], spec["W"], 0, [(0, 0, 0), (0, 7, 7)])
    ref15 = oracle_bwd_slices(inp, spec["sched"], spec["W"], 15, [(0, 3, 5)])
    return list(ref.values()) + list(ref15.values())


def test_absolute_bound_alone_cannot_fail_at_this_scale(c5_grads):
    for rq, rk, rv, ro, rl in c5_grads:
        assert np.abs(rq).max() < TOL["bf16"] and np.abs(rk).max() < TOL["bf16"]


def test_gate_rejects_zero_gradients(c5_grads):
    for grads in c5_grads:
        for ref in grads[:3]:
            ok, err, rel = grad_gate(np.zeros_like(ref), ref, "bf16")
            assert not ok and rel == pytest.approx(1.0)


def test_gate_rejects_a_scaled_or_sign_flipped_gradient(c5_grads):
    # a dropped factor (5 % too small) and a wrong sign on one tensor
    for grads in c5_grads:
        for ref in grads[:3]:
            assert not grad_gate(0.95 * ref, ref, "bf16")[0]
            assert not grad_gate(-ref, ref, "bf16")[0]


def test_gate_rejects_a_transposed_key_gradient(c5_grads):
    # dk written at the wrong key rows (shifted by one row)
    for rq, rk, rv, ro, rl in c5_grads:
        assert not grad_gate(np.roll(rk, 1, axis=0), rk, "bf16")[0]


def test_gate_accepts_the_bf16_rounding_of_the_reference(c5_grads):
    # the outputs are bf16: rounding the exact gradient once is the least error possible,
    # and a further error of the same size (inputs of the products rounded) must pass too
    for grads in c5_grads:
        for ref in grads[:3]:
            once = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
            assert grad_gate(once, ref, "bf16")[0]
            noisy = once * (1 + 2.0 ** -8 * np.sign(np.sin(np.arange(ref.size))).reshape(ref.shape))
            assert grad_gate(noisy, ref, "bf16")[0]


def test_gate_fp32_bounds():
    ref = np.linspace(-0.3, 0.4, 640).reshape(10, 64)
    assert grad_gate(ref + 5e-6, ref, "f32")[0]
    assert not grad_gate(ref + 2e-5, ref, "f32")[0]          # over the 1e-5 bound
    small = ref * 1e-3
    assert not grad_gate(small + 5e-6, small, "f32")[0]      # 1e-5 bound met, relative not
    # a gradient that vanishes identically (one query) is met to rounding
    assert grad_gate(np.full((1, 64), 1e-9), np.zeros((1, 64)), "f32")[0]
