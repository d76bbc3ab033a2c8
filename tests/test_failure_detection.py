"""Failure detection on the GPU without a fault: a bounded in-kernel wait that
runs out is reported, and the CUDA context stays usable.

The main kernel bounds every wait on an mbarrier (tensor copies, MMA
completion, the epilogue's accumulator hand-off) by a time limit; when one
runs out the CTA records DGRAD_ERR_DEVICE_TIMEOUT in the plan's device error
word, lets its copies land, frees its tensor memory and exits.  The plan
option ``wait_test=1`` makes the MMA warp first wait on a barrier that
nothing completes, so that this path runs on purpose: nothing faults, traps
or hangs, and the whole launch ends within a few multiples of the
(here short) wait limit.  The pages' own error handling is the host-side
argument checks of doppler's conv2d_backward.js / bias_add_backward.js,
covered by the CPU tests; this file covers the device half.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import conv2d_backward_implicit_dgrad_gb300 as dg
from conv2d_backward_implicit_dgrad_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TIMEOUT_STATUS = 7   # DGRAD_ERR_DEVICE_TIMEOUT
SHORT_US = 2000      # wait limit of the stalled launches: 2 ms


def assert_tf32(gpu, ref, mag):
    assert np.isfinite(gpu).all()
    assert np.all(np.abs(gpu - ref) <= 2e-3 * mag)


@pytest.mark.parametrize("a_source", ["frame", "producers", "staged", "tmem"])
@pytest.mark.parametrize("name", ["tiny", "resnet_stage", "strided_downsample", "pointwise"])
def test_wait_that_runs_out_is_reported_and_context_survives(name, a_source):
    wl = WORKLOADS[name]
    try:
        dg.describe(*wl.plan_args(), "tf32", a_source=a_source)
    except dg.DgradError as e:
        if e.status == 2:
            pytest.skip("this source does not apply to this shape")
        raise
    go_h, w_h = make_inputs(wl, 5)
    go, w = go_h.cuda(), w_h.cuda()
    with dg.Plan(*wl.plan_args(), precision="tf32", a_source=a_source, timeout_us=SHORT_US, wait_test=1) as plan:
        gi = torch.full(wl.gi_shape, float("nan"), device="cuda")
        t0 = time.perf_counter()
        plan.run(go, w, gi)
        torch.cuda.synchronize()   # the launch ends by itself: every wait is bounded
        elapsed = time.perf_counter() - t0
        with pytest.raises(dg.DgradError) as exc:
            plan.check()
        assert exc.value.status == TIMEOUT_STATUS
        plan.check()   # reading the error word cleared it
    # a handful of sequential 2 ms limits, not a hang (generous for a shared box)
    assert elapsed < 5.0
    # the context is intact: a normal plan on the same inputs is correct
    ref, mag = oracle.dgrad(go_h, w_h, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    with dg.Plan(*wl.plan_args(), precision="tf32", a_source=a_source) as plan:
        out = plan.run(go, w)
        torch.cuda.synchronize()
        plan.check()
    assert_tf32(out.cpu().double().numpy(), ref, mag)


def test_short_wait_limit_alone_raises_nothing():
    # A 50 ms limit is far above any wait of a normal launch: no false timeout.
    wl = WORKLOADS["resnet_stage"]
    go_h, w_h = make_inputs(wl, 6)
    go, w = go_h.cuda(), w_h.cuda()
    ref, mag = oracle.dgrad(go_h, w_h, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    with dg.Plan(*wl.plan_args(), precision="tf32", timeout_us=50000) as plan:
        for _ in range(3):
            out = plan.run(go, w)
        torch.cuda.synchronize()
        plan.check()
    assert_tf32(out.cpu().double().numpy(), ref, mag)


def test_host_pipeline_reports_a_sub_plan_timeout():
    # dgrad_run_host runs the batch through sub-plans and reads their error
    # words behind its last copy: a stalled sub-plan surfaces as the call's status.
    wl = WORKLOADS["tiny"]
    go_h, w_h = make_inputs(wl, 7)
    with dg.Plan(*wl.plan_args(), precision="tf32", timeout_us=SHORT_US, wait_test=1) as plan:
        with pytest.raises(dg.DgradError) as exc:
            plan.run_host(go_h.contiguous(), w_h.contiguous(), torch.empty(wl.gi_shape, pin_memory=True))
        assert exc.value.status == TIMEOUT_STATUS


@pytest.mark.parametrize("name", ["tiny", "pointwise"])
def test_ffma_pipeline_wait_that_runs_out(name):
    # The FFMA path's frame pipeline bounds its waits the same way: with
    # wait_test the compute warps first wait on a barrier nothing completes,
    # the loader's wait for a free stage then runs out too, and the launch
    # ends by itself with the timeout recorded.
    wl = WORKLOADS[name]
    go_h, w_h = make_inputs(wl, 8)
    go, w = go_h.cuda(), w_h.cuda()
    with dg.Plan(*wl.plan_args(), precision="fp32", a_source="frame", timeout_us=SHORT_US, wait_test=1) as plan:
        gi = torch.full(wl.gi_shape, float("nan"), device="cuda")
        t0 = time.perf_counter()
        plan.run(go, w, gi)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        with pytest.raises(dg.DgradError) as exc:
            plan.check()
        assert exc.value.status == TIMEOUT_STATUS
        plan.check()
    assert elapsed < 5.0
    ref, _ = oracle.dgrad(go_h, w_h, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    with dg.Plan(*wl.plan_args(), precision="fp32", a_source="frame") as plan:
        out = plan.run(go, w)
        torch.cuda.synchronize()
        plan.check()
    got = out.cpu().double().numpy()
    assert np.linalg.norm((got - ref).ravel()) <= 1e-5 * np.linalg.norm(ref.ravel())


@pytest.mark.parametrize("name,precision,mode", [
    ("resnet_stage", "tf32", 3),          # plane mode
    ("resnet_stage", "tf32x3", 1),        # run mode
    ("strided_downsample", "tf32", 0),    # segment mode
    ("pointwise", "tf32", 2),             # direct mode
])
def test_wgrad_wait_that_runs_out(name, precision, mode):
    # Each weight-gradient main kernel bounds its waits the same way: with
    # wait_test its MMA warp first waits on a barrier nothing completes, the
    # copy and epilogue waits then run out in turn, the launch (and the
    # reduction after it) ends by itself with the timeout recorded, and a
    # normal plan on the same context is correct afterwards.
    wl = WORKLOADS[name]
    go_h, _ = make_inputs(wl, 9)
    x_h = torch.randn((wl.N, wl.Ci, wl.H, wl.W), generator=torch.Generator().manual_seed(10))
    go, x = go_h.cuda(), x_h.cuda()
    with dg.WgradPlan(*wl.plan_args(), precision=precision, timeout_us=SHORT_US, wait_test=1) as plan:
        assert plan.info["mode"] == mode
        t0 = time.perf_counter()
        plan.run(go, x)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        with pytest.raises(dg.DgradError) as exc:
            plan.check()
        assert exc.value.status == TIMEOUT_STATUS
        plan.check()
    assert elapsed < 5.0
    ref, mag = oracle.wgrad(go_h, x_h, wl.kH, wl.kW, wl.stride, wl.pad_h, wl.pad_w)
    with dg.WgradPlan(*wl.plan_args(), precision=precision) as plan:
        dw = plan.run(go, x)
        torch.cuda.synchronize()
        plan.check()
    bound = 1e-5 if precision == "tf32x3" else 2e-3
    assert np.all(np.abs(dw.cpu().double().numpy() - ref) <= bound * mag)
