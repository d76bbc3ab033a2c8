"""GPU parity of the weight gradient (wgrad) against the CPU oracle (O-w).

Bar: the TF32 bar of the dgrad path, per element
|gpu - ref| <= 2e-3 * sum|terms|, and exactly 0 where no term reaches the
element.  Split precision (tf32x3) takes the FP32 bar, relative L2 error
<= 1e-5, and per element |gpu - ref| <= 1e-5 * sum|terms|: each product is
off by at most about 3 * 2^-22 of its size (the dropped lo*lo term and the
rounding of lo), and the fp32 accumulation adds a few 2^-24 per addition of
similar size, far below 1e-5 for the K lengths here.  grad_weight is
poisoned with NaN before every run, so an element the kernels fail to write
fails the bar, and it sits between two guard bands of canary values that must
come back unchanged (no store past either end).

TF32 runs are also held to the products they compute: the oracle on the
inputs reduced to TF32 the way the mode reduces them (the frame modes round
to nearest, ties away from zero, when they pack; the direct and plane modes
let the tensor core take the TF32 part of the caller's values, i.e.
truncate) gives the exact sum of those products, and the GPU must match it
within fp32 accumulation error, 2e-6 * sum|terms|.  A term dropped or taken
from the wrong position moves an element by about 1 / (N*oH*oW) of its
sum|terms|, far below the TF32 bar but above this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import conv2d_backward_implicit_dgrad_gb300 as dg
from conv2d_backward_implicit_dgrad_gb300.workloads import ORDER, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TF32_REL_TERMS = 2e-3
TF32_PRODUCTS_REL_TERMS = 2e-6
SPLIT_REL_TERMS = 1e-5
SPLIT_REL_L2 = 1e-5


def tf32_truncate(t):
    """The TF32 part of fp32 values: the 13 low mantissa bits cleared."""
    b = t.contiguous().view(torch.int32) & -8192
    return b.view(torch.float32)


def tf32_round(t):
    """fp32 rounded to TF32, to nearest with ties away from zero: half of the
    dropped bits' unit added to the magnitude, then those bits cleared."""
    b = (t.contiguous().view(torch.int32) + 4096) & -8192
    return b.view(torch.float32)


def out_ext(n, k, s, p):
    return (n + 2 * p - k) // s + 1


def inputs(N, Ci, Co, H, W, kH, kW, s, ph, pw, seed):
    g = torch.Generator().manual_seed(seed)
    go = torch.randn((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), generator=g)
    x = torch.randn((N, Ci, H, W), generator=g)
    return go, x


GUARD = 4096          # floats of canary on each side of grad_weight (16 KiB: keeps 16-byte alignment)
CANARY = -1234.5625


def run_gpu(args, go, x, precision="tf32"):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    n = Co * Ci * kH * kW
    with dg.WgradPlan(*args, precision=precision) as plan:
        buf = torch.full((n + 2 * GUARD,), CANARY, device="cuda")
        buf[GUARD:GUARD + n] = float("nan")
        dw = buf[GUARD:GUARD + n].view((Co, Ci, kH, kW))
        plan.run(go.cuda(), x.cuda(), dw)
        torch.cuda.synchronize()
        plan.check()
        info = plan.info
    head, tail = buf[:GUARD].cpu(), buf[-GUARD:].cpu()
    assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), "a store landed outside grad_weight"
    return dw.cpu().double().numpy(), info


def check(args, go, x, precision="tf32"):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    ref, mag = oracle.wgrad(go, x, kH, kW, s, ph, pw)
    gpu, info = run_gpu(args, go, x, precision)
    assert info["precision"] == precision
    assert np.isfinite(gpu).all(), "non-finite output (unwritten element?)"
    err = np.abs(gpu - ref)
    bound = SPLIT_REL_TERMS if precision == "tf32x3" else TF32_REL_TERMS
    bad = err > bound * mag
    pos = mag > 0
    worst = np.max(err[pos] / mag[pos]) if pos.any() else 0.0
    assert not bad.any(), f"{bad.sum()} elements over the bound; worst err/sum|terms| = {worst:.3e}"
    assert np.all(gpu[~pos] == 0)
    rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel < (SPLIT_REL_L2 if precision == "tf32x3" else 1e-3), rel
    if precision == "tf32":
        reduce = tf32_truncate if info["mode"] in (2, 3) else tf32_round
        pref, pmag = oracle.wgrad(reduce(go), reduce(x), kH, kW, s, ph, pw)
        perr = np.abs(gpu - pref)
        assert np.all(perr <= TF32_PRODUCTS_REL_TERMS * pmag), \
            f"mode {info['mode']}: worst |gpu - sum of TF32 products| / sum|terms| = {np.max(perr[pmag > 0] / pmag[pmag > 0]):.3e}"
    return info


EDGE = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw
    (1, 1, 1, 5, 7, 3, 3, 1, 0, 0),
    (3, 3, 4, 9, 11, 5, 5, 1, 1, 1),
    (1, 5, 33, 10, 9, 3, 3, 2, 0, 0),
    (3, 65, 4, 7, 13, 3, 3, 3, 1, 1),
    (1, 129, 33, 6, 10, 1, 1, 2, 0, 0),
    (1, 3, 4, 23, 21, 7, 7, 2, 3, 3),
    (3, 5, 33, 12, 14, 2, 2, 2, 0, 0),
    (1, 3, 1, 11, 17, 3, 5, 1, 2, 1),
    (1, 65, 33, 17, 19, 4, 3, 2, 1, 2),
    (1, 3, 4, 2, 2, 3, 3, 2, 1, 1),        # a kernel row that only meets padding
    (1, 4, 3, 1, 1, 1, 1, 2, 1, 1),        # no term reaches any weight element
    (3, 16, 20, 31, 29, 3, 3, 1, 1, 1),
    (1, 20, 40, 40, 40, 3, 3, 4, 1, 1),    # stride 4
    (2, 8, 300, 9, 7, 3, 3, 1, 1, 1),      # two column tiles
    (2, 200, 16, 6, 6, 3, 3, 1, 1, 1),     # input channels over one segment
    (5, 3, 4, 9, 11, 3, 3, 1, 1, 1),       # four images interleaved along K, a ragged last group
    (4, 6, 8, 12, 10, 3, 3, 2, 1, 1),
    (7, 2, 3, 10, 13, 7, 7, 2, 3, 3),
    (6, 4, 5, 11, 9, 5, 3, 3, 2, 1),
    (9, 16, 24, 15, 17, 3, 3, 1, 1, 1),
    (32, 3, 4, 7, 9, 3, 3, 1, 1, 1),       # batch-blocked frames (32 images per K chunk)
    (35, 5, 3, 8, 6, 3, 3, 2, 1, 1),       # 35 images: four interleaved (blocking would pad 29)
    (60, 5, 3, 8, 6, 3, 3, 2, 1, 1),       # blocked, four padding images
    (33, 2, 2, 5, 7, 5, 3, 3, 2, 1),
    (64, 70, 20, 6, 5, 3, 3, 1, 1, 1),     # blocked, two image groups (segment mode: run tiles do not fit)
    (64, 40, 20, 6, 5, 3, 3, 1, 1, 1),     # run mode, two image groups
    (32, 16, 40, 9, 11, 5, 3, 1, 2, 1),    # run mode, 5 x 3 taps
    (32, 3, 8, 40, 44, 3, 3, 1, 1, 1),     # run mode, 16 position blocks per tile
    (32, 130, 24, 9, 8, 3, 3, 1, 1, 1),    # two input-channel blocks
    (3, 40, 24, 6, 10, 1, 1, 1, 0, 0),     # 1x1: direct mode (the caller's tensors, no frames)
    (2, 8, 300, 4, 9, 1, 1, 1, 0, 0),      # direct mode, two column tiles
    (5, 130, 20, 12, 12, 1, 1, 1, 0, 0),   # direct mode, two input-channel segments
    (2, 8, 16, 5, 5, 1, 1, 1, 0, 0),       # 1x1 with 25 positions per plane: frames
]

PLANE = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw: TF32 plane mode (stride 1, oH = H, oW = W, W a multiple of 4)
    (2, 5, 7, 6, 8, 3, 3, 1, 1, 1),        # channel rows padded to 8, B columns padded to 32
    (3, 40, 24, 6, 12, 3, 3, 1, 1, 1),     # one row tile of 120 rows
    (2, 64, 64, 8, 8, 3, 3, 1, 1, 1),      # two row tiles
    (2, 3, 4, 5, 4, 5, 5, 1, 2, 2),        # 5 x 5 taps, a ragged chunk per image
    (1, 16, 16, 7, 12, 3, 5, 1, 1, 2),     # 3 x 5 taps
    (2, 130, 40, 6, 8, 3, 3, 1, 1, 1),     # four row tiles x 128 columns: all of tensor memory
    (1, 8, 8, 3, 4, 3, 3, 1, 1, 1),        # one chunk in all: a grid of one CTA
    (200, 8, 8, 8, 8, 3, 3, 1, 1, 1),      # 400 chunks on 152 CTAs, ranges crossing images
    (2, 256, 8, 8, 8, 3, 3, 1, 1, 1),      # six row tiles of a 32-column B
    (32, 3, 8, 40, 44, 3, 3, 1, 1, 1),
    (32, 130, 24, 9, 8, 3, 3, 1, 1, 1),
]


@pytest.mark.parametrize("shape", EDGE)
def test_wgrad_edge_shapes(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, x = inputs(*shape, seed=90)
    check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, x)


@pytest.mark.parametrize("shape", PLANE)
def test_wgrad_plane_shapes(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, x = inputs(*shape, seed=95)
    info = check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, x)
    assert info["mode"] == 3


def test_wgrad_plane_maps_follow_the_tensors():
    """Plane mode encodes its tensor maps on the caller's tensors and keeps
    them while the pointers stay the same: runs on other tensors, then on the
    first ones again, are each correct."""
    args = (3, 16, 8, 12, 24, 3, 3, 1, 1, 1)
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    pairs = [inputs(N, Ci, Co, H, W, kH, kW, s, ph, pw, seed=96 + i) for i in range(2)]
    refs = [oracle.wgrad(go, x, kH, kW, s, ph, pw) for go, x in pairs]
    dev = [(go.cuda(), x.cuda()) for go, x in pairs]
    with dg.WgradPlan(*args, precision="tf32") as plan:
        assert plan.info["mode"] == 3
        for i in (0, 1, 0, 1):
            dw = torch.full((Co, Ci, kH, kW), float("nan"), device="cuda")
            plan.run(dev[i][0], dev[i][1], dw)
            torch.cuda.synchronize()
            plan.check()
            ref, mag = refs[i]
            assert np.all(np.abs(dw.cpu().double().numpy() - ref) <= TF32_REL_TERMS * mag)


@pytest.mark.parametrize("name", ORDER)
def test_wgrad_workloads(name):
    """Every workload at full size against the whole oracle result."""
    wl = WORKLOADS[name]
    go, _ = make_inputs(wl, 0)
    x = torch.randn((wl.N, wl.Ci, wl.H, wl.W), generator=torch.Generator().manual_seed(91))
    info = check(wl.plan_args(), go, x)
    assert info["grid"] <= 152


@pytest.mark.parametrize("shape", EDGE)
def test_wgrad_split_edge_shapes(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, x = inputs(*shape, seed=93)
    check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, x, "tf32x3")


@pytest.mark.parametrize("name", ORDER)
def test_wgrad_split_workloads(name):
    wl = WORKLOADS[name]
    go, _ = make_inputs(wl, 0)
    x = torch.randn((wl.N, wl.Ci, wl.H, wl.W), generator=torch.Generator().manual_seed(94))
    check(wl.plan_args(), go, x, "tf32x3")


def test_wgrad_overwrites_and_leaves_inputs_alone():
    args = (2, 16, 12, 12, 24, 3, 3, 1, 1, 1)
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    go, x = inputs(N, Ci, Co, H, W, kH, kW, s, ph, pw, seed=92)
    g, xx = go.cuda(), x.cuda()
    g0, x0 = g.clone(), xx.clone()
    with dg.WgradPlan(*args) as plan:
        a = plan.run(g, xx, torch.full((Co, Ci, kH, kW), 7.0, device="cuda"))
        b = plan.run(g, xx, torch.full((Co, Ci, kH, kW), -3.0, device="cuda"))
        torch.cuda.synchronize()
        plan.check()
    assert torch.equal(a, b)            # deterministic, and nothing of the old contents survives
    assert torch.equal(g, g0) and torch.equal(xx, x0)


def test_wgrad_rejects_bad_arguments():
    args = (1, 8, 8, 8, 8, 3, 3, 1, 1, 1)
    with dg.WgradPlan(*args) as plan:
        lib = dg.load_library()
        go = torch.zeros((1, 8, 8, 8), device="cuda")
        x = torch.zeros((1, 8, 8, 8), device="cuda")
        buf = torch.zeros(8 * 8 * 9 + 16, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
        assert lib.wgrad_run(plan._h, P(go), P(x), P(buf, 4), stream) == 3      # misaligned
        assert lib.wgrad_run(plan._h, P(go), P(x), None, stream) == 3           # NULL
        assert lib.wgrad_run(plan._h, P(go), P(x), P(x), stream) == 4           # grad_weight over the input
        torch.cuda.synchronize()
        plan.check()
    with pytest.raises(dg.DgradError) as e:
        dg.WgradPlan(*args, precision="fp32")
    assert e.value.status == 2


def test_wgrad_plane_replayed_in_a_cuda_graph():
    """A CUDA graph of a plane-mode wgrad_run (the plane kernel and the
    reduction, chained by a dependent launch; tensor maps encoded before the
    capture), replayed on new inputs copied into the same tensors, is correct
    on every replay."""
    args = (3, 16, 12, 24, 8, 3, 3, 1, 1, 1)
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    with dg.WgradPlan(*args, precision="tf32") as plan:
        assert plan.info["mode"] == 3
        go_d = torch.zeros((N, Co, H, W), device="cuda")
        x_d = torch.zeros((N, Ci, H, W), device="cuda")
        dw = torch.zeros((Co, Ci, kH, kW), device="cuda")
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            plan.run(go_d, x_d, dw)   # maps encoded before capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            plan.run(go_d, x_d, dw)
        for seed in range(3):
            go, x = inputs(N, Ci, Co, H, W, kH, kW, s, ph, pw, seed=97 + seed)
            go_d.copy_(go)
            x_d.copy_(x)
            dw.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            plan.check()
            ref, mag = oracle.wgrad(go, x, kH, kW, s, ph, pw)
            assert np.all(np.abs(dw.cpu().double().numpy() - ref) <= TF32_REL_TERMS * mag)
