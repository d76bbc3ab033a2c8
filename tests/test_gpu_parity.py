"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars (fixed by the tolerance the method is held to):
  * FP32 path: relative L2 error ||gpu - ref||_2 / ||ref||_2 <= 1e-5 (fp64).
  * TF32 path: per element |gpu - ref| <= 2e-3 * sum|terms|, and exactly 0
    wherever no term reaches the element (sum|terms| = 0).
  * TF32X3 (split precision) path: the FP32 bar, and per element
    |gpu - ref| <= (2^-20 + (3K + 2) 2^-23) * sum|terms| (K = Co*kH*kW): each
    split product is within 2^-20 of its size of the exact one, and the 3K
    fp32 additions add at most 2^-23 of the running sum each (truncating
    accumulation allowed for).
TF32 runs of the tensor-core path are also held to the products they
compute: the weights are rounded to TF32 (to nearest, ties away from zero)
when packed, and grad_out likewise by the frame, staged and tensor-memory
sources, while the producer warps either round it the same way (16-byte
loads) or let the tensor core truncate it (4-byte asynchronous copies).  The
oracle on the inputs so reduced gives the exact sum of those products, and
the GPU must match it within 1e-5 * sum|terms| (fp32 accumulation over at
most a few hundred MMAs); a dropped or misplaced term moves an element by
about 1/K of its sum|terms| (K = Co*kH*kW), which the TF32 bar alone would
miss for long K.
grad_input is poisoned with NaN before every run, so an element the kernels
fail to write fails both bars, and it sits between two guard bands of canary
values that must come back unchanged, so a store past either end of it fails
too.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import conv2d_backward_implicit_dgrad_gb300 as dg
from conv2d_backward_implicit_dgrad_gb300.workloads import ORDER, WORKLOADS, make_inputs, make_tensors

pytestmark = pytest.mark.gpu

FP32_REL_L2 = 1e-5
TF32_PRODUCTS_REL_TERMS = 1e-5


def tf32_round(t):
    """fp32 rounded to TF32, to nearest with ties away from zero: half of the
    dropped bits' unit added to the magnitude, then those bits cleared."""
    b = (t.contiguous().view(torch.int32) + 4096) & -8192
    return b.view(torch.float32)


def tf32_truncate(t):
    """The TF32 part of fp32 values: the 13 low mantissa bits cleared."""
    return (t.contiguous().view(torch.int32) & -8192).view(torch.float32)


def assert_tf32_products(gpu, go, w, args, info):
    """The tensor-core TF32 result against the exact sum of the products it
    computes (see the module docstring)."""
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    wr = tf32_round(w)
    reductions = (tf32_round, tf32_truncate) if info["a_source"] == "producers" else (tf32_round,)
    worst = []
    for red in reductions:
        pref, pmag = oracle.dgrad(red(go), wr, H, W, s, ph, pw)
        err = np.abs(gpu - pref)
        if np.all(err <= TF32_PRODUCTS_REL_TERMS * pmag):
            return
        pos = pmag > 0
        worst.append(float(np.max(err[pos] / pmag[pos])))
    raise AssertionError(f"{info['a_source']}: worst |gpu - sum of TF32 products| / sum|terms| = {worst}")
TF32_REL_TERMS = 2e-3


def out_ext(n, k, s, p):
    return (n + 2 * p - k) // s + 1


GUARD = 4096          # floats of canary on each side of an output tensor (16 KiB: keeps 16-byte alignment)
CANARY = -1234.5625   # exactly representable, and no dgrad of these inputs produces it by chance


def guarded(shape, fill=float("nan")):
    """An output tensor in the middle of a larger buffer whose two ends hold
    canary values; returns (buffer, tensor view)."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), CANARY, device="cuda")
    buf[GUARD:GUARD + n] = fill
    return buf, buf[GUARD:GUARD + n].view(shape)


def assert_guards(buf):
    """Both guard bands still hold the canary: nothing was stored past either end."""
    head, tail = buf[:GUARD].cpu(), buf[-GUARD:].cpu()
    assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), "a store landed outside grad_input"


def run_gpu(args, go, w, precision, **opts):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    with dg.Plan(*args, precision=precision, **opts) as plan:
        buf, gi = guarded((N, Ci, H, W))
        plan.run(go.cuda(), w.cuda(), gi)
        torch.cuda.synchronize()
        plan.check()
        info = plan.info
    assert_guards(buf)
    return gi.cpu().double().numpy(), info


def assert_fp32(gpu, ref):
    assert np.isfinite(gpu).all(), "non-finite output (unwritten element?)"
    num = np.linalg.norm((gpu - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    rel = num / den if den > 0 else num
    assert rel <= FP32_REL_L2, f"relative L2 error {rel:.3e} > {FP32_REL_L2}"


def assert_tf32(gpu, ref, mag):
    assert np.isfinite(gpu).all(), "non-finite output (unwritten element?)"
    err = np.abs(gpu - ref)
    bad = err > TF32_REL_TERMS * mag
    pos = mag > 0
    worst = np.max(err[pos] / mag[pos]) if pos.any() else 0.0
    assert not bad.any(), f"{bad.sum()} elements over the bound; worst err/sum|terms| = {worst:.3e}"
    assert np.all(gpu[~pos] == 0)


def split_bound(Co, kH, kW):
    return 2.0 ** -20 + (3 * Co * kH * kW + 2) * 2.0 ** -23


def assert_split(gpu, ref, mag, Co, kH, kW):
    assert_fp32(gpu, ref)
    err = np.abs(gpu - ref)
    bad = err > split_bound(Co, kH, kW) * mag
    assert not bad.any(), f"{bad.sum()} elements over the split-precision bound"
    assert np.all(gpu[mag == 0] == 0)


def check(args, go, w, precision, **opts):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    ref, mag = oracle.dgrad(go, w, H, W, s, ph, pw)
    gpu, info = run_gpu(args, go, w, precision, **opts)
    if precision == "fp32":
        assert_fp32(gpu, ref)
    elif precision == "tf32x3":
        assert_split(gpu, ref, mag, Co, kH, kW)
    else:
        assert_tf32(gpu, ref, mag)
        if info["path"] == "tcgen05":
            assert_tf32_products(gpu, go, w, args, info)
    return info


# ----------------------------------------------------------------- workloads
@pytest.mark.parametrize("precision", ["tf32", "fp32", "tf32x3"])
@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", ORDER)
def test_workload_parity(name, seed, precision):
    wl = WORKLOADS[name]
    go, w = make_inputs(wl, seed)
    info = check(wl.plan_args(), go, w, precision)
    assert info["path"] == ("simt" if precision == "fp32" else "tcgen05")


@pytest.mark.parametrize("a_source", ["frame", "staged", "producers", "tmem"])
@pytest.mark.parametrize("name", ["tiny", "resnet_stage", "strided_downsample", "pointwise"])
def test_workload_parity_each_source(name, a_source):
    """The TF32 path with every way grad_out can reach the MMA, on the
    workloads: the packed frame, tensor copies of grad_out transposed in
    shared memory (staged), producer warps, and (1x1 only) tensor copies
    moved into tensor memory as the MMA's A operand."""
    wl = WORKLOADS[name]
    try:
        dg.describe(*wl.plan_args(), "tf32", a_source=a_source)
    except dg.DgradError as e:
        if e.status == 2:
            pytest.skip("this source does not apply to this shape")
        raise
    go, w = make_inputs(wl, 5)
    info = check(wl.plan_args(), go, w, "tf32", a_source=a_source)
    assert info["a_source"] == a_source


@pytest.mark.parametrize("precision", ["tf32", "tf32x3"])
@pytest.mark.parametrize("shape", [WORKLOADS["pointwise"].plan_args(),   # (N, Ci, H, W, Co, kH, kW, s, ph, pw)
                                   (3, 33, 12, 12, 70, 1, 1, 1, 0, 0), (2, 300, 16, 16, 40, 1, 1, 1, 0, 0),
                                   (1, 17, 8, 16, 9, 1, 1, 1, 0, 0)])
def test_tmem_equals_frame_bitwise(shape, precision):
    """A in tensor memory holds the same TF32 operands (rounded to nearest,
    ties away) as the frame path's shared-memory A, and the K order is the
    same: the results agree bit for bit.  Shapes: the workload, tiles running
    across images, two input-channel slices (several units per tile), one
    image (no next image to copy from)."""
    N, Ci, H, W, Co, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, H, W), (Co, Ci, 1, 1), 88, "kaiming")
    a, ia = run_gpu(shape, go, w, precision, a_source="tmem")
    b, ib = run_gpu(shape, go, w, precision, a_source="frame")
    assert ia["a_source"] == "tmem" and ib["a_source"] == "frame"
    assert np.array_equal(a, b)
    ref, mag = oracle.dgrad(go, w, H, W, s, ph, pw)
    if precision == "tf32":
        assert_tf32(a, ref, mag)
    else:
        assert_split(a, ref, mag, Co, kH, kW)


@pytest.mark.parametrize("precision", ["tf32", "tf32x3"])
@pytest.mark.parametrize("name", ["tiny", "resnet_stage", "strided_downsample", "pointwise"])
def test_staged_equals_frame_bitwise(name, precision):
    """Both sources feed the MMAs the same TF32 operands (round to nearest,
    ties away) in the same K order, and every output's sum is formed in the
    same order whatever tile it falls in: the results agree bit for bit."""
    wl = WORKLOADS[name]
    go, w = make_inputs(wl, 7)
    a, ia = run_gpu(wl.plan_args(), go, w, precision, a_source="staged")
    b, ib = run_gpu(wl.plan_args(), go, w, precision, a_source="frame")
    assert ia["a_source"] == "staged" and ib["a_source"] == "frame"
    assert ia["group_taps"] == ib["group_taps"]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("name", ["tiny", "resnet_stage", "strided_downsample", "pointwise"])
def test_split_precision_staged(name):
    """Split precision with the staged source (hi and lo parts formed in
    shared memory from one copy per K pass)."""
    wl = WORKLOADS[name]
    go, w = make_inputs(wl, 6)
    info = check(wl.plan_args(), go, w, "tf32x3", a_source="staged")
    assert info["a_source"] == "staged"


# ----------------------------------------------------------------- edge sweep
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
    (3, 1, 4, 15, 8, 5, 3, 1, 1, 2),
    (1, 65, 33, 17, 19, 4, 3, 2, 1, 2),
    (1, 3, 4, 2, 2, 3, 3, 2, 1, 1),        # a kernel row that only meets padding
    (1, 4, 3, 1, 1, 1, 1, 2, 1, 1),        # no term reaches any input element
    (3, 16, 20, 31, 29, 3, 3, 1, 1, 1),    # ragged tiles, several tiles per image
    (1, 20, 40, 40, 40, 3, 3, 4, 1, 1),    # stride 4: 16 phases
]


@pytest.mark.parametrize("precision", ["tf32", "fp32", "tf32x3"])
@pytest.mark.parametrize("shape", EDGE)
def test_edge_shapes(shape, precision):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 71, "uniform")
    check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, precision)


# Tilings of the tcgen05 kernel: pipeline depth, chunk size, slices, persistent
# CTAs that walk several work units (grid smaller than the unit count).
TILINGS = [
    dict(tile_blocks=1), dict(tile_blocks=2), dict(tile_blocks=1, chunk_k=32, grid=3),
    dict(tile_blocks=2, grid=3), dict(tile_blocks=1, slice_n=16, grid=5), dict(tile_blocks=1, slice_n=32, grid=7),
    dict(tile_blocks=3, grid=2), dict(tile_blocks=4, grid=1), dict(tile_blocks=4, slice_n=16, grid=2),
    dict(group_taps="on", grid=3), dict(group_taps="on", slice_n=16, grid=5), dict(group_taps="on", grid=1),
    dict(group_taps="off", grid=3), dict(group_taps="on", slice_n=32),
    dict(group_taps="phases", grid=3), dict(group_taps="phases", tile_blocks=2, grid=2),
    dict(group_taps="phases", slice_n=16, grid=5),
]


@pytest.mark.parametrize("a_source", ["frame", "producers", "staged", "tmem"])
@pytest.mark.parametrize("opts", TILINGS)
@pytest.mark.parametrize("shape", [(2, 40, 36, 19, 23, 3, 3, 1, 1, 1), (2, 48, 20, 17, 18, 3, 3, 2, 1, 1),
                                   (3, 33, 70, 9, 14, 1, 1, 1, 0, 0), (2, 24, 40, 16, 16, 3, 3, 1, 1, 1),
                                   (2, 40, 36, 20, 24, 3, 3, 1, 1, 1), (2, 48, 20, 16, 16, 3, 3, 2, 1, 1),
                                   (3, 33, 70, 8, 14, 1, 1, 1, 0, 0), (3, 33, 70, 12, 12, 1, 1, 1, 0, 0)])
def test_tc_tilings(shape, opts, a_source):
    opts = dict(opts, a_source=a_source)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    try:
        dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, "tf32", path="tcgen05", **opts)
    except dg.DgradError as e:
        if e.status == 2:
            pytest.skip("this tiling does not fit (tensor memory, one staged copy per band, or not 1x1)")
        raise
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 73, "kaiming")
    info = check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "tf32", path="tcgen05", **opts)
    for k in ("tile_blocks", "slice_n", "chunk_k", "a_source"):
        if k in opts:
            assert info[k] == opts[k]
    if "group_taps" in opts:
        assert info["group_taps"] == {"on": 1, "off": 0, "phases": 2}[opts["group_taps"]]


@pytest.mark.parametrize("opts", [dict(slice_n=16), dict(slice_n=32, chunk_k=8), dict(chunk_k=32)])
def test_simt_tilings(opts):
    shape = (2, 40, 36, 19, 23, 3, 3, 2, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 79, "kaiming")
    check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "fp32", path="simt", **opts)


# FFMA path: grad_out reaches the FFMA loop either as tensor copies of the
# packed frame (the pipelined kernel) or through the CTA's own gather.  Both
# agree with the oracle, and, summing the same products in the same order,
# with each other bit for bit.  Shapes in plan order (N, Ci, H, W, Co, kH, kW,
# s, ph, pw): the workloads, ragged channel counts, several phases, a band of
# more than 256 rows (two tensor copies per channel group), a kernel wider
# than the stride, and phases without taps.
FFMA_SHAPES = [WORKLOADS[n].plan_args() for n in ("tiny", "strided_downsample", "pointwise")] + [
    (2, 64, 20, 20, 64, 3, 3, 1, 1, 1), (3, 33, 12, 12, 70, 3, 3, 1, 1, 1), (2, 40, 36, 19, 23, 3, 3, 2, 1, 1),
    (1, 3, 80, 80, 8, 7, 7, 2, 3, 3), (3, 5, 17, 19, 33, 1, 1, 2, 0, 0), (2, 17, 9, 11, 5, 5, 3, 3, 2, 1),
    (1, 20, 40, 40, 40, 3, 3, 4, 1, 1),
    # phases of different tap counts over several rounds of persistent CTAs with
    # a partial last one (the sorted schedule): 276 units on 152 CTAs, and with
    # 8 x 8 tiles 352 units on 304 CTAs
    (8, 40, 64, 64, 24, 3, 3, 2, 1, 1), (16, 64, 48, 48, 16, 5, 5, 2, 2, 2)]


@pytest.mark.parametrize("args", FFMA_SHAPES)
def test_ffma_sources_agree(args):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 91, "kaiming")
    ref, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    outs = {}
    for src in ("frame", "producers"):
        gpu, info = run_gpu(args, go, w, "fp32", a_source=src)
        assert info["path"] == "simt" and info["a_source"] == src
        assert_fp32(gpu, ref)
        outs[src] = gpu
    assert np.array_equal(outs["frame"], outs["producers"])


# Inputs of at most 4 channels large enough for the gather kernel's
# 4-channel slices (1024-position units): against the oracle, and bit for bit
# against the frame pipeline's 16-channel slices (the same products summed in
# the same order).  Plan order (N, Ci, H, W, Co, kH, kW, s, ph, pw).
NARROW_SHAPES = [(4, 3, 200, 200, 8, 3, 3, 1, 1, 1), (3, 1, 300, 260, 5, 5, 5, 2, 2, 2),
                 (3, 4, 230, 230, 16, 7, 7, 2, 3, 3), (2, 2, 330, 250, 33, 3, 5, 1, 1, 2)]


@pytest.mark.parametrize("args", NARROW_SHAPES)
def test_ffma_four_channel_slices(args):
    N, Ci, H, W, Co, kH, kW, s, ph, pw = args
    assert dg.describe(*args, "fp32")["slice_n"] == 4
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 93, "kaiming")
    ref, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    narrow, info = run_gpu(args, go, w, "fp32")
    assert info["slice_n"] == 4 and info["a_source"] == "producers"
    assert_fp32(narrow, ref)
    frame, info = run_gpu(args, go, w, "fp32", a_source="frame")
    assert info["slice_n"] == 16
    assert np.array_equal(narrow, frame)


@pytest.mark.parametrize("a_source", ["frame", "producers"])
@pytest.mark.parametrize("opts", [dict(slice_n=16), dict(slice_n=32, chunk_k=8), dict(chunk_k=32)])
def test_simt_tilings_each_source(opts, a_source):
    shape = (2, 40, 36, 19, 23, 3, 3, 2, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 79, "kaiming")
    info = check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "fp32", path="simt", a_source=a_source, **opts)
    assert info["a_source"] == a_source


def test_simt_with_tf32_operands():
    # The FFMA path on TF32-rounded operands satisfies the TF32 bar too.
    shape = (2, 24, 40, 13, 15, 3, 3, 1, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, H, W), (Co, Ci, kH, kW), 83, "kaiming")
    check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "tf32", path="simt")


STAGED_EDGE = [
    (1, 1, 1, 6, 6, 3, 3, 1, 1, 1), (3, 3, 4, 8, 12, 5, 5, 1, 2, 2), (1, 5, 33, 10, 9, 3, 3, 2, 1, 0),
    (3, 65, 4, 12, 12, 3, 3, 3, 1, 1), (1, 129, 33, 8, 8, 1, 1, 2, 0, 0), (3, 5, 33, 12, 16, 2, 2, 2, 0, 0),
    (1, 3, 1, 12, 16, 3, 5, 1, 2, 2), (3, 1, 4, 16, 8, 5, 3, 1, 2, 1), (1, 3, 4, 2, 8, 3, 3, 2, 1, 1),
    (3, 16, 20, 32, 28, 3, 3, 1, 1, 1), (1, 20, 40, 40, 40, 3, 3, 4, 1, 1), (5, 7, 9, 20, 4, 3, 3, 1, 1, 1),
]


@pytest.mark.parametrize("a_source", ["frame", "producers", "staged"])
@pytest.mark.parametrize("shape", EDGE[:10] + STAGED_EDGE)
def test_edge_shapes_both_sources(shape, a_source):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    if a_source == "staged":
        try:
            dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, "tf32", a_source="staged")
        except dg.DgradError as e:
            if e.status == 2:
                pytest.skip("grad_out planes not 16-byte aligned, or the band does not fit one copy")
            raise
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 72, "uniform")
    info = check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "tf32", a_source=a_source)
    assert info["a_source"] == a_source


@pytest.mark.parametrize("group_taps", ["on", "off", "phases"])
@pytest.mark.parametrize("shape", EDGE)
def test_edge_shapes_grouped_and_not(shape, group_taps):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    try:
        dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, "tf32", group_taps=group_taps)
    except dg.DgradError as e:
        if e.status == 2:
            pytest.skip("taps of a kernel row cannot share one MMA here")
        raise
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 74, "uniform")
    info = check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "tf32", group_taps=group_taps)
    assert info["group_taps"] == {"on": 1, "off": 0, "phases": 2}[group_taps]


# ----------------------------------------------------------------- fused epilogue
@pytest.mark.parametrize("precision", ["tf32", "fp32", "tf32x3"])
@pytest.mark.parametrize("mode", ["relu", "accumulate", "both"])
@pytest.mark.parametrize("shape", [(2, 5, 7, 9, 11, 3, 3, 1, 1, 1), (2, 48, 20, 17, 18, 3, 3, 2, 1, 1),
                                   (3, 33, 70, 9, 14, 1, 1, 1, 0, 0), (1, 20, 40, 40, 40, 3, 3, 4, 1, 1),
                                   (2, 16, 24, 12, 12, 3, 3, 1, 1, 1), (2, 48, 20, 16, 16, 3, 3, 2, 1, 1),
                                   (3, 33, 70, 8, 14, 1, 1, 1, 0, 0), (3, 33, 70, 12, 12, 1, 1, 1, 0, 0)])
def test_fused_epilogue(shape, mode, precision):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 77, "kaiming")
    gen = torch.Generator().manual_seed(78)
    relu_in = torch.randn((N, Ci, H, W), generator=gen) if mode in ("relu", "both") else None
    gi0 = torch.randn((N, Ci, H, W), generator=gen) if mode in ("accumulate", "both") else None
    ref, mag = oracle.dgrad_fused(go, w, H, W, s, ph, pw, relu_in=relu_in, grad_in=gi0)
    with dg.Plan(N, Ci, H, W, Co, kH, kW, s, ph, pw, precision=precision) as plan:
        gi = gi0.cuda() if gi0 is not None else torch.full((N, Ci, H, W), float("nan"), device="cuda")
        plan.run(go.cuda(), w.cuda(), gi, relu_in=relu_in.cuda() if relu_in is not None else None,
                 accumulate=gi0 is not None)
        torch.cuda.synchronize()
        plan.check()
    out = gi.cpu().double().numpy()
    assert np.isfinite(out).all()
    # bound: the dgrad part's own bound (the TF32 bar, or the classic fp32 dot-product bound
    # (K + 2) * 2^-24 * sum|terms| with K = Co*kH*kW terms) plus one fp32 rounding of the sum
    if precision == "tf32":
        part = TF32_REL_TERMS * mag
    elif precision == "tf32x3":
        part = split_bound(Co, kH, kW) * mag
    else:
        part = (Co * kH * kW + 2) * 2.0 ** -24 * mag
    bound = part + 2.0 ** -23 * np.abs(ref)
    err = np.abs(out - ref)
    assert (err <= bound + 1e-30).all(), f"worst err / bound = {np.max(err / (bound + 1e-30)):.3e}"
    if relu_in is not None and gi0 is None:
        assert (out[(relu_in <= 0).numpy()] == 0).all()   # masked elements are exactly 0


def test_fused_rejects_bad_arguments():
    wl = WORKLOADS["tiny"]
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        lib = dg.load_library()
        go = torch.zeros(wl.go_shape, device="cuda")
        w = torch.zeros(wl.w_shape, device="cuda")
        gi = torch.zeros(wl.gi_shape, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        assert lib.dgrad_run_fused(plan._h, P(go), P(w), P(gi), P(gi), 0, stream) == 4      # relu_in over grad_input
        assert lib.dgrad_run_fused(plan._h, P(go), P(w), P(gi), None, 2, stream) == 1        # accumulate not 0/1
        buf = torch.zeros(gi.numel() + 16, device="cuda")
        assert lib.dgrad_run_fused(plan._h, P(go), P(w), P(gi), ctypes.c_void_p(buf.data_ptr() + 4), 0,
                                   stream) == 3
        torch.cuda.synchronize()
        plan.check()


# ----------------------------------------------------------------- semantics
def test_infinite_weight_on_padding_only_tap_stays_finite():
    # H = W = 2, 3x3, pad 1, stride 2: kernel row 0 and column 0 only ever meet
    # padding, so the definition never multiplies them; the result is finite.
    N, Ci, Co, H, W = 1, 3, 4, 2, 2
    go, w = make_tensors((N, Co, 1, 1), (Co, Ci, 3, 3), 89, "uniform")
    w[:, :, 0, :] = float("inf")
    w[:, :, :, 0] = float("-inf")
    ref, mag = oracle.dgrad(go, w, H, W, 2, 1, 1)
    assert np.isfinite(ref).all()
    for prec in ("tf32", "fp32"):
        gpu, _ = run_gpu((N, Ci, H, W, Co, 3, 3, 2, 1, 1), go, w, prec)
        assert np.isfinite(gpu).all()
        if prec == "fp32":
            assert_fp32(gpu, ref)
        else:
            assert_tf32(gpu, ref, mag)


def test_overwrites_and_leaves_inputs_alone():
    wl = WORKLOADS["tiny"]
    go, w = make_inputs(wl, 5)
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        gd, wd = go.cuda(), w.cuda()
        gi = torch.full(wl.gi_shape, 123.0, device="cuda")
        plan.run(gd, wd, gi)
        first = gi.clone()
        plan.run(gd, wd, gi)
        torch.cuda.synchronize()
        plan.check()
        assert torch.equal(first, gi), "second run differs: not an overwrite, or not deterministic"
        assert torch.equal(gd.cpu(), go) and torch.equal(wd.cpu(), w)


def test_prepack_then_run_packed_matches_run():
    wl = WORKLOADS["strided_downsample"]
    go, w = make_tensors((2, wl.Co, wl.oH, wl.oW), wl.w_shape, 97, wl.dist)
    args = (2,) + wl.plan_args()[1:]
    with dg.Plan(*args, precision="tf32") as plan:
        gd, wd = go.cuda(), w.cuda()
        a = plan.run(gd, wd)
        plan.prepack(wd)
        b = plan.run_packed(gd)
        c = plan.run_packed(gd)
        torch.cuda.synchronize()
        assert torch.equal(a, b) and torch.equal(b, c)


@pytest.mark.parametrize("name", ["tiny", "strided_downsample"])
def test_staged_calls_match_run(name):
    """prepack + pack_grad_out + run_main, with the stages in separate calls
    and the main kernel run twice on one packing, equals run."""
    wl = WORKLOADS[name]
    go, w = make_tensors((2, wl.Co, wl.oH, wl.oW), wl.w_shape, 41, wl.dist)
    args = (2,) + wl.plan_args()[1:]
    with dg.Plan(*args, precision="tf32") as plan:
        gd, wd = go.cuda(), w.cuda()
        a = plan.run(gd, wd)
        other = torch.randn_like(gd)
        plan.run(other, wd)                  # leaves another tensor's frame behind
        plan.prepack(wd)
        plan.pack_grad_out(gd)
        b = plan.run_main(gd)
        c = plan.run_main(gd)
        torch.cuda.synchronize()
        plan.check()
        assert torch.equal(a, b) and torch.equal(b, c)


def test_run_main_before_packing_is_rejected():
    wl = WORKLOADS["tiny"]
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        gd = torch.zeros(wl.go_shape, device="cuda")
        with pytest.raises(dg.DgradError) as e:
            plan.run_main(gd)
        assert e.value.status == 1
        plan.prepack(torch.zeros(wl.w_shape, device="cuda"))
        if plan.info["a_source"] == "frame":  # frame path: the frame was never packed
            with pytest.raises(dg.DgradError) as e:
                plan.run_main(gd)
            assert e.value.status == 1
        plan.pack_grad_out(gd)
        plan.run_main(gd)
        torch.cuda.synchronize()
        plan.check()


def test_run_host_matches_device():
    wl = WORKLOADS["tiny"]
    go, w = make_inputs(wl, 7)
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        dev = plan.run(go.cuda(), w.cuda())
        host = plan.run_host(go.pin_memory(), w.pin_memory())
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu(), host)
        plan.check()


@pytest.mark.parametrize("shape,precision,pinned", [
    ((32, 64, 56, 56, 64, 3, 3, 1, 1, 1), "tf32", True),    # four chunks of eight images
    ((11, 5, 17, 19, 33, 3, 3, 2, 1, 1), "tf32", True),     # chunks of three and a remainder of two
    ((11, 5, 17, 19, 33, 3, 3, 2, 1, 1), "fp32", False),    # FFMA path, pageable host memory
    ((3, 3, 40, 38, 64, 7, 7, 2, 3, 3), "tf32x3", True),
])
def test_run_host_pipeline_matches_device(shape, precision, pinned):
    """The host entry point runs the batch in chunks through sub-plans, copies
    overlapping the runs; every element is the device run's, bit for bit (the
    per-element summation order does not depend on the batch)."""
    N, Ci, H, W, Co, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 83, "kaiming")
    with dg.Plan(*shape, precision=precision) as plan:
        dev = plan.run(go.cuda(), w.cuda()).cpu()
        gh, wh = (go.pin_memory(), w.pin_memory()) if pinned else (go, w)
        out = torch.empty((N, Ci, H, W), pin_memory=pinned)
        for _ in range(2):   # the pipeline is made on the first call and reused
            out.fill_(float("nan"))
            plan.run_host(gh, wh, out)
            assert torch.equal(dev, out)
        plan.check()


def test_side_stream():
    wl = WORKLOADS["tiny"]
    go, w = make_inputs(wl, 8)
    ref, mag = oracle.dgrad(go, w, wl.H, wl.W, 1, 1, 1)
    s = torch.cuda.Stream()
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        with torch.cuda.stream(s):
            gd, wd = go.cuda(), w.cuda()
            gi = plan.run(gd, wd, stream=s)
        s.synchronize()
        assert_tf32(gi.cpu().double().numpy(), ref, mag)


def test_rejects_bad_pointers():
    wl = WORKLOADS["tiny"]
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        lib = dg.load_library()
        go = torch.zeros(wl.go_shape, device="cuda")
        w = torch.zeros(wl.w_shape, device="cuda")
        gi = torch.zeros(wl.gi_shape, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        buf = torch.zeros(go.numel() + 16, device="cuda")
        misaligned = ctypes.c_void_p(buf.data_ptr() + 4)
        assert lib.dgrad_run(plan._h, misaligned, ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(gi.data_ptr()), stream) == 3
        assert lib.dgrad_run(plan._h, ctypes.c_void_p(go.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(go.data_ptr()), stream) == 4
        assert lib.dgrad_run(plan._h, None, ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(gi.data_ptr()), stream) == 3
        assert lib.dgrad_run(None, ctypes.c_void_p(go.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(gi.data_ptr()), stream) == 1
        torch.cuda.synchronize()
        plan.check()


def test_run_packed_before_prepack_is_rejected():
    wl = WORKLOADS["tiny"]
    with dg.Plan(*wl.plan_args(), precision="tf32") as plan:
        with pytest.raises(dg.DgradError) as e:
            plan.run_packed(torch.zeros(wl.go_shape, device="cuda"))
        assert e.value.status == 1


# ----------------------------------------------------------------- full size, sampled
@pytest.mark.parametrize("precision", ["tf32", "tf32x3"])
@pytest.mark.parametrize("name", ["resnet_stage", "strided_downsample", "pointwise", "stem"])
def test_full_size_sampled_definition(name, precision):
    """At full size in the benchmark's launch configuration: 4096 sampled
    elements against the definition computed one by one."""
    wl = WORKLOADS[name]
    go, w = make_inputs(wl, 0)
    gpu, _ = run_gpu(wl.plan_args(), go, w, precision)
    rng = np.random.default_rng(101)
    idx = np.stack([rng.integers(0, wl.N, 4096), rng.integers(0, wl.Ci, 4096),
                    rng.integers(0, wl.H, 4096), rng.integers(0, wl.W, 4096)], 1)
    acc, mag = oracle.dgrad_at(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w, idx)
    g = gpu[idx[:, 0], idx[:, 1], idx[:, 2], idx[:, 3]]
    rel = TF32_REL_TERMS if precision == "tf32" else split_bound(wl.Co, wl.kH, wl.kW)
    assert np.all(np.abs(g - acc) <= rel * mag)
    if precision == "tf32x3":
        assert np.linalg.norm(g - acc) <= FP32_REL_L2 * np.linalg.norm(acc)


# ----------------------------------------------------------------- split precision
@pytest.mark.parametrize("shape", [(2, 48, 20, 17, 18, 3, 3, 2, 1, 1), (3, 33, 70, 9, 14, 1, 1, 1, 0, 0),
                                   (1, 3, 64, 40, 38, 7, 7, 2, 3, 3)])
def test_split_precision_beats_tf32(shape):
    """The split path's error is far below the TF32 path's on the same inputs
    (values with full 24-bit mantissas, where TF32 rounding shows)."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 79, "kaiming")
    ref, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    e = {}
    for prec in ("tf32", "tf32x3"):
        gpu, _ = run_gpu(shape[:1] + (Ci, H, W, Co, kH, kW, s, ph, pw), go, w, prec)
        e[prec] = np.linalg.norm(gpu - ref) / np.linalg.norm(ref)
    assert e["tf32x3"] <= FP32_REL_L2 and e["tf32x3"] * 50 < e["tf32"], e


def test_split_precision_rejects_other_sources():
    with pytest.raises(dg.DgradError) as e:
        dg.Plan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, precision="tf32x3", path="simt")
    assert e.value.status == 2
    with pytest.raises(dg.DgradError) as e:
        dg.Plan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, precision="tf32x3", a_source="producers")
    assert e.value.status == 2


# ----------------------------------------------------------------- GEMM + col2im path (few input channels)
C2I_SHAPES = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw
    (2, 3, 64, 40, 38, 7, 7, 2, 3, 3),      # stem-like
    (3, 3, 4, 9, 11, 5, 5, 1, 1, 1),
    (1, 1, 1, 5, 7, 3, 3, 1, 0, 0),
    (1, 3, 33, 23, 21, 7, 7, 2, 3, 3),
    (3, 4, 33, 12, 14, 2, 2, 2, 0, 0),
    (1, 3, 1, 11, 17, 3, 5, 1, 2, 1),
    (1, 3, 4, 2, 2, 3, 3, 2, 1, 1),         # a kernel row that only meets padding
    (1, 4, 3, 1, 1, 1, 1, 2, 1, 1),         # no term reaches any input element
    (2, 2, 70, 130, 9, 3, 3, 1, 1, 1),      # several bands per image, ragged last band
    (1, 4, 40, 40, 40, 3, 3, 4, 1, 1),      # stride 4
    (2, 4, 16, 20, 22, 8, 8, 1, 3, 4),      # 256 GEMM columns, non-same padding
]


@pytest.mark.parametrize("shape", C2I_SHAPES)
def test_col2im_path(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 80, "uniform")
    info = check((N, Ci, H, W, Co, kH, kW, s, ph, pw), go, w, "tf32", path="col2im")
    assert info["path"] == "col2im"


@pytest.mark.parametrize("mode", ["relu", "accumulate", "both"])
def test_col2im_fused_epilogue(mode):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = (2, 3, 20, 17, 18, 7, 7, 2, 3, 3)
    go, w = make_tensors((N, Co, out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)), (Co, Ci, kH, kW), 81, "kaiming")
    gen = torch.Generator().manual_seed(82)
    relu_in = torch.randn((N, Ci, H, W), generator=gen) if mode in ("relu", "both") else None
    gi0 = torch.randn((N, Ci, H, W), generator=gen) if mode in ("accumulate", "both") else None
    ref, mag = oracle.dgrad_fused(go, w, H, W, s, ph, pw, relu_in=relu_in, grad_in=gi0)
    with dg.Plan(N, Ci, H, W, Co, kH, kW, s, ph, pw, precision="tf32", path="col2im") as plan:
        gi = gi0.cuda() if gi0 is not None else torch.full((N, Ci, H, W), float("nan"), device="cuda")
        plan.run(go.cuda(), w.cuda(), gi, relu_in=relu_in.cuda() if relu_in is not None else None,
                 accumulate=gi0 is not None)
        torch.cuda.synchronize()
        plan.check()
    out = gi.cpu().double().numpy()
    bound = TF32_REL_TERMS * mag + 2.0 ** -23 * np.abs(ref)
    assert (np.abs(out - ref) <= bound + 1e-30).all()


def test_col2im_full_size_stem_sampled():
    wl = WORKLOADS["stem"]
    go, w = make_inputs(wl, 0)
    gpu, info = run_gpu(wl.plan_args(), go, w, "tf32", path="col2im")
    assert info["path"] == "col2im"
    rng = np.random.default_rng(103)
    idx = np.stack([rng.integers(0, wl.N, 4096), rng.integers(0, wl.Ci, 4096),
                    rng.integers(0, wl.H, 4096), rng.integers(0, wl.W, 4096)], 1)
    acc, mag = oracle.dgrad_at(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w, idx)
    g = gpu[idx[:, 0], idx[:, 1], idx[:, 2], idx[:, 3]]
    assert np.all(np.abs(g - acc) <= TF32_REL_TERMS * mag)
    assert np.isfinite(gpu).all()


def test_col2im_rejects_unsupported():
    with pytest.raises(dg.DgradError) as e:
        dg.Plan(1, 3, 16, 16, 8, 3, 3, 1, 1, 1, precision="fp32", path="col2im")
    assert e.value.status == 2
    with pytest.raises(dg.DgradError) as e:
        dg.Plan(1, 4, 16, 16, 8, 9, 9, 1, 1, 1, precision="tf32", path="col2im")   # 324 GEMM columns > 256
    assert e.value.status == 2
    with pytest.raises(dg.DgradError) as e:
        dg.Plan(1, 5, 16, 16, 8, 3, 3, 1, 1, 1, precision="tf32", path="col2im")   # more than 4 input channels
    assert e.value.status == 2
