"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/dgrad.h declares, validates shapes, and its phase / tap /
frame tables reproduce the oracle when the main kernels' arithmetic is
emulated with numpy on the CPU."""
import os
import re

import numpy as np
import pytest

import oracle
import conv2d_backward_implicit_dgrad_gb300 as dg
from conv2d_backward_implicit_dgrad_gb300 import binding
from conv2d_backward_implicit_dgrad_gb300.workloads import ORDER, WORKLOADS, make_tensors

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b((?:dgrad|wgrad)_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_function():
    lib = dg.load_library()
    declared = header_functions()
    assert declared, "no declarations found"
    assert declared == set(binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    lib = dg.load_library()
    for code in range(10):
        assert lib.dgrad_status_string(code)
    assert lib.dgrad_status_string(99) == b"unknown status"


@pytest.mark.parametrize("bad", [
    (0, 1, 4, 4, 1, 3, 3, 1, 1, 1), (1, 0, 4, 4, 1, 3, 3, 1, 1, 1), (1, 1, 4, 4, 1, 3, 3, 0, 1, 1),
    (1, 1, 4, 4, 1, 3, 3, 1, -1, 1), (1, 1, 2, 2, 1, 5, 5, 1, 0, 0), (1, 1, 4, 4, 0, 3, 3, 1, 1, 1)])
def test_describe_rejects_invalid(bad):
    with pytest.raises(dg.DgradError) as e:
        dg.describe(*bad)
    assert e.value.status == 1


@pytest.mark.parametrize("bad", [(1, 1, 32, 32, 1, 3, 3, 5, 1, 1), (1, 1, 40, 40, 1, 12, 12, 1, 0, 0)])
def test_describe_rejects_unsupported(bad):
    with pytest.raises(dg.DgradError) as e:
        dg.describe(*bad)
    assert e.value.status == 2


def test_describe_rejects_bad_options():
    with pytest.raises(dg.DgradError) as e:
        dg.describe(2, 8, 8, 8, 8, 3, 3, 1, 1, 1, "fp32", path="tcgen05")
    assert e.value.status == 2
    for bad in (dict(slice_n=24), dict(chunk_k=12), dict(chunk_k=16), dict(tile_blocks=5)):
        with pytest.raises(dg.DgradError) as e:
            dg.describe(2, 8, 8, 8, 8, 3, 3, 1, 1, 1, "tf32", **bad)
        assert e.value.status == 1


def test_plan_without_device_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(dg.DgradError) as e:
        dg.Plan(1, 1, 4, 4, 1, 3, 3, 1, 1, 1)
    assert e.value.status in (8, 6)


@pytest.mark.parametrize("name", ORDER)
def test_describe_workloads(name):
    wl = WORKLOADS[name]
    for prec in ("tf32", "fp32"):
        d = dg.describe(*wl.plan_args(), precision=prec)
        assert (d["oH"], d["oW"]) == (wl.oH, wl.oW)
        assert d["useful_flops"] == 2 * wl.N * wl.Co * wl.oH * wl.oW * wl.Ci * wl.kH * wl.kW
        assert d["path"] == ("tcgen05" if prec == "tf32" else "simt")
        assert d["n_phases"] == min(wl.stride, wl.H) * min(wl.stride, wl.W)
        assert d["smem_bytes"] <= 232448
        if prec == "tf32":
            assert 32 <= d["tmem_cols"] <= 512
            assert d["slice_n"] % 16 == 0 and 16 <= d["slice_n"] <= 256
            assert d["grid"] <= 152


def test_phase_taps_partition_the_kernel():
    # Every kernel tap belongs to exactly one phase when none is pruned.
    phases, taps = dg.describe_taps(2, 3, 28, 28, 4, 3, 3, 2, 1, 1)
    assert sorted((t["kh"], t["kw"]) for t in taps) == [(kh, kw) for kh in range(3) for kw in range(3)]
    assert sum(p["tap_count"] for p in phases) == 9
    phases, taps = dg.describe_taps(2, 3, 224, 224, 4, 7, 7, 2, 3, 3)
    assert sorted(p["tap_count"] for p in phases) == [9, 12, 12, 16]
    phases, taps = dg.describe_taps(2, 3, 8, 8, 4, 1, 1, 2, 0, 0)   # 1x1 stride 2: three phases have no taps
    assert sorted(p["tap_count"] for p in phases) == [0, 0, 0, 1]


def test_padding_only_taps_are_pruned():
    # H = 2, k = 3, pad 1, stride 2: kernel row 0 only ever meets padding.
    phases, taps = dg.describe_taps(1, 1, 2, 2, 1, 3, 3, 2, 1, 1)
    assert all(t["kh"] != 0 and t["kw"] != 0 for t in taps)


def emulate(go, w, H, W, s, ph, pw):
    """The main kernels' arithmetic in numpy, driven only by the library's tables:
    shifted windows of the zero-padded flattened frame, one GEMM per tap and phase."""
    N, Co, oH, oW = go.shape
    _, Ci, kH, kW = w.shape
    info = dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw)
    phases, taps = dg.describe_taps(N, Ci, H, W, Co, kH, kW, s, ph, pw)
    Ph, Pw, Hv, Wp = info["Ph"], info["Pw"], info["Hv"], info["Wp"]
    assert Hv >= oH + Ph and Wp >= oW + Pw
    P = N * Hv * Wp
    V = np.zeros((P + info["max_shift"] + 8, Co))
    frame = np.zeros((N, Hv, Wp, Co))
    frame[:, Ph:Ph + oH, Pw:Pw + oW, :] = go.transpose(0, 2, 3, 1)
    V[:P] = frame.reshape(P, Co)
    gi = np.full((N, Ci, H, W), np.nan)
    pos = np.arange(P)
    n_idx, rem = pos // (Hv * Wp), pos % (Hv * Wp)
    q_idx, u_idx = rem // Wp, rem % Wp
    for p in phases:
        D = np.zeros((P, Ci))
        for t in taps[p["tap_begin"]:p["tap_begin"] + p["tap_count"]]:
            D += V[t["shift"]:t["shift"] + P] @ w[:, :, t["kh"], t["kw"]].astype(np.float64)
        ok = (q_idx < p["Hq"]) & (u_idx < p["Wq"])
        ih, iw = s * q_idx[ok] + p["a"], s * u_idx[ok] + p["b"]
        for ci in range(Ci):
            gi[n_idx[ok], ci, ih, iw] = D[ok, ci]
    return gi


def emulate_grouped(go, w, H, W, s, ph, pw, block=128):
    """The grouped MMA's arithmetic in numpy: per tile of tile_step positions,
    a 128-row block; the taps of one kernel row share the A window at the
    row's smallest shift, sub-accumulator g holds tap g's products, and the
    result of row o adds sub-accumulator g at row o + (row_len - 1 - g)."""
    N, Co, oH, oW = go.shape
    _, Ci, kH, kW = w.shape
    info = dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, group_taps="on")
    assert info["group_taps"] == 1
    phases, taps = dg.describe_taps(N, Ci, H, W, Co, kH, kW, s, ph, pw)
    Ph, Pw, Hv, Wp = info["Ph"], info["Pw"], info["Hv"], info["Wp"]
    max_row = max(p["row_len"] for p in phases)
    assert info["tile_step"] == 128 - (max_row - 1)
    T = block - (max_row - 1)   # the same construction on smaller blocks, so that small shapes span many tiles
    P = N * Hv * Wp
    n_tiles = -(-P // T)
    V = np.zeros((n_tiles * T + block + info["max_shift"], Co))
    frame = np.zeros((N, Hv, Wp, Co))
    frame[:, Ph:Ph + oH, Pw:Pw + oW, :] = go.transpose(0, 2, 3, 1)
    V[:P] = frame.reshape(P, Co)
    gi = np.full((N, Ci, H, W), np.nan)
    for p in phases:
        R = max(1, p["row_len"])
        ptaps = taps[p["tap_begin"]:p["tap_begin"] + p["tap_count"]]
        for r0 in range(0, len(ptaps), R):          # shifts fall by one inside a kernel row
            row = ptaps[r0:r0 + R]
            assert [t["shift"] for t in row] == list(range(row[0]["shift"], row[0]["shift"] - R, -1))
        for k in range(n_tiles):
            P0 = k * T
            D = np.zeros((R, block, Ci))
            for r0 in range(0, len(ptaps), R):
                row = ptaps[r0:r0 + R]
                a0 = P0 + row[-1]["shift"]
                for g, t in enumerate(row):
                    D[g] += V[a0:a0 + block] @ w[:, :, t["kh"], t["kw"]].astype(np.float64)
            out = np.zeros((T, Ci))
            for g in range(R):
                sh = R - 1 - g
                out += D[g, sh:sh + T]
            for o in range(T):
                pos = P0 + o
                if pos >= P:
                    break
                n, rem = divmod(pos, Hv * Wp)
                q, u = divmod(rem, Wp)
                if q < p["Hq"] and u < p["Wq"]:
                    gi[n, :, s * q + p["a"], s * u + p["b"]] = out[o] if p["tap_count"] else 0.0
    return gi


def emulate_staged(go, w, H, W, s, ph, pw, block=None):
    """The staged A source in numpy, driven only by the library's plan: per
    image, img_tiles tiles of tile_step positions; each tile's band is built
    from ONE copy of grad_out's plane elements [x0, x0 + stg_box) (x0 = the
    band's first element rounded down to a multiple of 4, zeros past the
    plane), row r taking the element at frame position P0 + r of the tile's
    image (zero for padding and for positions past the image); then one GEMM
    per tap over the band's shifted windows.  Checks that every element a
    row needs lies inside the copy."""
    N, Co, oH, oW = go.shape
    _, Ci, kH, kW = w.shape
    info = dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, a_source="staged", group_taps="off")
    assert info["a_source"] == "staged"
    phases, taps = dg.describe_taps(N, Ci, H, W, Co, kH, kW, s, ph, pw)
    Ph, Pw, Hv, Wp = info["Ph"], info["Pw"], info["Hv"], info["Wp"]
    img, plane = Hv * Wp, oH * oW
    T, rows, box = info["tile_step"], info["band_rows"], info["stg_box"]
    assert rows == T + info["max_shift"] and box % 4 == 0 and box <= 256 and info["a_rows"] >= max(rows, box)
    # the frame position of every plane element of an image
    el_pos = np.array([(oh + Ph) * Wp + ow + Pw for oh in range(oH) for ow in range(oW)])
    gi = np.full((N, Ci, H, W), np.nan)
    for n in range(N):
        flat = go[n].reshape(Co, plane)
        for k in range(info["img_tiles"]):
            r0 = k * T                                        # tile origin inside the image
            x0 = int(np.sum(el_pos < r0)) & ~3
            copy = np.zeros((Co, box))
            seg = flat[:, x0:x0 + box]
            copy[:, :seg.shape[1]] = seg
            band = np.zeros((rows, Co))
            for r in range(rows):
                rel = r0 + r
                if rel >= img:
                    continue
                y, x = divmod(rel, Wp)
                oh, ow = y - Ph, x - Pw
                if 0 <= oh < oH and 0 <= ow < oW:
                    loc = oh * oW + ow - x0
                    assert 0 <= loc < box, (loc, box)
                    band[r] = copy[:, loc]
            for p in phases:
                D = np.zeros((T, Ci))
                for t in taps[p["tap_begin"]:p["tap_begin"] + p["tap_count"]]:
                    D += band[t["shift"]:t["shift"] + T] @ w[:, :, t["kh"], t["kw"]].astype(np.float64)
                for o in range(T):
                    rel = r0 + o
                    if rel >= img:
                        break
                    q, u = divmod(rel, Wp)
                    if q < p["Hq"] and u < p["Wq"]:
                        gi[n, :, s * q + p["a"], s * u + p["b"]] = D[o]
    return gi


STAGED_SHAPES = [
    (2, 3, 4, 8, 8, 3, 3, 1, 1, 1), (1, 2, 3, 7, 8, 3, 3, 1, 0, 0), (2, 2, 3, 6, 8, 5, 3, 1, 2, 1),
    (1, 2, 3, 9, 9, 3, 3, 2, 1, 1), (2, 3, 2, 8, 7, 3, 3, 2, 0, 0), (1, 2, 3, 10, 9, 3, 3, 3, 1, 1),
    (2, 3, 2, 6, 6, 1, 1, 2, 0, 0), (1, 2, 2, 8, 8, 2, 2, 2, 0, 0), (3, 2, 3, 4, 13, 1, 3, 1, 0, 1),
    (2, 2, 3, 30, 22, 3, 3, 1, 1, 1), (3, 2, 2, 28, 28, 1, 1, 1, 0, 0), (2, 2, 3, 29, 31, 3, 3, 2, 1, 1),
]


@pytest.mark.parametrize("shape", STAGED_SHAPES)
def test_emulated_staged_bands_match_oracle(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    oH, oW = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
    if (oH * oW) % 4:
        with pytest.raises(dg.DgradError) as e:
            dg.describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, a_source="staged")
        assert e.value.status == 2
        return
    go, w = make_tensors((N, Co, oH, oW), (Co, Ci, kH, kW), 64, "uniform")
    go, w = go.numpy(), w.numpy()
    ref, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    emu = emulate_staged(go, w, H, W, s, ph, pw)
    assert not np.isnan(emu).any(), "an input element was never written"
    np.testing.assert_allclose(emu, ref, rtol=1e-12, atol=1e-12)


def test_tmem_source_plans():
    """1x1 / stride 1 / no padding with planes of >= 128 elements: A in tensor
    memory automatically (no frame in the workspace); other shapes refuse it."""
    pw = WORKLOADS["pointwise"]
    d = dg.describe(*pw.plan_args(), precision="tf32", sm_count=152)
    assert d["a_source"] == "tmem" and d["workspace_bytes"] == d["packed_weight_bytes"] + 256
    assert d["tmem_cols"] <= 512 and d["tile_blocks"] == 1 and d["n_phases"] == 1 and d["n_taps"] == 1
    assert dg.describe(*pw.plan_args(), precision="tf32x3", sm_count=152)["a_source"] == "tmem"
    for bad in [WORKLOADS["resnet_stage"].plan_args(), (2, 8, 8, 8, 8, 1, 1, 1, 0, 0),   # 3x3; plane of 64
                (2, 8, 14, 14, 8, 1, 1, 2, 0, 0), (2, 8, 15, 15, 8, 1, 1, 1, 0, 0)]:   # stride 2; plane % 4
        with pytest.raises(dg.DgradError) as e:
            dg.describe(*bad, precision="tf32", a_source="tmem")
        assert e.value.status == 2


@pytest.mark.parametrize("name", ["resnet_stage", "strided_downsample", "pointwise"])
def test_staged_source_plans(name):
    wl = WORKLOADS[name]
    assert dg.describe(*wl.plan_args(), precision="tf32", sm_count=152)["a_source"] in ("frame", "tmem")   # opt-in
    d = dg.describe(*wl.plan_args(), precision="tf32", sm_count=152, a_source="staged")
    assert d["a_source"] == "staged" and d["workspace_bytes"] == d["packed_weight_bytes"] + 256   # no frame
    assert d["stg_box"] <= 256 and d["a_rows"] >= max(d["band_rows"], d["stg_box"])
    # every output position of an image lies in one of its tiles
    assert d["img_tiles"] * d["tile_step"] >= (wl.H - 1) // wl.stride * d["Wp"] + 1
    # the stem's band does not fit one copy
    with pytest.raises(dg.DgradError):
        dg.describe(*WORKLOADS["stem"].plan_args(), precision="tf32", a_source="staged")


EMU_SHAPES = [
    (2, 3, 4, 8, 8, 3, 3, 1, 1, 1), (1, 2, 3, 7, 5, 3, 3, 1, 0, 0), (2, 2, 3, 6, 7, 5, 3, 1, 2, 1),
    (1, 2, 3, 9, 9, 3, 3, 2, 1, 1), (2, 3, 2, 8, 7, 3, 3, 2, 0, 0), (1, 2, 2, 9, 10, 7, 7, 2, 3, 3),
    (1, 2, 3, 10, 9, 3, 3, 3, 1, 1), (2, 3, 2, 6, 6, 1, 1, 2, 0, 0), (1, 2, 2, 8, 8, 2, 2, 2, 0, 0),
    (1, 2, 2, 9, 8, 4, 3, 2, 1, 2), (1, 1, 2, 2, 2, 3, 3, 2, 1, 1), (2, 2, 2, 5, 6, 3, 5, 1, 2, 2),
    (1, 2, 2, 11, 12, 5, 5, 3, 2, 2), (1, 1, 1, 1, 1, 1, 1, 1, 0, 0), (1, 2, 3, 3, 3, 3, 3, 1, 2, 2),
    (3, 2, 3, 4, 13, 1, 3, 1, 0, 1), (1, 2, 2, 13, 13, 3, 3, 4, 1, 1), (1, 1, 2, 1, 9, 1, 3, 2, 0, 1),
]


@pytest.mark.parametrize("shape", EMU_SHAPES)
def test_emulated_decomposition_matches_oracle(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    oH, oW = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
    go, w = make_tensors((N, Co, oH, oW), (Co, Ci, kH, kW), 61, "uniform")
    go, w = go.numpy(), w.numpy()
    ref, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    emu = emulate(go, w, H, W, s, ph, pw)
    assert not np.isnan(emu).any(), "an input element was never written"
    np.testing.assert_allclose(emu, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", ["tiny", "strided_downsample"])
def test_emulated_decomposition_workload_shapes(name):
    wl = WORKLOADS[name]
    N = min(wl.N, 1)
    go, w = make_tensors((N, wl.Co, wl.oH, wl.oW), wl.w_shape, 62, wl.dist)
    go, w = go.numpy(), w.numpy()
    ref, _ = oracle.dgrad(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    emu = emulate(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    np.testing.assert_allclose(emu, ref, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("shape", EMU_SHAPES)
def test_emulated_grouped_taps_match_oracle(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    if max(kW, -(-kW // s)) > 4 and s == 1:
        pytest.skip("rows longer than four taps are not grouped")
    oH, oW = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
    go, w = make_tensors((N, Co, oH, oW), (Co, Ci, kH, kW), 63, "uniform")
    go, w = go.numpy(), w.numpy()
    ref, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    emu = emulate_grouped(go, w, H, W, s, ph, pw, block=16)
    assert not np.isnan(emu).any(), "an input element was never written"
    np.testing.assert_allclose(emu, ref, rtol=1e-12, atol=1e-12)


def test_grouping_plans():
    r = dg.describe(*WORKLOADS["resnet_stage"].plan_args(), precision="tf32")
    assert r["group_taps"] == 1 and r["tile_step"] == 126   # automatic for one phase with bn < 128
    on = dg.describe(*WORKLOADS["resnet_stage"].plan_args(), precision="tf32", group_taps="on")
    assert on["group_taps"] == 1 and on["tile_step"] == 126 and on["tmem_cols"] == 512
    off = dg.describe(*WORKLOADS["resnet_stage"].plan_args(), precision="tf32", group_taps="off")
    assert off["group_taps"] == 0 and off["tile_step"] == 128 * off["tile_blocks"]
    pw = dg.describe(*WORKLOADS["pointwise"].plan_args(), precision="tf32")
    assert pw["group_taps"] == 0                              # 1x1: one tap per row
    t2 = dg.describe(*WORKLOADS["resnet_stage"].plan_args(), precision="tf32", tile_blocks=2)
    assert t2["group_taps"] == 0 and t2["tile_step"] == 256   # two blocks per unit: ungrouped
    st = dg.describe(*WORKLOADS["stem"].plan_args(), precision="tf32", group_taps="on")
    assert st["group_taps"] == 1 and st["tile_step"] == 125
    with pytest.raises(dg.DgradError) as e:    # 5 taps per row cannot share one MMA
        dg.describe(2, 16, 16, 16, 16, 5, 5, 1, 2, 2, precision="tf32", group_taps="on")
    assert e.value.status == 2


def test_shared_shift_plans():
    st = dg.describe(*WORKLOADS["strided_downsample"].plan_args(), precision="tf32")
    assert st["group_taps"] == 2                       # automatic for stride 2
    off = dg.describe(*WORKLOADS["strided_downsample"].plan_args(), precision="tf32", group_taps="off")
    assert off["group_taps"] == 0 and off["packed_weight_bytes"] == st["packed_weight_bytes"]
    for bad in [(2, 8, 8, 8, 8, 3, 3, 1, 1, 1),        # one phase: nothing to share
                (1, 20, 40, 40, 40, 3, 3, 4, 1, 1)]:   # sixteen phases
        with pytest.raises(dg.DgradError) as e:
            dg.describe(*bad, precision="tf32", group_taps="phases")
        assert e.value.status == 2


# ----------------------------------------------------------------- split precision (TF32X3)
def test_split_precision_plans():
    for name in ORDER:
        wl = WORKLOADS[name]
        d = dg.describe(*wl.plan_args(), precision="tf32x3")
        t = dg.describe(*wl.plan_args(), precision="tf32")
        assert d["path"] == "tcgen05" and d["precision"] == "tf32x3"
        # the packed frame, except 1x1 unpadded stride-1 shapes, whose A goes to tensor memory
        assert d["a_source"] == ("tmem" if name == "pointwise" else "frame")
        assert d["n_chunks"] == 3 * -(-wl.Co // 32)           # three K passes per channel chunk
        assert d["smem_bytes"] <= 232448 and d["tmem_cols"] <= 512
        assert d["useful_flops"] == t["useful_flops"]
    # a frame above the size at which TF32 plans switch to producer warps stays a frame
    big = (64, 64, 224, 224, 256, 3, 3, 1, 1, 1)   # a 3.3 GB frame
    assert dg.describe(*big, precision="tf32")["a_source"] == "producers"
    assert dg.describe(*big, precision="tf32x3")["a_source"] == "frame"
    for bad in (dict(path="simt"), dict(a_source="producers")):
        with pytest.raises(dg.DgradError) as e:
            dg.describe(2, 8, 8, 8, 8, 3, 3, 1, 1, 1, "tf32x3", **bad)
        assert e.value.status == 2


def _rna_tf32(x):
    """Round fp32 values to TF32 (10 stored mantissa bits), to nearest with
    ties away from zero: add half of the dropped part to the magnitude bits,
    then clear the 13 dropped bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def test_tf32_rounding_model():
    # values with a known TF32 rounding: 1 + 2^-11 is a tie (rounds away), 1 + 2^-11 + 2^-23 rounds up,
    # 1 + 2^-12 rounds down, and negative values mirror positive ones
    x = np.array([1.0, 1 + 2.0 ** -11, 1 + 2.0 ** -11 + 2.0 ** -23, 1 + 2.0 ** -12, -(1 + 2.0 ** -11)], np.float32)
    assert _rna_tf32(x).tolist() == [1.0, 1 + 2.0 ** -10, 1 + 2.0 ** -10, 1.0, -(1 + 2.0 ** -10)]


def test_split_arithmetic_bound():
    """The split-precision arithmetic, modelled on the CPU with exact products:
    go = hi + lo + r and w likewise, the three partial products hi*lo, lo*hi
    and hi*hi summed exactly.  Each product is then within 2^-20 of its size of
    the true one, so the result is within 2^-20 * sum|terms| of the definition;
    plain TF32 (hi*hi alone) is not."""
    rng = np.random.default_rng(9)
    N, Ci, Co, H, W, k, s, p = 2, 5, 7, 9, 10, 3, 2, 1
    oH, oW = (H + 2 * p - k) // s + 1, (W + 2 * p - k) // s + 1
    go = rng.standard_normal((N, Co, oH, oW)).astype(np.float32)
    w = (rng.standard_normal((Co, Ci, k, k)) * 0.3).astype(np.float32)
    ref, mag = oracle.dgrad(go, w, H, W, s, p, p)
    go_hi, w_hi = _rna_tf32(go), _rna_tf32(w)
    go_lo, w_lo = _rna_tf32(go - go_hi), _rna_tf32(w - w_hi)
    assert np.all(np.abs(go - go_hi - go_lo) <= 2.0 ** -22 * np.abs(go))
    split = sum(oracle.dgrad(a, b, H, W, s, p, p, with_mag=False)[0]
                for a, b in ((go_hi, w_lo), (go_lo, w_hi), (go_hi, w_hi)))
    assert np.all(np.abs(split - ref) <= 2.0 ** -20 * mag)
    one = oracle.dgrad(go_hi, w_hi, H, W, s, p, p, with_mag=False)[0]
    assert np.max(np.abs(one - ref) / np.maximum(mag, 1e-30)) > 2.0 ** -16


# ----------------------------------------------------------------- weight gradient: plan tables
WG_SHAPES = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw
    (2, 3, 4, 8, 8, 3, 3, 1, 1, 1),
    (1, 5, 33, 10, 9, 3, 3, 2, 0, 0),
    (3, 65, 4, 7, 13, 3, 3, 3, 1, 1),
    (1, 129, 33, 6, 10, 1, 1, 2, 0, 0),
    (1, 3, 4, 23, 21, 7, 7, 2, 3, 3),
    (2, 5, 20, 12, 14, 2, 2, 2, 0, 0),
    (1, 3, 1, 11, 17, 3, 5, 1, 2, 1),
    (1, 65, 33, 17, 19, 4, 3, 2, 1, 2),
    (1, 3, 4, 2, 2, 3, 3, 2, 1, 1),
    (2, 4, 300, 9, 7, 3, 3, 1, 1, 1),
    (5, 3, 4, 9, 11, 3, 3, 1, 1, 1),       # four images interleaved, a ragged last group
    (4, 6, 8, 12, 10, 3, 3, 2, 1, 1),
    (7, 2, 3, 10, 13, 7, 7, 2, 3, 3),
    (6, 4, 5, 11, 9, 5, 3, 3, 2, 1),
    (3, 3, 2, 8, 9, 3, 4, 1, 1, 2),
    (3, 40, 24, 6, 10, 1, 1, 1, 0, 0),     # 1x1: direct mode, no frames
    (2, 8, 16, 5, 5, 1, 1, 1, 0, 0),       # 1x1 with 25 positions per plane: frames
    (32, 3, 4, 7, 9, 3, 3, 1, 1, 1),       # batch-blocked frames (32 images per K chunk)
    (35, 5, 3, 8, 6, 3, 3, 2, 1, 1),       # 35 images: four interleaved (blocking would pad 29)
    (60, 5, 3, 8, 6, 3, 3, 2, 1, 1),       # blocked, four padding images
    (33, 2, 2, 5, 7, 5, 3, 3, 2, 1),
]


def emulate_wgrad(go, x, kH, kW, s, ph, pw):
    """The wgrad kernels' arithmetic in numpy, driven by the library's tables:
    grad_out and input position frames with f images interleaved along K, one
    GEMM row per (tap, input channel) reading its input copy at the tap's K
    offset, row tiles and the reduction's index map back to OIHW."""
    N, Co, oH, oW = go.shape
    _, Ci, H, W = x.shape
    info = dg.wgrad_describe(N, Ci, H, W, Co, kH, kW, s, ph, pw)
    if info["mode"] == 3:   # TF32 runs the plane mode here; split precision keeps the frames
        info = dg.wgrad_describe(N, Ci, H, W, Co, kH, kW, s, ph, pw, "tf32x3")
    tab = dg.wgrad_describe_taps(N, Ci, H, W, Co, kH, kW, s, ph, pw)
    f, Wf, Kimg, Lx, Ty, Tu = tab["interleave"], info["Wf"], info["Kimg"], info["Lx"], tab["Ty"], tab["Tu"]
    assert f == info["interleave"] and f in (1, 2, 4, 32) and (info["mode"] == 2 or Wf % max(1, 4 // f) == 0)
    assert f != 32 or all(sh == 0 for sh in tab["copy_shift"])
    if info["mode"] == 2:   # direct: the caller's NCHW planes, K = image x position, no frame padding
        assert f == 1 and Wf == oW and Kimg == Lx == oH * oW and Kimg % 4 == 0 and (kH, kW, s) == (1, 1, 1)
    else:
        assert Kimg % 32 == 0 and Lx % 4 == 0 and Kimg >= oH * Wf * f and Wf >= oW
    Q = -(-N // f)
    k = np.arange(Kimg)
    j, pos = k % f, k // f
    oh, ow = pos // Wf, pos % Wf
    gf = np.zeros((Q, Co, Kimg))
    for q in range(Q):
        n = q * f + j
        ok = (n < N) & (oh < oH) & (ow < oW)
        gf[q][:, ok] = go[n[ok], :, oh[ok], ow[ok]].T
    nc = info["n_copies"]
    xc = np.zeros((nc, Q, Ci, Lx))
    kx = np.arange(Lx)
    jx, px = kx % f, kx // f
    y, u = px // Wf, px % Wf
    for c in range(nc):
        ih = s * (y - Ty) + tab["copy_rh"][c]
        iw = s * (u - Tu + tab["copy_shift"][c]) + tab["copy_rw"][c]
        for q in range(Q):
            n = q * f + jx
            ok = (n < N) & (ih >= 0) & (ih < H) & (iw >= 0) & (iw < W)
            xc[c, q][:, ok] = x[n[ok], :, ih[ok], iw[ok]].T
    dw = np.full((Co, Ci, kH * kW), np.nan)
    seg_rows = info["seg_rows"]
    cpt = -(-Ci // seg_rows)
    spt = 128 // seg_rows
    n_segs = kH * kW * cpt
    segment = info["mode"] == 0   # the run mode's rows are checked by test_wgrad_run_schedule
    assert not segment or info["n_mt"] == -(-n_segs // spt)
    for t in range(kH * kW):
        off = tab["offset"][t]
        assert off % 4 == 0 and Kimg + off <= Lx      # 16-byte aligned, inside the copy's plane
        rows = xc[tab["copy"][t], :, :, off:off + Kimg]   # [Q, Ci, Kimg]
        prod = np.einsum("qck,qik->ci", gf, rows)
        for ci in range(Ci):
            seg = t * cpt + ci // seg_rows
            mt, row = divmod(seg, spt)
            row = row * seg_rows + ci % seg_rows
            assert not segment or (mt < info["n_mt"] and row < 128)
            assert np.isnan(dw[0, ci, t])                  # each (tap, ci) row is produced once
            dw[:, ci, t] = prod[:, ci]
    assert not np.isnan(dw).any()
    return dw.reshape(Co, Ci, kH, kW)


@pytest.mark.parametrize("shape", WG_SHAPES)
def test_emulated_wgrad_matches_oracle(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    oH, oW = (H + 2 * ph - kH) // s + 1, (W + 2 * pw - kW) // s + 1
    rng = np.random.default_rng(60)
    go = rng.standard_normal((N, Co, oH, oW)).astype(np.float32)
    x = rng.standard_normal((N, Ci, H, W)).astype(np.float32)
    emu = emulate_wgrad(go.astype(np.float64), x.astype(np.float64), kH, kW, s, ph, pw)
    ref, mag = oracle.wgrad(go, x, kH, kW, s, ph, pw)
    assert np.abs(emu - ref).max() <= 1e-12 * max(1.0, mag.max())


PLANE_SHAPES = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw: stride 1, oH = H, oW = W, W a multiple of 4
    (2, 5, 7, 6, 8, 3, 3, 1, 1, 1),        # channel rows padded to 8, B columns padded to 32
    (3, 40, 24, 6, 12, 3, 3, 1, 1, 1),     # one row tile of 120 rows
    (2, 64, 64, 8, 8, 3, 3, 1, 1, 1),      # two row tiles, the second half used
    (2, 3, 4, 5, 4, 5, 5, 1, 2, 2),        # 5 x 5 taps, 20 positions: one ragged chunk per image
    (1, 16, 16, 7, 12, 3, 5, 1, 1, 2),     # 3 x 5 taps
    (2, 130, 40, 6, 8, 3, 3, 1, 1, 1),     # four row tiles x 128 columns: all of tensor memory
    (1, 8, 8, 3, 4, 3, 3, 1, 1, 1),        # one chunk in all
    (9, 8, 8, 8, 8, 3, 3, 1, 1, 1),        # K splits crossing images
]


def emulate_wgrad_plane(go, x, kH, kW, ph, pw, sm_count):
    """Plane mode in numpy, driven by the library's plan: per image, A rows
    (kw, ci) = the input shifted by kw - pw columns within each row, B rows
    (kh, co) = grad_out moved down by kh - ph rows, both over the input
    plane's positions in 32-position chunks (zero past the plane and where a
    shift leaves it); each CTA sums its contiguous chunk range into one
    partial split laid out as the kernel writes it ([row tile][column][rows
    of the tile]); the splits are added and mapped back to OIHW as the
    reduction does."""
    N, Co, H, W = go.shape
    Ci = x.shape[1]
    info = dg.wgrad_describe(N, Ci, H, W, Co, kH, kW, 1, ph, pw, sm_count=sm_count)
    assert info["mode"] == 3 and info["interleave"] == 1 and W % 4 == 0
    ci_rows, nb, n_mt, G = info["seg_rows"], info["slice_n"], info["n_mt"], info["grid"]
    co_rows = -(-Co // 8) * 8
    assert ci_rows == -(-Ci // 8) * 8 and nb == -(-kH * co_rows // 16) * 16 and nb <= 256
    a_rows = kW * ci_rows
    assert n_mt == -(-a_rows // 128) and n_mt * nb <= info["tmem_cols"] <= 512
    HW = H * W
    cpi = -(-HW // 32)
    T = N * cpi
    assert G == min(sm_count, T) and info["n_ks"] == G
    K = cpi * 32
    q = np.arange(K)
    col = q % W
    A = np.zeros((N, n_mt * 128, K))
    B = np.zeros((N, nb, K))
    xf, gf = x.reshape(N, Ci, HW), go.reshape(N, Co, HW)
    for kw in range(kW):
        d = kw - pw
        ok = (q < HW) & (col + d >= 0) & (col + d < W)
        A[:, kw * ci_rows:kw * ci_rows + Ci, ok] = xf[:, :, q[ok] + d]
    for kh in range(kH):
        src = q - (kh - ph) * W
        ok = (src >= 0) & (src < HW)
        B[:, kh * co_rows:kh * co_rows + Co, ok] = gf[:, :, src[ok]]
    total = np.zeros(a_rows * nb)
    for b in range(G):
        c0, c1 = b * T // G, (b + 1) * T // G
        assert c1 > c0
        acc = np.zeros((n_mt * 128, nb))
        for c in range(c0, c1):
            n, k0 = divmod(c, cpi)
            acc += A[n, :, 32 * k0:32 * k0 + 32] @ B[n, :, 32 * k0:32 * k0 + 32].T
        split = np.zeros(a_rows * nb)
        for mt in range(n_mt):
            rows = min(128, a_rows - mt * 128)
            split[mt * 128 * nb:mt * 128 * nb + rows * nb] = acc[mt * 128:mt * 128 + rows].T.reshape(-1)
        total += split
    dw = np.full((Co, Ci, kH, kW), np.nan)
    for i in range(a_rows * nb):
        mt, w = divmod(i, 128 * nb)
        rows = min(128, a_rows - mt * 128)
        c, row = divmod(w, rows)
        kw, ci = divmod(mt * 128 + row, ci_rows)
        kh, co = divmod(c, co_rows)
        if ci < Ci and co < Co and kh < kH:
            assert np.isnan(dw[co, ci, kh, kw])   # each weight element is produced once
            dw[co, ci, kh, kw] = total[i]
    assert not np.isnan(dw).any()
    return dw


@pytest.mark.parametrize("shape", PLANE_SHAPES)
def test_emulated_wgrad_plane_matches_oracle(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    rng = np.random.default_rng(61)
    go = rng.standard_normal((N, Co, H, W))
    x = rng.standard_normal((N, Ci, H, W))
    for sms in (152, 5):
        emu = emulate_wgrad_plane(go, x, kH, kW, ph, pw, sms)
        ref, mag = oracle.wgrad(go.astype(np.float32), x.astype(np.float32), kH, kW, s, ph, pw)
        assert np.abs(emu - ref).max() <= 1e-5 * max(1.0, mag.max())   # inputs rounded to fp32 for the oracle


def test_wgrad_plane_mode_choice():
    assert dg.wgrad_describe(32, 64, 56, 56, 64, 3, 3, 1, 1, 1)["mode"] == 3
    assert dg.wgrad_describe(32, 64, 56, 56, 64, 3, 3, 1, 1, 1, "tf32x3")["mode"] == 1   # split: the run mode
    assert dg.wgrad_describe(32, 64, 56, 54, 64, 3, 3, 1, 1, 1)["mode"] != 3            # rows of 54 positions
    assert dg.wgrad_describe(2, 8, 8, 8, 8, 3, 3, 2, 1, 1)["mode"] != 3                 # stride 2
    assert dg.wgrad_describe(2, 8, 8, 8, 8, 3, 3, 1, 0, 0)["mode"] != 3                 # oH < H
    assert dg.wgrad_describe(2, 8, 8, 8, 8, 1, 1, 1, 0, 0)["mode"] == 2                 # 1x1: direct
    assert dg.wgrad_describe(2, 256, 8, 8, 64, 3, 3, 1, 1, 1)["mode"] != 3              # 6 x 192 accumulator columns
    assert dg.wgrad_describe(2, 256, 8, 8, 8, 3, 3, 1, 1, 1)["mode"] == 3               # 6 x 32 fit
    d = dg.wgrad_describe(32, 64, 56, 56, 64, 3, 3, 1, 1, 1, sm_count=152)
    assert d["workspace_bytes"] < (24 << 20)   # partial splits only, no frames
    assert d["stages"] >= 3 and d["smem_bytes"] <= 232448 and d["slice_n"] == 192 and d["n_mt"] == 2


RUN_SHAPES = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw: batch-blocked TF32 shapes that run the run mode
    (32, 64, 64, 56, 54, 3, 3, 1, 1, 1),   # the resnet_stage channels on rows of 54 (no plane mode)
    (32, 3, 4, 7, 9, 3, 3, 1, 1, 1),
    (60, 5, 3, 8, 6, 3, 3, 2, 1, 1),
    (64, 40, 20, 6, 5, 3, 3, 1, 1, 1),     # two image groups
    (32, 16, 40, 9, 11, 5, 3, 1, 2, 1),
]


@pytest.mark.parametrize("shape", RUN_SHAPES)
def test_wgrad_run_schedule(shape):
    """Run mode on the CPU: the tap groups against the tap table; each tile's
    tensor copy (L + spt - 1 position blocks from the stage's first chunk on)
    holding, for every chunk of the stage, the spt positions its taps read;
    the copies within the 256-row box limit and shared memory; the units
    covering every (tile, chunk) once; and the reduction's map back to
    (tap, ci) covering each weight row exactly once."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    args = (N, Ci, H, W, Co, kH, kW, s, ph, pw)
    info = dg.wgrad_describe(*args, sm_count=152)
    d = dg.wgrad_describe_run(*args, sm_count=152)
    tab = dg.wgrad_describe_taps(*args)
    assert info["mode"] == 1 and d is not None and info["interleave"] == 32
    spt, sr, L, tpu, bn = d["spt"], d["seg_rows"], d["L"], d["tpu"], info["slice_n"]
    assert spt * sr == 128 and sr >= min(Ci, 128) and info["stages"] >= 2
    assert (L + spt - 1) * sr <= 256 and L * bn <= 256           # tensor-copy boxes of at most 256 rows
    stage = tpu * (L + spt - 1) * sr * 128 + L * bn * 128
    assert info["smem_bytes"] >= info["stages"] * stage and info["smem_bytes"] <= 232448
    assert tpu * bn <= 512 and info["tmem_cols"] <= 512
    seen = []
    for g in d["groups"]:
        for j in range(g["n_taps"]):
            t = d["taps"][g["tap0"] + j]
            assert tab["copy"][t] == g["copy"] and tab["offset"][t] == 32 * (g["base"] + j)
            seen.append(t)
        assert g["n_mt"] == -(-g["n_taps"] // spt)
    assert sorted(seen) == list(range(kH * kW))
    assert d["tiles"] == [(gi, m * spt) for gi, g in enumerate(d["groups"]) for m in range(g["n_mt"])]
    assert d["n_sets"] == -(-d["n_tiles"] // tpu)
    Pg, cps = d["Pg"], d["cps"]
    assert cps % L == 0 and d["nksq"] == -(-Pg // cps)
    assert info["n_units"] == d["Q"] * d["nksq"] * d["cpt"] * d["n_nt"] * d["n_sets"]
    # a tile's copy for the stage starting at chunk c holds positions c + base + m0 + [0, L + spt - 1); chunk
    # c + i reads blocks i .. i + spt - 1 of it, i.e. positions c + i + base + m0 + j for its taps j < spt
    covered = set()
    for ks in range(d["nksq"]):
        c0, c1 = ks * cps, min(ks * cps + cps, Pg)
        for c in range(c0, c1, L):
            for t, (gi, m0) in enumerate(d["tiles"]):
                g = d["groups"][gi]
                copy_pos = [c + g["base"] + m0 + b for b in range(L + spt - 1)]
                for i in range(min(L, c1 - c)):
                    rows = copy_pos[i:i + spt]
                    assert rows == [(c + i) + g["base"] + m0 + j for j in range(spt)]
                    for j in range(spt):
                        if m0 + j < g["n_taps"]:
                            assert rows[j] <= d["Px"] - 1    # a real tap never reads past its image group
                    covered.add((t, c + i))
    assert covered == {(t, c) for t in range(d["n_tiles"]) for c in range(Pg)}
    # the reduction's (tile, row) -> (tap, ci) map: every weight row exactly once
    rows = []
    for cb in range(d["cpt"]):
        for gi, m0 in d["tiles"]:
            g = d["groups"][gi]
            for r in range(128):
                j = m0 + r // sr
                ci = cb * sr + r % sr
                if j < g["n_taps"] and ci < Ci:
                    rows.append((d["taps"][g["tap0"] + j], ci))
    assert sorted(rows) == [(t, ci) for t in range(kH * kW) for ci in range(Ci)]


def test_wgrad_direct_mode_choice():
    pw = WORKLOADS["pointwise"]
    d = dg.wgrad_describe(*pw.plan_args(), sm_count=152)
    assert d["mode"] == 2 and d["workspace_bytes"] < 64 << 20      # partial tiles only, no frames
    assert dg.wgrad_describe(*pw.plan_args(), precision="tf32x3")["mode"] == 0
    assert dg.wgrad_describe(2, 8, 5, 5, 16, 1, 1, 1, 0, 0)["mode"] == 0     # 25 positions: not a multiple of 4
    assert dg.wgrad_describe(2, 8, 8, 8, 16, 1, 1, 2, 0, 0)["mode"] == 0     # stride 2


def test_wgrad_run_mode_choice():
    assert dg.wgrad_describe_run(2, 3, 8, 8, 4, 3, 3, 1, 1, 1) is None            # small batch: segment mode
    assert dg.wgrad_describe(32, 64, 56, 56, 64, 3, 3, 1, 1, 1, "tf32x3")["mode"] == 1  # split precision too
    assert dg.wgrad_describe(32, 64, 56, 54, 64, 3, 3, 1, 1, 1)["mode"] == 1


def test_wgrad_plan_ex_rejects_bad_options():
    """wgrad_plan_ex validates its options before it touches a device: a
    negative wait limit or a wait_test other than 0 or 1 is an argument error,
    and a NULL plan pointer too."""
    import ctypes
    from conv2d_backward_implicit_dgrad_gb300 import binding
    lib = binding.load_library()
    h = ctypes.c_void_p()
    args = (2, 8, 8, 8, 8, 3, 3, 1, 1, 1, 1)
    for timeout_us, wait_test in ((-1, 0), (0, 2), (0, -1)):
        opts = binding.WgradOptions(timeout_us, wait_test)
        h.value = 0x1234   # NULL on failure
        assert lib.wgrad_plan_ex(*args, ctypes.byref(opts), ctypes.byref(h)) == 1
        assert not h.value
    assert lib.wgrad_plan_ex(*args, None, None) == 1


def test_wgrad_plans():
    for name in ORDER:
        wl = WORKLOADS[name]
        d = dg.wgrad_describe(*wl.plan_args(), sm_count=152)
        assert d["oH"] == wl.oH and d["oW"] == wl.oW
        assert d["smem_bytes"] <= 232448 and d["tmem_cols"] <= 512 and 16 <= d["slice_n"] <= 256
        if d["mode"] == 0:    # units: row tiles x column tiles x K splits
            assert d["n_units"] == d["n_mt"] * d["n_nt"] * d["n_ks"]
        else:                 # units: tile sets x ci blocks x column tiles x K splits
            assert d["n_units"] % (d["n_nt"] * d["n_ks"]) == 0
        assert d["grid"] <= 152
        assert d["useful_flops"] == 2 * wl.N * wl.Co * wl.oH * wl.oW * wl.Ci * wl.kH * wl.kW
    for bad, status in (((0, 1, 4, 4, 1, 3, 3, 1, 1, 1), 1), ((1, 1, 2, 2, 1, 5, 5, 1, 0, 0), 1),
                        ((1, 1, 32, 32, 1, 3, 3, 5, 1, 1), 2)):
        with pytest.raises(dg.DgradError) as e:
            dg.wgrad_describe(*bad)
        assert e.value.status == status
    with pytest.raises(dg.DgradError) as e:
        dg.wgrad_describe(2, 3, 8, 8, 4, 3, 3, 1, 1, 1, "fp32")
    assert e.value.status == 2


def test_wgrad_split_plans():
    """Split precision: same tiling, both frames twice, a stage ring of at
    least two (hi | lo) stages within the shared-memory limit."""
    for name in ORDER:
        wl = WORKLOADS[name]
        a = dg.wgrad_describe(*wl.plan_args(), sm_count=152)
        b = dg.wgrad_describe(*wl.plan_args(), precision="tf32x3", sm_count=152)
        assert b["precision"] == "tf32x3" and a["precision"] == "tf32"
        same = ("n_mt", "n_nt", "slice_n", "seg_rows") if a["mode"] == 0 and b["mode"] == 0 else ()
        frames_too = ("Kimg", "Lx", "n_copies") if a["mode"] != 2 else ()   # direct mode has no frames
        for k in same + frames_too + ("useful_flops",):
            assert a[k] == b[k], k
        chunks = -(-wl.N // b["interleave"]) * b["Kimg"] // 32
        assert -(-chunks // b["n_ks"]) <= 12   # short accumulation chains
        if b["mode"] == 0:
            assert b["n_units"] == b["n_mt"] * b["n_nt"] * b["n_ks"]
            stage = 2 * (128 * 128 + b["slice_n"] * 128)
            assert b["smem_bytes"] >= b["stages"] * stage
        assert b["stages"] >= 2 and b["smem_bytes"] <= 232448
        Q = -(-wl.N // b["interleave"])
        frames = 4 * (Q * wl.Co * b["Kimg"] + b["n_copies"] * Q * wl.Ci * b["Lx"])
        assert b["workspace_bytes"] >= 2 * frames                                     # hi and lo halves
        assert a["mode"] in (2, 3) or a["workspace_bytes"] >= frames   # direct and plane modes: no frames


def test_col2im_plans():
    wl = WORKLOADS["stem"]
    d = dg.describe(*wl.plan_args(), path="col2im", sm_count=152)
    assert d["path"] == "col2im" and d["a_source"] == "frame"
    assert d["slice_n"] == 160                      # 3 x 7 x 7 = 147 GEMM columns, padded to 16
    assert d["smem_bytes"] <= 232448 and d["tmem_cols"] <= 512 and d["grid"] <= 152
    assert dg.describe(*wl.plan_args(), sm_count=152)["path"] == "tcgen05"   # never chosen automatically
    for bad in (dict(precision="fp32"), dict(precision="tf32x3")):
        with pytest.raises(dg.DgradError) as e:
            dg.describe(*wl.plan_args(), path="col2im", **bad)
        assert e.value.status == 2


def test_ffma_source_plans():
    # FFMA path: the frame pipeline automatically where every phase has at most
    # 4 taps (the band fill is then a large share of a chunk's work) or where
    # it runs 8 x 8 register tiles (64-channel slices), the CTA's own gather
    # elsewhere; either on request; no staged or tensor-memory source.
    expect = {"tiny": "producers", "resnet_stage": "frame", "strided_downsample": "frame",
              "pointwise": "frame", "stem": "producers"}
    for name, src in expect.items():
        wl = WORKLOADS[name]
        d = dg.describe(*wl.plan_args(), "fp32")
        assert d["path"] == "simt" and d["a_source"] == src, name
        f = dg.describe(*wl.plan_args(), "fp32", a_source="frame")
        assert f["a_source"] == "frame"
        # one persistent CTA per SM, or two (8 x 8 tiles for 64-channel slices,
        # each CTA then within half of the SM's 228 KB less its reserved 1 KB)
        two = f["slice_n"] == 64
        assert f["grid"] == min(f["n_work"], 152 * (2 if two else 1)) and 2 <= f["a_stages"] <= 6
        assert f["smem_bytes"] <= 232448
        # the band: 128 rows plus the largest tap shift, in copies of at most 256 rows
        assert f["a_rows"] >= 128 + f["max_shift"] and f["a_rows"] % 8 == 0
        g = dg.describe(*wl.plan_args(), "fp32", a_source="producers")
        assert g["a_source"] == "producers" and g["grid"] == g["n_work"]
        for bad in ("staged", "tmem"):
            with pytest.raises(dg.DgradError) as e:
                dg.describe(*wl.plan_args(), "fp32", a_source=bad)
            assert e.value.status == 2


def test_ffma_four_channel_slices_plans():
    # At most 4 input channels: 4-channel slices (1024-position units) in the
    # gather kernel where those units fill a wave of CTAs; 16 otherwise, and
    # always in the frame pipeline.
    stem = WORKLOADS["stem"].plan_args()
    d = dg.describe(*stem, "fp32")
    assert d["slice_n"] == 4 and d["tile_step"] == 1024 and d["a_source"] == "producers"
    assert d["n_work"] == -(-d["positions"] // 1024) * d["n_phases"]
    assert dg.describe(*stem, "fp32", a_source="frame")["slice_n"] == 16
    assert dg.describe(*WORKLOADS["tiny"].plan_args(), "fp32")["slice_n"] == 16
    assert dg.describe(4, 3, 200, 200, 8, 3, 3, 1, 1, 1, "fp32")["slice_n"] == 4
    assert dg.describe(4, 5, 200, 200, 8, 3, 3, 1, 1, 1, "fp32")["slice_n"] == 16
    assert dg.describe(*stem, "fp32", slice_n=16)["slice_n"] == 16
