"""Pins for the CPU oracle (CPU only).

Each check ties the oracle to something other than itself: hand-worked
fixtures, the forward convolution it is the adjoint of (brute force on unit
vectors, inner-product identity, finite differences), the stride-1
transposed-padding identity, closed forms (delta response, 1x1 = matmul, the
sum identity), torch's fp64 CPU convolution routines, and the pages' two other
formulations (doppler's gather, meganeura's GEMM index map, the phase split).
``test_mutants_are_caught`` plants plausible mistakes in a copy of the oracle
and checks that these pins reject each one.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_dgrad_gb300.workloads import ORDER, WORKLOADS, make_inputs, make_tensors

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def out_ext(n, k, s, p):
    return (n + 2 * p - k) // s + 1


def rand_case(N, Ci, Co, H, W, kH, kW, s, ph, pw, seed=0, dist="uniform"):
    oH, oW = out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)
    go, w = make_tensors((N, Co, oH, oW), (Co, Ci, kH, kW), seed, dist)
    return go.numpy(), w.numpy()


def rel_err(a, b):
    den = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() / den


# Small shapes that exercise stride, both paddings, rectangular kernels and
# inputs, kernels larger than the stride, strides larger than the kernel and
# rows that no term reaches.
SMALL = [
    # N, Ci, Co, H, W, kH, kW, s, ph, pw
    (1, 1, 1, 3, 3, 2, 2, 1, 0, 0),
    (2, 3, 4, 5, 5, 3, 3, 1, 1, 1),
    (1, 2, 3, 6, 5, 3, 3, 2, 1, 1),
    (1, 2, 2, 6, 6, 3, 3, 1, 0, 0),
    (2, 2, 3, 5, 6, 3, 2, 1, 2, 0),
    (1, 3, 2, 6, 6, 5, 5, 1, 1, 1),
    (1, 2, 2, 5, 5, 3, 3, 3, 1, 1),
    (1, 2, 3, 5, 4, 1, 1, 2, 0, 0),
    (1, 2, 2, 6, 6, 2, 2, 2, 0, 0),
    (2, 1, 2, 6, 6, 3, 3, 2, 0, 0),
    (1, 2, 2, 6, 5, 4, 3, 2, 1, 2),
    (1, 1, 2, 2, 2, 3, 3, 2, 1, 1),
]


# --------------------------------------------------------------------------- fixtures
def load_fixture(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    N, Ci, H, W, Co, kH, kW, s, ph, pw = (int(x) for x in vals["shape"])
    oH, oW = out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)
    go = np.array(vals["grad_out"], np.float32).reshape(N, Co, oH, oW)
    w = np.array(vals["weight"], np.float32).reshape(Co, Ci, kH, kW)
    gi = np.array(vals["grad_input"]).reshape(N, Ci, H, W)
    mag = np.array(vals["mag"]).reshape(N, Ci, H, W)
    p1 = np.array(vals["p1_gemm"]).reshape(N, Ci, H, W) if "p1_gemm" in vals else None
    return (H, W, s, ph, pw), go, w, gi, mag, p1


FIXTURES = sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt"))


@pytest.mark.parametrize("name", FIXTURES)
def test_golden_fixture(name):
    (H, W, s, ph, pw), go, w, gi, mag, p1 = load_fixture(os.path.join(GOLDEN, name))
    acc, m = oracle.dgrad(go, w, H, W, s, ph, pw)
    np.testing.assert_array_equal(acc, gi)
    np.testing.assert_array_equal(m, mag)
    np.testing.assert_array_equal(oracle.dgrad_gather(go, w, H, W, s, ph, pw), gi)
    np.testing.assert_array_equal(oracle.dgrad_phase(go, w, H, W, s, ph, pw), gi)
    idx = np.array([(n, c, y, x) for n in range(gi.shape[0]) for c in range(gi.shape[1])
                    for y in range(H) for x in range(W)])
    a, m2 = oracle.dgrad_at(go, w, H, W, s, ph, pw, idx)
    np.testing.assert_array_equal(a, gi.reshape(-1))
    np.testing.assert_array_equal(m2, mag.reshape(-1))
    if p1 is not None:
        np.testing.assert_array_equal(oracle.dgrad_gemm_p1(go, w, H, W, s, ph, pw), p1)


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("shape", SMALL)
def test_bruteforce_adjoint_matrix(shape):
    """dgrad = A^T g exactly, with A the forward-conv matrix built column by column
    from unit vectors."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=3)
    n_in = Ci * H * W
    oH, oW = go.shape[2], go.shape[3]
    A = np.zeros((Co * oH * oW, n_in))
    for i in range(n_in):
        e = np.zeros((1, Ci, H, W))
        e.reshape(-1)[i] = 1.0
        A[:, i] = oracle.conv2d_fwd(e, w.astype(np.float64), s, ph, pw).reshape(-1)
    acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    for n in range(N):
        ref = A.T @ go[n].astype(np.float64).reshape(-1)
        assert rel_err(acc[n].reshape(-1), ref) < 1e-12


@pytest.mark.parametrize("shape", SMALL)
def test_fwd_matches_torch(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    rng = np.random.default_rng(5)
    x = rng.standard_normal((N, Ci, H, W))
    w = rng.standard_normal((Co, Ci, kH, kW))
    y = oracle.conv2d_fwd(x, w, s, ph, pw)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w), stride=s,
                                     padding=(ph, pw)).numpy()
    assert y.shape == ref.shape
    assert rel_err(y, ref) < 1e-12


@pytest.mark.parametrize("shape", SMALL)
def test_dgrad_matches_torch(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=7)
    acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    ref = torch.nn.grad.conv2d_input((N, Ci, H, W), torch.from_numpy(w).double(),
                                     torch.from_numpy(go).double(), stride=s,
                                     padding=(ph, pw)).numpy()
    assert rel_err(acc, ref) < 1e-12


# --------------------------------------------------------------------------- identities
@pytest.mark.parametrize("name", ORDER)
def test_adjoint_identity_workloads(name):
    """<conv2d(x, w), g> = <x, dgrad(g, w)> in fp64 at each workload's shape
    (batch cut to 2 images to keep the CPU suite short)."""
    wl = WORKLOADS[name]
    N = min(wl.N, 2)
    go, w = make_tensors((N, wl.Co, wl.oH, wl.oW), wl.w_shape, 11, wl.dist)
    x = torch.randn((N, wl.Ci, wl.H, wl.W), generator=torch.Generator().manual_seed(12),
                    dtype=torch.float32).numpy()
    y = oracle.conv2d_fwd(x, w.numpy(), wl.stride, wl.pad_h, wl.pad_w)
    acc, _ = oracle.dgrad(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    lhs = float(np.dot(y.reshape(-1), go.numpy().astype(np.float64).reshape(-1)))
    rhs = float(np.dot(x.astype(np.float64).reshape(-1), acc.reshape(-1)))
    scale = float(np.abs(y).reshape(-1) @ np.abs(go.numpy().astype(np.float64)).reshape(-1))
    assert abs(lhs - rhs) <= 1e-12 * scale


@pytest.mark.parametrize("shape", SMALL[:8])
def test_finite_differences(shape):
    """L(x) = <conv2d(x, w), g> is linear in x, so a central difference with step 1
    equals dL/dx = dgrad(g, w) up to fp64 rounding."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=13)
    rng = np.random.default_rng(14)
    x = rng.standard_normal((N, Ci, H, W))
    g64, w64 = go.astype(np.float64), w.astype(np.float64)
    acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)

    def L(xx):
        return float(np.sum(oracle.conv2d_fwd(xx, w64, s, ph, pw) * g64))

    flat = rng.choice(x.size, size=min(12, x.size), replace=False)
    for i in flat:
        xp, xm = x.copy(), x.copy()
        xp.reshape(-1)[i] += 1.0
        xm.reshape(-1)[i] -= 1.0
        fd = (L(xp) - L(xm)) / 2.0
        assert abs(fd - acc.reshape(-1)[i]) <= 1e-10 * (1 + abs(acc.reshape(-1)[i]))


@pytest.mark.parametrize("kH,kW,ph,pw", [(3, 3, 1, 1), (3, 3, 0, 0), (3, 3, 2, 2), (5, 3, 1, 2),
                                         (2, 2, 1, 0), (1, 1, 0, 0), (4, 2, 3, 1)])
def test_transposed_padding_identity(kH, kW, ph, pw):
    """Stride 1, pad <= k-1: dgrad(g, w, p) equals the forward conv of g padded by
    (k-1-p) with the kernel rotated 180 degrees and its channel axes swapped."""
    N, Ci, Co, H, W = 2, 3, 4, 6, 5
    go, w = rand_case(N, Ci, Co, H, W, kH, kW, 1, ph, pw, seed=17)
    acc, _ = oracle.dgrad(go, w, H, W, 1, ph, pw)
    w_rot = np.ascontiguousarray(w[:, :, ::-1, ::-1].transpose(1, 0, 2, 3)).astype(np.float64)
    y = oracle.conv2d_fwd(go.astype(np.float64), w_rot, 1, kH - 1 - ph, kW - 1 - pw)
    assert y.shape == acc.shape
    assert rel_err(acc, y) < 1e-12


# --------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("shape", [(1, 2, 3, 7, 6, 3, 3, 2, 1, 1), (1, 3, 2, 6, 6, 5, 3, 1, 2, 1),
                                   (2, 2, 2, 9, 9, 7, 7, 2, 3, 3)])
def test_delta_response(shape):
    """A single 1 at go[n,co,oh,ow] gives w[co,ci,kh,kw] at (oh*s - ph + kh, ow*s - pw + kw)."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    oH, oW = out_ext(H, kH, s, ph), out_ext(W, kW, s, pw)
    _, w = rand_case(*shape, seed=19)
    for (n, co, oh, ow) in [(0, 0, 0, 0), (N - 1, Co - 1, oH - 1, oW - 1), (0, Co // 2, oH // 2, oW - 1)]:
        go = np.zeros((N, Co, oH, oW), np.float32)
        go[n, co, oh, ow] = 1.0
        acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
        exp = np.zeros((N, Ci, H, W))
        for ci in range(Ci):
            for kh in range(kH):
                for kw in range(kW):
                    ih, iw = oh * s - ph + kh, ow * s - pw + kw
                    if 0 <= ih < H and 0 <= iw < W:
                        exp[n, ci, ih, iw] = w[co, ci, kh, kw]
        np.testing.assert_array_equal(acc, exp)


def test_pointwise_is_matmul():
    """1x1 kernel, stride 1, no padding: gi[n] = W^T G[n] with G[n] = go[n] as [Co, H*W]."""
    go, w = rand_case(3, 5, 7, 4, 6, 1, 1, 1, 0, 0, seed=23)
    acc, _ = oracle.dgrad(go, w, 4, 6, 1, 0, 0)
    W2 = w[:, :, 0, 0].astype(np.float64)              # [Co, Ci]
    for n in range(3):
        ref = W2.T @ go[n].astype(np.float64).reshape(7, -1)
        assert rel_err(acc[n].reshape(5, -1), ref) < 1e-13


@pytest.mark.parametrize("shape", [(2, 3, 4, 7, 7, 3, 3, 2, 0, 0), (1, 2, 3, 6, 8, 2, 3, 1, 0, 0),
                                   (1, 2, 2, 9, 9, 3, 3, 3, 0, 0)])
def test_sum_identity_no_padding(shape):
    """With no padding every tap lands inside, so
    sum_{ih,iw} gi[n,ci] = sum_co (sum_{kh,kw} w[co,ci]) * (sum_{oh,ow} go[n,co])."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=29)
    acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    lhs = acc.sum(axis=(2, 3))
    rhs = go.astype(np.float64).sum(axis=(2, 3)) @ w.astype(np.float64).sum(axis=(2, 3))
    assert rel_err(lhs, rhs) < 1e-12


def test_linearity():
    shape = (2, 3, 4, 7, 6, 3, 3, 2, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    g1, w1 = rand_case(*shape, seed=31)
    g2, w2 = rand_case(*shape, seed=32)
    a1, _ = oracle.dgrad(g1, w1, H, W, s, ph, pw)
    a2, _ = oracle.dgrad(g2, w1, H, W, s, ph, pw)
    a12, _ = oracle.dgrad(g1 + g2, w1, H, W, s, ph, pw)
    # g1 + g2 is rounded to fp32 on the way in; compare against that exact sum.
    gsum = (g1 + g2).astype(np.float32)
    assert rel_err(a12, oracle.dgrad(gsum, w1, H, W, s, ph, pw)[0]) == 0
    assert rel_err(a12, a1 + a2) < 1e-6
    b1, _ = oracle.dgrad(g1, w2, H, W, s, ph, pw)
    bh, _ = oracle.dgrad(g1, (0.5 * w2).astype(np.float32), H, W, s, ph, pw)
    np.testing.assert_array_equal(bh, 0.5 * b1)


def test_mag_invariants():
    shape = (2, 3, 4, 7, 6, 3, 3, 2, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=37)
    acc, mag = oracle.dgrad(go, w, H, W, s, ph, pw)
    assert np.all(mag >= np.abs(acc))
    abs_acc, _ = oracle.dgrad(np.abs(go), np.abs(w), H, W, s, ph, pw)
    np.testing.assert_allclose(mag, abs_acc, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------- cross-formulations
@pytest.mark.parametrize("shape", SMALL)
def test_gather_and_phase_match_scatter(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=41)
    acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    assert rel_err(oracle.dgrad_gather(go, w, H, W, s, ph, pw), acc) < 1e-13
    assert rel_err(oracle.dgrad_phase(go, w, H, W, s, ph, pw), acc) < 1e-13


@pytest.mark.parametrize("shape", SMALL)
def test_p1_gemm_agrees_only_for_same_padding(shape):
    """meganeura's map matches the definition for strides > 1 and for 'same'
    stride-1 padding (2*pad = k-1); elsewhere its stride-1 shortcut differs."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=43)
    acc, _ = oracle.dgrad(go, w, H, W, s, ph, pw)
    p1 = oracle.dgrad_gemm_p1(go, w, H, W, s, ph, pw)
    same = (2 * ph == kH - 1) and (2 * pw == kW - 1)
    if s > 1 or same:
        assert rel_err(p1, acc) < 1e-13
    else:
        assert rel_err(p1, acc) > 1e-3


@pytest.mark.parametrize("name", ORDER)
def test_sampled_matches_scatter(name):
    wl = WORKLOADS[name]
    N = min(wl.N, 2)
    go, w = make_tensors((N, wl.Co, wl.oH, wl.oW), wl.w_shape, 47, wl.dist)
    acc, mag = oracle.dgrad(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    rng = np.random.default_rng(48)
    idx = np.stack([rng.integers(0, N, 200), rng.integers(0, wl.Ci, 200),
                    rng.integers(0, wl.H, 200), rng.integers(0, wl.W, 200)], 1)
    a, m = oracle.dgrad_at(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w, idx)
    ref = acc[idx[:, 0], idx[:, 1], idx[:, 2], idx[:, 3]]
    refm = mag[idx[:, 0], idx[:, 1], idx[:, 2], idx[:, 3]]
    assert rel_err(a, ref) < 1e-12
    assert rel_err(m, refm) < 1e-12


def test_tiny_workload_full():
    go, w = make_inputs("tiny", 0)
    wl = WORKLOADS["tiny"]
    acc, _ = oracle.dgrad(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    ref = torch.nn.grad.conv2d_input(wl.gi_shape, w.double(), go.double(), stride=1, padding=1).numpy()
    assert rel_err(acc, ref) < 1e-13


def test_threads_do_not_change_result():
    shape = (5, 3, 4, 9, 8, 3, 3, 2, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, w = rand_case(*shape, seed=53)
    a1, m1 = oracle.dgrad(go, w, H, W, s, ph, pw, nthreads=1)
    a4, m4 = oracle.dgrad(go, w, H, W, s, ph, pw, nthreads=4)
    np.testing.assert_array_equal(a1, a4)
    np.testing.assert_array_equal(m1, m4)


def test_rejects_bad_shapes():
    go = np.zeros((1, 1, 1, 1), np.float32)
    w = np.zeros((1, 1, 5, 5), np.float32)
    assert oracle.out_extent(3, 5, 1, 0) == 0
    with pytest.raises(ValueError):
        oracle.dgrad(go, w, 3, 3, 1, 0, 0)


# --------------------------------------------------------------------------- mutants
MUTANTS = [
    ("wrong sign of the padding offset",
     "int ih = oh * sh->s - sh->ph + kh;", "int ih = oh * sh->s + sh->ph - kh;"),
    ("kernel flipped",
     "double t = g * (double)j->w[w_at(sh, co, ci, kh, kw)];",
     "double t = g * (double)j->w[w_at(sh, co, ci, sh->kH - 1 - kh, sh->kW - 1 - kw)];"),
    ("column 0 dropped",
     "if (iw < 0 || iw >= sh->W) continue;\n                                double t",
     "if (iw <= 0 || iw >= sh->W) continue;\n                                double t"),
    ("row padding used for columns",
     "int iw = ow * sh->s - sh->pw + kw;", "int iw = ow * sh->s - sh->ph + kw;"),
    ("overwrite instead of accumulate", "j->acc[o] += t;", "j->acc[o] = t;"),
    ("stride ignored on rows", "int ih = oh * sh->s - sh->ph + kh;", "int ih = oh - sh->ph + kh;"),
    ("channel axes transposed in the weight index (square channel counts only)",
     "double t = g * (double)j->w[w_at(sh, co, ci, kh, kw)];",
     "double t = g * (double)j->w[w_at(sh, ci, co, kh, kw)];"),
]


def _scatter_from(lib, go, w, H, W, s, ph, pw):
    N, Co, oH, oW = go.shape
    _, Ci, kH, kW = w.shape
    acc = np.empty((N, Ci, H, W))
    mag = np.empty_like(acc)
    p = ctypes.c_void_p
    lib.oracle_dgrad_scatter.argtypes = [ctypes.c_int] * 10 + [p, p, p, p, ctypes.c_int]
    rc = lib.oracle_dgrad_scatter(N, Ci, H, W, Co, kH, kW, s, ph, pw,
                                  go.ctypes.data_as(p), w.ctypes.data_as(p),
                                  acc.ctypes.data_as(p), mag.ctypes.data_as(p), 1)
    assert rc == 0
    return acc


def _pins_pass(lib):
    """The pins above, restricted to what a mutated scatter changes."""
    for name in FIXTURES:
        (H, W, s, ph, pw), go, w, gi, mag, _ = load_fixture(os.path.join(GOLDEN, name))
        if not np.array_equal(_scatter_from(lib, go, w, H, W, s, ph, pw), gi):
            return False
    for shape in SMALL + [(1, 3, 3, 5, 6, 3, 3, 1, 1, 1)]:
        N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
        go, w = rand_case(*shape, seed=59)
        ref = torch.nn.grad.conv2d_input((N, Ci, H, W), torch.from_numpy(w).double(),
                                         torch.from_numpy(go).double(), stride=s,
                                         padding=(ph, pw)).numpy()
        if rel_err(_scatter_from(lib, go, w, H, W, s, ph, pw), ref) > 1e-12:
            return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_mutants_are_caught(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "dgrad_oracle.c")).read()
    assert _pins_pass(ctypes.CDLL(oracle.build()))
    for label, old, new in MUTANTS:
        assert src.count(old) >= 1, label
        mut = src.replace(old, new, 1)
        c = tmp_path / "mut.c"
        so = tmp_path / f"mut_{MUTANTS.index((label, old, new))}.so"
        c.write_text(mut)
        subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-pthread", str(c), "-o", str(so), "-lm"])
        assert not _pins_pass(ctypes.CDLL(str(so))), f"mutant survived: {label}"



# ----------------------------------------------------------------- fused epilogue composition
def test_fused_oracle_special_cases():
    """relu_backward (ferrotensor kernels.wgsl section 12) and gradient
    accumulation (section 20) composed with O1, pinned by special cases."""
    rng = np.random.default_rng(5)
    N, Ci, Co, H, W, k, s, p = 2, 3, 4, 7, 6, 3, 2, 1
    oH, oW = oracle.out_extent(H, k, s, p), oracle.out_extent(W, k, s, p)
    go = rng.standard_normal((N, Co, oH, oW)).astype(np.float32)
    w = rng.standard_normal((Co, Ci, k, k)).astype(np.float32)
    ref, mag = oracle.dgrad(go, w, H, W, s, p, p)
    pos = np.full((N, Ci, H, W), 0.5, np.float32)
    a, m = oracle.dgrad_fused(go, w, H, W, s, p, p, relu_in=pos)
    assert np.array_equal(a, ref) and np.array_equal(m, mag)            # every input > 0: the plain dgrad
    nonpos = np.zeros((N, Ci, H, W), np.float32)
    nonpos[0, 0, 0, 0] = -1.0
    nonpos[1, 2, 3, 4] = np.nan                                        # NaN is not > 0
    a, m = oracle.dgrad_fused(go, w, H, W, s, p, p, relu_in=nonpos)
    assert not a.any() and not m.any()                                  # 0 and negatives block everything
    gi0 = rng.standard_normal((N, Ci, H, W)).astype(np.float32)
    a, _ = oracle.dgrad_fused(go, w, H, W, s, p, p, grad_in=gi0)
    np.testing.assert_allclose(a - gi0.astype(np.float64), ref, rtol=0, atol=1e-12)   # accumulate = add the stored gradient
    a, _ = oracle.dgrad_fused(go, np.zeros_like(w), H, W, s, p, p, grad_in=gi0)
    assert np.array_equal(a, gi0.astype(np.float64))                   # nothing to add
    mix = rng.standard_normal((N, Ci, H, W)).astype(np.float32)
    a, _ = oracle.dgrad_fused(go, w, H, W, s, p, p, relu_in=mix, grad_in=gi0)
    expect = gi0.astype(np.float64) + np.where(mix > 0, ref, 0.0)
    assert np.array_equal(a, expect)
    # the mask applies to the new gradient only, not to what is accumulated into
    assert (a[mix <= 0] == gi0[mix <= 0]).all()


# ----------------------------------------------------------------- O-w: the weight gradient
def wgrad_case(shape, seed):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, _ = rand_case(*shape, seed=seed)
    x = np.random.default_rng(seed + 1).uniform(-1, 1, (N, Ci, H, W)).astype(np.float32)
    return go, x


@pytest.mark.parametrize("shape", SMALL)
def test_wgrad_brute_force(shape):
    """dW[e] = <conv2d(x, unit weight e), g> for every weight element e: the
    gradient of the linear map w -> <conv2d(x, w), g>, built element by element."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, x = wgrad_case(shape, 40)
    acc, mag = oracle.wgrad(go, x, kH, kW, s, ph, pw)
    g64, x64 = go.astype(np.float64), x.astype(np.float64)
    ref = np.zeros((Co, Ci, kH, kW))
    for e in range(ref.size):
        w = np.zeros(ref.size)
        w[e] = 1.0
        y = oracle.conv2d_fwd(x64, w.reshape(ref.shape), s, ph, pw)
        ref.reshape(-1)[e] = float(np.dot(y.reshape(-1), g64.reshape(-1)))
    assert np.abs(acc - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    assert np.all(mag >= np.abs(acc) - 1e-12)


@pytest.mark.parametrize("shape", SMALL)
def test_wgrad_matches_torch_conv2d_weight(shape):
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, x = wgrad_case(shape, 41)
    acc, _ = oracle.wgrad(go, x, kH, kW, s, ph, pw)
    ref = torch.nn.grad.conv2d_weight(torch.from_numpy(x).double(), (Co, Ci, kH, kW),
                                      torch.from_numpy(go).double(), stride=s, padding=(ph, pw)).numpy()
    assert rel_err(acc, ref) <= 1e-12


@pytest.mark.parametrize("name", ORDER)
def test_wgrad_dgrad_cross_adjoint(name):
    """<dgrad(g, w), x> = <g, conv2d(x, w)> = <w, wgrad(x, g)>: O-w against O1 and
    O-fwd at each workload's shape (batch cut to 2 images)."""
    wl = WORKLOADS[name]
    N = min(wl.N, 2)
    go, w = make_tensors((N, wl.Co, wl.oH, wl.oW), wl.w_shape, 42, wl.dist)
    go, w = go.numpy(), w.numpy()
    x = np.random.default_rng(43).standard_normal((N, wl.Ci, wl.H, wl.W)).astype(np.float32)
    dw, _ = oracle.wgrad(go, x, wl.kH, wl.kW, wl.stride, wl.pad_h, wl.pad_w)
    gi, _ = oracle.dgrad(go, w, wl.H, wl.W, wl.stride, wl.pad_h, wl.pad_w)
    y = oracle.conv2d_fwd(x, w, wl.stride, wl.pad_h, wl.pad_w)
    a = float(np.dot(w.astype(np.float64).reshape(-1), dw.reshape(-1)))
    b = float(np.dot(gi.reshape(-1), x.astype(np.float64).reshape(-1)))
    c = float(np.dot(go.astype(np.float64).reshape(-1), y.reshape(-1)))
    scale = float(np.abs(go.astype(np.float64)).reshape(-1) @ np.abs(y).reshape(-1)) + 1.0
    assert abs(a - c) <= 1e-11 * scale and abs(b - c) <= 1e-11 * scale


def test_wgrad_pointwise_is_a_matmul():
    """1x1 kernel, stride 1, no padding: dW[co, ci] = sum_n G_n X_n^T."""
    rng = np.random.default_rng(44)
    go = rng.standard_normal((3, 5, 4, 6)).astype(np.float32)
    x = rng.standard_normal((3, 7, 4, 6)).astype(np.float32)
    acc, _ = oracle.wgrad(go, x, 1, 1, 1, 0, 0)
    ref = sum(go[n].reshape(5, -1).astype(np.float64) @ x[n].reshape(7, -1).astype(np.float64).T for n in range(3))
    assert np.abs(acc[:, :, 0, 0] - ref).max() <= 1e-12 * np.abs(ref).max()


@pytest.mark.parametrize("shape", [(2, 3, 4, 7, 6, 3, 3, 2, 1, 1), (1, 2, 3, 6, 6, 3, 2, 1, 2, 0)])
def test_wgrad_delta_input(shape):
    """x = one unit value at (n0, ci0, ih0, iw0): dW[co, ci0, kh, kw] = go[n0, co, oh, ow]
    where oh*s - ph + kh = ih0 and ow*s - pw + kw = iw0 (0 when no such oh, ow); other
    input channels get 0."""
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, _ = wgrad_case(shape, 45)
    oH, oW = go.shape[2:]
    n0, ci0, ih0, iw0 = N - 1, Ci - 1, H // 2, W // 2
    x = np.zeros((N, Ci, H, W), np.float32)
    x[n0, ci0, ih0, iw0] = 1.0
    acc, _ = oracle.wgrad(go, x, kH, kW, s, ph, pw)
    ref = np.zeros_like(acc)
    for kh in range(kH):
        for kw in range(kW):
            nh, nw = ih0 + ph - kh, iw0 + pw - kw
            if nh % s or nw % s:
                continue
            oh, ow = nh // s, nw // s
            if 0 <= oh < oH and 0 <= ow < oW:
                ref[:, ci0, kh, kw] = go[n0, :, oh, ow]
    assert np.array_equal(acc, ref)


def test_wgrad_magnitude_and_linearity():
    shape = (2, 3, 4, 7, 6, 3, 3, 2, 1, 1)
    N, Ci, Co, H, W, kH, kW, s, ph, pw = shape
    go, x = wgrad_case(shape, 46)
    acc, mag = oracle.wgrad(go, x, kH, kW, s, ph, pw)
    mabs, _ = oracle.wgrad(np.abs(go), np.abs(x), kH, kW, s, ph, pw)
    assert np.abs(mag - mabs).max() <= 1e-12 * mabs.max()
    a2, _ = oracle.wgrad(go, 2 * x, kH, kW, s, ph, pw)   # exact: scaling by 2 is exact in fp32 and fp64
    assert np.array_equal(a2, 2 * acc)
    neg, _ = oracle.wgrad(-go, x, kH, kW, s, ph, pw)
    assert np.array_equal(neg, -acc)
