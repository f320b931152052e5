"""The FMA-pipe exp2: its polynomial is the committed fit (re-run here, on the
CPU) and, on the GPU, the device routine stays within the fit's error bound
against fp64 exp2 over the softmax's range, as ex2.approx does within its
own."""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_online_gb300", "csrc")


def load_fit():
    spec = importlib.util.spec_from_file_location("fit_exp2_poly",
                                                  os.path.join(CSRC, "fit_exp2_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def header_constants():
    txt = open(os.path.join(CSRC, "exp2_poly.h")).read()
    coef = [float(v) for _, v in sorted(re.findall(r"kExp2C(\d) = ([-0-9.e+]+)f", txt))]
    err = float(re.search(r"kExp2PolyMaxRelErr = ([-0-9.e+]+)f", txt).group(1))
    return np.array(coef, dtype=np.float32), err


def test_header_is_the_committed_fit():
    fit = load_fit()
    c32, err = fit.fit(fit.DEG)
    hc, herr = header_constants()
    assert np.array_equal(hc, c32)
    assert abs(herr - err) <= 1e-9
    assert err < 1e-4           # a cubic on [-1/2, 1/2]


def test_fit_equioscillates():
    """Minimax: the relative error reaches its maximum with alternating signs
    at degree + 2 points (checked on the fp64 coefficients)."""
    fit = load_fit()
    c = fit.remez(3)
    x = np.linspace(-0.5, 0.5, 200001)
    e = np.polyval(c[::-1], x) / np.exp2(x) - 1.0
    m = np.abs(e).max()
    peaks = np.flatnonzero(np.abs(e) >= 0.999 * m)
    signs = np.sign(e[peaks])
    changes = np.count_nonzero(np.diff(signs))
    assert changes >= 4, (m, changes)


@pytest.mark.gpu
def test_device_exp2_within_bound():
    import torch
    import exact_attention_online_gb300 as fa
    _, err = header_constants()
    # results in the normal range (the softmax's p lies in (0, 256]; below
    # 2^-125 both routines leave the normal range: ex2.approx.ftz flushes)
    x = torch.cat([torch.linspace(-125.0, 8.0, 1 << 20), torch.tensor([0.0, -0.5, 0.5, 1.0, -1.0]),
                   torch.rand(1 << 16) * 16 - 8]).float().cuda()
    y_fma, y_ex2 = torch.empty_like(x), torch.empty_like(x)
    fa.fa_exp2_check(x, y_fma, y_ex2)
    torch.cuda.synchronize()
    ref = np.exp2(x.double().cpu().numpy())
    rel_fma = np.abs(y_fma.double().cpu().numpy() / ref - 1.0)
    rel_ex2 = np.abs(y_ex2.double().cpu().numpy() / ref - 1.0)
    # the fit's bound, plus the fp32 rounding of x * 1 (x is exact) and of the
    # final scale (exact: a power of two)
    assert rel_fma.max() <= err * 1.0001 + 2.0 ** -23, rel_fma.max()
    assert rel_ex2.max() <= 2.0 ** -20, rel_ex2.max()
    # masked scores (-inf) come out below the normal range: zero for the softmax
    m = torch.tensor([-float("inf"), -1000.0], device="cuda")
    yf, ye = torch.empty_like(m), torch.empty_like(m)
    fa.fa_exp2_check(m, yf, ye)
    torch.cuda.synchronize()
    assert (yf.abs() < 2.0 ** -125).all()


@pytest.mark.gpu
def test_device_ex2_rate_chains_reach_the_fixed_point():
    """fa_ex2_rate iterates x <- 2^(-x), a contraction (|slope| = ln 2 * 2^-x
    <= 0.6 on [1/2, 1]) whose fixed point x* solves x = 2^-x; after 64 rounds
    each thread's sum of its eight chains is 8 x* to within the exponential's
    error, and no lane is left unwritten."""
    import torch
    import exact_attention_online_gb300 as fa
    xs = 0.5
    for _ in range(200):
        xs = 2.0 ** -xs
    assert abs(xs - 2.0 ** -xs) < 1e-15
    blocks = 12
    out = torch.full((blocks * 256,), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_ex2_rate(out, blocks, 64)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - 8.0 * xs).max() <= 1e-4, np.abs(got - 8.0 * xs).max()
