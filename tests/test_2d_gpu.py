"""Parity of the CUDA 2-D circulant attention (cat2d_*, through the C ABI)
with the fp64 oracle (oracle.forward2d: the BCCB product of the page "Vision
Transformers are Circulant Attention Learners", O = σ(a) ⊛ V, with the
reading a = channel-averaged 2-D circular cross-correlation of Q and K;
pinned in test_oracle_2d_pins.py).

Bounds (fp32 arithmetic):
  a : 1e-5·max|a| per (b, h) row — an FFT correlation, as dz* in the
      backward;
  O : (2·tol(a) + 2e-5)·max|V| (fp32 storage), with 8e-3 in place of 2e-5
      for bf16 — the softmax turns an absolute score error e into a relative
      weight error of at most 2e, and the circulant product itself is held
      to the forward's bound.
"""
import numpy as np
import pytest
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth
from _gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

A_TOL = 1e-5
O_TOL = {"f32": 2e-5, "bf16": 8e-3}


@pytest.fixture(autouse=True)
def _needs_gpu(cuda_device):
    from fft_circulant_attention_gb300 import build
    build.build()
    yield


def run2d(B, h, w, D, H, dtype, seed=0):
    N = h * w
    Q, K, V = synth.make_qkv(B, N, D, dtype, seed)
    Qd, Kd, Vd = to_dev(Q, K, V)
    with cat.Plan2D(B, h, w, D, H, dtype) as plan:
        O = plan.forward(Qd, Kd, Vd)
        a = plan.scores(Qd, Kd)
        plan.sync()
        desc = plan.describe()
    torch.cuda.synchronize()
    return (Q, K, V), O.cpu(), a.cpu(), desc


def check2d(B, h, w, D, H, dtype, seed=0):
    (Q, K, V), O, a, desc = run2d(B, h, w, D, H, dtype, seed)
    O_ref, a_ref, _ = oracle.forward2d(Q, K, V, H, h, w)
    tol_a = A_TOL * np.abs(a_ref).max(axis=-1, keepdims=True)
    err_a = np.abs(a.double().numpy() - a_ref)
    assert (err_a <= tol_a).all(), "a error %.3e" % float((err_a / tol_a).max())
    vmax = float(np.abs(V.double().numpy()).max())
    bound = (2 * float(tol_a.max()) + O_TOL[dtype]) * vmax
    err = float(np.abs(O.double().numpy() - O_ref).max())
    assert err <= bound, "O error %.3e > %.3e" % (err, bound)
    return err / vmax, desc


@pytest.mark.parametrize("B,h,w,D,H,dtype", [
    (1, 14, 14, 64, 2, "f32"),
    (2, 7, 12, 16, 2, "f32"),
    (1, 1, 9, 8, 2, "f32"),
    (1, 9, 1, 8, 2, "f32"),
    (1, 12, 10, 9, 3, "f32"),
    (1, 16, 16, 32, 1, "bf16"),
    (2, 5, 4, 4, 2, "bf16"),
])
def test_grid_shapes(B, h, w, D, H, dtype):
    err, desc = check2d(B, h, w, D, H, dtype, seed=h * w)
    print("B%d %dx%d D%d H%d %s: max|dO|/max|V| = %.2e [%s]" % (B, h, w, D, H, dtype, err, desc))


# Square grids of side 8, 14, 16 or 32 take the register kernels (the 2-D
# DFT as the register transform's two steps without the twiddle); both paths
# are held to the oracle, and to each other.
@pytest.mark.parametrize("B,side,D,H,dtype", [
    (2, 8, 64, 1, "f32"),
    (3, 14, 96, 2, "f32"),
    (2, 14, 30, 2, "bf16"),        # head width 15: a half pair
    (1, 16, 64, 4, "f32"),
    (1, 32, 128, 2, "f32"),
    (2, 32, 64, 2, "bf16"),
    (4, 14, 384, 6, "f32"),        # ViT-S widths
])
@pytest.mark.parametrize("reg", ["1", "0"])
def test_square_grids_register_and_generic(B, side, D, H, dtype, reg, monkeypatch):
    monkeypatch.setenv("CAT_2D_REG", reg)
    err, desc = check2d(B, side, side, D, H, dtype, seed=side + D)
    assert ("reg2d=1" in desc) == (reg == "1"), desc
    print("B%d %dx%d D%d H%d %s reg=%s: max|dO|/max|V| = %.2e" % (B, side, side, D, H, dtype,
                                                                  reg, err))


def test_register_and_generic_2d_agree(monkeypatch):
    B, side, D, H = 2, 14, 384, 6
    Q, K, V = to_dev(*synth.make_qkv(B, side * side, D, "f32", 4))
    outs = []
    for reg in ("1", "0"):
        monkeypatch.setenv("CAT_2D_REG", reg)
        with cat.Plan2D(B, side, side, D, H, "f32") as plan:
            outs.append((plan.forward(Q, K, V), plan.scores(Q, K)))
            plan.sync()
    (O1, a1), (O0, a0) = outs
    assert float((a1 - a0).abs().max()) <= 2e-5 * float(a0.abs().max())
    assert float((O1 - O0).abs().max()) <= 4e-5 * float(V.abs().max())


# Square grids of side 64, 96 or 128 take the row/column passes (length-M
# DFTs as a register DFT-32 and a DFT-M/32 in shared memory, five passes over
# grid rows and columns); both they and the generic passes are held to the
# oracle.  The 128 x 128 case at head width 64 needs two chunks of (b, h)
# rows, and head width 5 leaves a half pair.
@pytest.mark.parametrize("B,side,D,H,dtype", [
    (1, 64, 64, 2, "f32"),
    (2, 64, 15, 3, "f32"),         # head width 5: a half pair
    (1, 96, 96, 2, "bf16"),
    (1, 128, 48, 2, "f32"),
    (1, 128, 384, 6, "bf16"),      # two chunks of (b, h) rows
])
@pytest.mark.parametrize("gp", ["1", "0"])
def test_square_grids_row_column_passes(B, side, D, H, dtype, gp, monkeypatch):
    monkeypatch.setenv("CAT_2D_REG", gp)
    err, desc = check2d(B, side, side, D, H, dtype, seed=side + D)
    assert ("gp=1" in desc) == (gp == "1"), desc
    if gp == "1" and side == 128 and D == 384:
        assert "launches=10" in desc, desc
    print("B%d %dx%d D%d H%d %s gp=%s: max|dO|/max|V| = %.2e" % (B, side, side, D, H, dtype,
                                                                 gp, err))


def test_row_column_passes_and_generic_2d_agree(monkeypatch):
    B, side, D, H = 1, 96, 384, 6
    Q, K, V = to_dev(*synth.make_qkv(B, side * side, D, "f32", 5))
    outs = []
    for gp in ("1", "0"):
        monkeypatch.setenv("CAT_2D_REG", gp)
        with cat.Plan2D(B, side, side, D, H, "f32") as plan:
            outs.append((plan.forward(Q, K, V), plan.scores(Q, K)))
            plan.sync()
    (O1, a1), (O0, a0) = outs
    assert float((a1 - a0).abs().max()) <= 2e-5 * float(a0.abs().max())
    assert float((O1 - O0).abs().max()) <= 4e-5 * float(V.abs().max())


@pytest.mark.parametrize("name", list(synth.GRID_CONFIGS))
def test_grid_workloads(name):
    c = synth.GRID_CONFIGS[name]
    err, _ = check2d(c["B"], c["h"], c["w"], c["D"], c["H"], c["dtype"])
    print("%s: max|dO|/max|V| = %.2e" % (name, err))


def test_one_row_grid_matches_cat_product_of_the_same_weights():
    """A 1 x N grid's product is the 1-D circulant product: with K = 0 the
    scores vanish, σ(a) is uniform and O is the column mean of V."""
    B, h, w, D, H = 1, 1, 64, 8, 2
    Q, K, V = synth.make_qkv(B, h * w, D, "f32", 1)
    K = torch.zeros_like(K)
    Qd, Kd, Vd = to_dev(Q, K, V)
    with cat.Plan2D(B, h, w, D, H, "f32") as plan:
        O = plan.forward(Qd, Kd, Vd).cpu()
        plan.sync()
    ref = V.double().mean(dim=1, keepdim=True).expand_as(V)
    assert float((O.double() - ref).abs().max()) <= 2e-5 * float(V.abs().max())


def test_plan_kinds_do_not_mix():
    B, h, w, D, H = 1, 4, 4, 8, 2
    Q, K, V = to_dev(*synth.make_qkv(B, h * w, D, "f32"))
    O = torch.empty_like(V)
    L = cat.lib()
    p = lambda t: t.data_ptr()
    with cat.Plan2D(B, h, w, D, H, "f32") as p2, cat.Plan(B, h * w, D, H, "f32") as p1:
        assert L.cat_forward(p2.handle, p(Q), p(K), p(V), p(O), B, h * w, D, H, 0) == \
            cat.CAT_ERR_PLAN_MISMATCH
        assert L.cat2d_forward(p1.handle, p(Q), p(K), p(V), p(O), B, h, w, D, H, 0) == \
            cat.CAT_ERR_PLAN_MISMATCH
        assert L.cat2d_forward(p2.handle, p(Q), p(K), p(V), p(O), B, 2, 8, D, H, 0) == \
            cat.CAT_ERR_PLAN_MISMATCH
        assert L.cat2d_forward(p2.handle, p(Q), p(K), p(V), p(V), B, h, w, D, H, 0) == \
            cat.CAT_ERR_ALIAS
        assert L.cat2d_forward(p2.handle, p(Q), p(K), p(V), p(O), B, h, w, D, H, 0) == cat.CAT_OK
        p2.sync()
        p1.sync()
