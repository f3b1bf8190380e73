"""Parity of the direct ("gather") circulant product with the fp64 oracle.

The direct path evaluates O[b, i, c] = sum_j z*[(i - j) mod N] · V[b, j, c]
term by term (the gather-based O(N²) evaluation the CAT notes page reports in
section 局限与展望, limitations), with the scores either from the score kernel
or computed inside the product kernel (fused, one launch).  CAT_FORCE_PATH=
direct sends every supported shape down it; each case is compared element by
element with the oracle under the forward's bounds (O: 2e-5·max|V| fp32,
8e-3·max|V| bf16; z*: 1e-5 relative), and the backward's dV — which reruns the
plan's product kernel on dO with the scores reversed — with the oracle's
chain rule.
"""
import numpy as np
import pytest
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth
from _gpu_helpers import check_out, check_zstar, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _direct(cuda_device, monkeypatch):
    from fft_circulant_attention_gb300 import build
    build.build()
    monkeypatch.setenv("CAT_FORCE_PATH", "direct")
    yield


CASES = [
    # (B, N, D, H, dtype, wa_scale)
    (1, 256, 64, 2, "f32", 1.0),        # the smallest workload (fused scores)
    (64, 196, 384, 6, "f32", 1.0),      # ViT 14x14 patches
    (16, 1024, 768, 12, "f32", 1.0),    # GPT-2 small
    (16, 1024, 768, 12, "bf16", 1.0),
    (16, 1024, 768, 12, "f32", 8.0),    # peaked softmax
    (4, 64, 384, 6, "f32", 1.0),
    (3, 100, 48, 3, "bf16", 1.0),       # ragged row tiles, head width 16
    (2, 1000, 128, 1, "f32", 1.0),      # head width 128
    (5, 7, 8, 2, "f32", 1.0),           # head width 4, N < one row tile
    (2, 1, 16, 4, "bf16", 1.0),         # N = 1
    (1, 343, 96, 3, "f32", 1.0),        # 7^3, head width 32
]


# Every case with the plan's own choice, the scores forced separate ("0")
# and forced fused ("1"); the fused kernel serves small N·D only, so the
# forced-fused variant runs where N·D <= 2^17.
PARITY_CASES = [c + (f,) for c in CASES for f in ("auto", "0", "1")
                if f != "1" or c[1] * c[2] <= (1 << 17)]


@pytest.mark.parametrize("B,N,D,H,dtype,wa,fused", PARITY_CASES)
def test_direct_parity(B, N, D, H, dtype, wa, fused, monkeypatch):
    if fused != "auto":
        monkeypatch.setenv("CAT_DIRECT_FUSED", fused)
    with cat.Plan(B, N, D, H, dtype) as p:
        assert "path=direct" in p.describe(), p.describe()
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=N + D + H, wa_scale=wa)
    O, zs = run_gpu(X, WA, V, dtype)
    mode = "direct" if B * N * N * D <= 2e9 else "fft"
    O_ref, zs_ref = oracle.forward(X, WA, V, mode=mode)
    errO = check_out(O, O_ref, V, dtype)
    errZ = check_zstar(zs, zs_ref)
    print("direct B=%d N=%d D=%d H=%d %s: max|dO|/max|V| = %.2e, max rel dz* = %.2e"
          % (B, N, D, H, dtype, errO, errZ))


def test_direct_matches_transform_path(monkeypatch):
    """The direct product and the register FFT path agree on the same inputs
    within the fp32 output bound."""
    B, N, D, H = 8, 256, 256, 4
    X, WA, V = to_dev(*synth.make_inputs(B, N, D, H, "f32", seed=3))
    with cat.Plan(B, N, D, H, "f32") as p:
        O_dir = p.forward(X, WA, V)
        p.sync()
    monkeypatch.setenv("CAT_FORCE_PATH", "smem")
    with cat.Plan(B, N, D, H, "f32") as p:
        assert "path=smem" in p.describe()
        O_fft = p.forward(X, WA, V)
        p.sync()
    assert float((O_dir - O_fft).abs().max()) <= 2e-5 * float(V.abs().max())


def test_direct_bit_identical_repeats():
    B, N, D, H = 4, 196, 384, 6
    X, WA, V = to_dev(*synth.make_inputs(B, N, D, H, "f32", seed=9))
    with cat.Plan(B, N, D, H, "f32") as p:
        O0 = p.forward(X, WA, V)
        for _ in range(5):
            O1 = p.forward(X, WA, V)
            assert torch.equal(O0, O1)
        p.sync()


@pytest.mark.parametrize("B,N,D,H,dtype", [(1, 256, 64, 2, "f32"), (4, 196, 384, 6, "f32"),
                                           (2, 1024, 768, 12, "bf16")])
def test_direct_backward_dv(B, N, D, H, dtype):
    """dV = circ(z*)^T dO through the direct kernel (scores reversed)."""
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=5)
    G = synth.make_grad(B, N, D, dtype, seed=5)
    Xd, Wd, Vd, Gd = to_dev(X, WA, V, G)
    with cat.Plan(B, N, D, H, dtype) as p:
        assert "path=direct" in p.describe()
        dX, dWA, dV = p.backward(Xd, Wd, Vd, Gd)
        p.sync()
    ref = oracle.backward(X, WA, V, G, mode="direct" if B * N * N * D <= 2e9 else "fft")
    gmax = float(np.abs(G.double().numpy()).max())
    tol = (8e-3 if dtype == "bf16" else 2e-5) * gmax
    assert float(np.abs(dV.double().cpu().numpy() - ref["dV"]).max()) <= tol
    # The score-side gradients do not touch the product kernel; a loose
    # check that the plan's workspace use is consistent.
    dwa_ref = ref["dWA"]
    assert float(np.abs(dWA.double().cpu().numpy() - dwa_ref).max()) <= \
        (5e-5 + (2.0 ** -8 if dtype == "bf16" else 0)) * float(np.abs(dwa_ref).max()) * 4


def test_direct_empty_batch():
    X = torch.empty(0, 196, 384, device="cuda:0")
    WA = torch.randn(384, 6, device="cuda:0")
    with cat.Plan(0, 196, 384, 6, "f32") as p:
        O = p.forward(X, WA, X)
        p.sync()
    assert O.shape == (0, 196, 384)
