"""Parity of the fused projection (tensor cores, tcgen05) with the oracle.

cat_project and cat_forward_fused compute V = X·W_V and the scores X·W_A in
one pass over X (the two projections of a CAT layer, notes page section
整体框架), then — for cat_forward_fused — the forward on that V.  Bounds:
  V  : bf16 rounding of an fp32-accumulated sum of exact products,
       |V - V_ref| <= 2^-8·|V_ref| + 1e-6·max|V_ref|;
  z* : 1e-5 relative elementwise (the forward's bound), peaked case
       included;
  O  : the forward's bf16 bound 8e-3·max|V| against the oracle's O on the
       oracle's V; and against cat_forward on the V the projection wrote
       (the kernels after the scores are the same and the scores agree to
       rounding, so the two differ by at most a bf16 rounding step).
"""
import numpy as np
import pytest
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth
from _gpu_helpers import check_zstar, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _built(cuda_device):
    from fft_circulant_attention_gb300 import build
    build.build()
    yield


CASES = [
    # (B, N, D, H, wa_scale)
    (1, 256, 64, 2, 1.0),           # one value tile of 64 columns
    (3, 100, 128, 2, 1.0),          # ragged token tiles (300 tokens)
    (2, 196, 320, 5, 1.0),          # value tiles of 256 + 64 columns
    (4, 1024, 768, 12, 1.0),        # GPT-2 small width, three value tiles
    (4, 1024, 768, 12, 8.0),        # peaked scores
    (1, 16384, 1024, 16, 1.0),      # the long-sequence fast path
    (2, 512, 128, 16, 1.0),         # 16 heads: no padding of the score tile
]


def _inputs(B, N, D, H, wa, seed):
    X, WA, _ = synth.make_inputs(B, N, D, H, "bf16", seed=seed, wa_scale=wa)
    WV = synth.make_wv(D, "bf16", seed=seed)
    return X, WV, WA


@pytest.mark.parametrize("B,N,D,H,wa", CASES)
def test_project_parity(B, N, D, H, wa):
    X, WV, WA = _inputs(B, N, D, H, wa, seed=N + D)
    Xd, WVd, WAd = to_dev(X, WV, WA)
    with cat.Plan(B, N, D, H, "bf16") as p:
        V, zs = p.project(Xd, WVd, WAd)
        p.sync()
    V_ref = oracle.project(X, WV)
    Vg = V.double().cpu().numpy()
    bound = 2.0 ** -8 * np.abs(V_ref) + 1e-6 * np.abs(V_ref).max()
    assert (np.abs(Vg - V_ref) <= bound).all(), float(np.abs(Vg - V_ref).max())
    errZ = check_zstar(zs.cpu(), oracle.zstar(X, WA))
    print("project B=%d N=%d D=%d H=%d: max rel dz* = %.2e" % (B, N, D, H, errZ))


@pytest.mark.parametrize("B,N,D,H,wa", CASES)
def test_forward_fused_parity(B, N, D, H, wa):
    X, WV, WA = _inputs(B, N, D, H, wa, seed=N + 7)
    Xd, WVd, WAd = to_dev(X, WV, WA)
    with cat.Plan(B, N, D, H, "bf16") as p:
        V, O = p.forward_fused(Xd, WVd, WAd)
        O_plain = p.forward(Xd, WAd, V)
        p.sync()
    vmax = float(V.float().abs().max())
    assert torch.allclose(O.float(), O_plain.float(), rtol=2.0 ** -7, atol=1e-6 * vmax)
    V_ref = oracle.project(X, WV)
    zs_ref = oracle.zstar(X, WA)
    if N <= 4096:
        rows = list(range(N))
        O_ref = oracle.circ_direct(zs_ref, V_ref) if B * N * N * D <= 2e9 else \
            oracle.circ_fft(zs_ref, V_ref)
    else:
        rows = list(range(0, N, 64))
        O_ref = oracle.circ_direct_rows(zs_ref, V_ref, rows)
    err = float(np.abs(O.double().cpu().numpy()[:, rows] - O_ref[:, :len(rows)] if N > 4096
                       else O.double().cpu().numpy() - O_ref).max())
    assert err <= 8e-3 * float(np.abs(V_ref).max()), err


def test_fused_rejects_unsupported():
    X = torch.zeros(1, 64, 96, dtype=torch.bfloat16, device="cuda:0")
    W = torch.zeros(96, 96, dtype=torch.bfloat16, device="cuda:0")
    A = torch.zeros(96, 2, dtype=torch.bfloat16, device="cuda:0")
    with cat.Plan(1, 64, 96, 2, "bf16") as p:          # D not a multiple of 64
        with pytest.raises(cat.CatError) as e:
            p.forward_fused(X, W, A)
        assert e.value.status == cat.CAT_ERR_INVALID_ARG
    Xf = torch.zeros(1, 64, 64, device="cuda:0")
    with cat.Plan(1, 64, 64, 2, "f32") as p:            # fp32 storage
        with pytest.raises(cat.CatError) as e:
            cat.cat_forward_fused(p.handle, Xf, Xf, Xf, Xf, Xf, 1, 64, 64, 2, "f32")
        assert e.value.status == cat.CAT_ERR_INVALID_ARG
    X = torch.zeros(1, 64, 64, dtype=torch.bfloat16, device="cuda:0")
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda:0")
    A = torch.zeros(64, 2, dtype=torch.bfloat16, device="cuda:0")
    with cat.Plan(1, 64, 64, 2, "bf16") as p:          # V aliasing X
        with pytest.raises(cat.CatError) as e:
            p.forward_fused(X, W, A, V=X)
        assert e.value.status == cat.CAT_ERR_ALIAS
