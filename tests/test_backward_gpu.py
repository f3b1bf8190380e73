"""Parity of the CUDA backward pass (through the C ABI) with the fp64 oracle.

Each case draws seeded inputs (synth.make_inputs) and an upstream gradient
dO (synth.make_grad), runs cat_backward and cat_backward_dz on cuda:0 and
compares element by element with oracle.backward — the chain rule through
the definitions of the CAT notes page, section 方法详解, pinned in
test_oracle_backward_pins.py.

Bounds (all arithmetic fp32; derived from the forward's bounds and from an
fp32 emulation of the same steps, whose errors they exceed tenfold or more):
  dV   : 2e-5·max|dO| (fp32 storage) or 8e-3·max|dO| (bf16) — the same
         circulant product as the forward, with dO in place of V;
  dz*  : 1e-5·max_k|dz*[b, h, k]| per (b, h) row (an FFT correlation of
         length N: the emulation stays below 3e-7);
  dz   : z*[n]·(2·tol(dz*) + 1e-5·|dz*[n] - <z*, dz*>|) elementwise — the
         softmax Jacobian applied to dz* and z* within their bounds;
  dW_A : 5e-5·max|dW_A|;  dX : 2e-5·max|dX| (fp32 sums of dz products);
  bf16 gradients also carry their round-to-nearest-even error, 2^-8·|ref|.
"""
import numpy as np
import pytest
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth
from _gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

DV_TOL = {"f32": 2e-5, "bf16": 8e-3}
DZS_TOL = 1e-5
Z_REL = 1e-5
DWA_TOL = 5e-5
DX_TOL = 2e-5
BF16_U = 2.0 ** -8


@pytest.fixture(autouse=True)
def _needs_gpu(cuda_device):
    from fft_circulant_attention_gb300 import build
    build.build()
    yield


def _np(t):
    return t.double().numpy() if hasattr(t, "double") else np.asarray(t, np.float64)


def run_bw(X, WA, V, G, dtype):
    """cat_backward and cat_backward_dz on cuda:0; CPU tensors back."""
    B, N, D = V.shape
    H = WA.shape[1]
    Xd, Wd, Vd, Gd = to_dev(X, WA, V, G)
    with cat.Plan(B, N, D, H, dtype) as plan:
        dX, dWA, dV = plan.backward(Xd, Wd, Vd, Gd)
        dzs, dz = plan.backward_dz(Xd, Wd, Vd, Gd)
        plan.sync()
        desc = plan.describe()
    torch.cuda.synchronize()
    return dict(dX=dX.cpu(), dWA=dWA.cpu(), dV=dV.cpu(), dzs=dzs.cpu(), dz=dz.cpu(), desc=desc)


def _grad_bound(ref, rel, dtype):
    tol = rel * np.abs(ref).max()
    if dtype == "bf16":
        return (1 + BF16_U) * tol + BF16_U * np.abs(ref)
    return tol


def check_dzs(got, ref):
    tol = DZS_TOL * np.abs(ref).max(axis=-1, keepdims=True)
    err = np.abs(_np(got) - ref)
    assert (err <= tol).all(), "dz* error %.3e > bound %.3e" % (
        float((err / np.maximum(tol, 1e-300)).max()), DZS_TOL)
    return tol


def check_dz(got, ref, zs_ref, dzs_ref, tol_dzs):
    s = np.sum(zs_ref * dzs_ref, axis=-1, keepdims=True)
    tol = zs_ref * (2 * tol_dzs + Z_REL * np.abs(dzs_ref - s))
    err = np.abs(_np(got) - ref)
    assert (err <= tol + 1e-300).all(), "dz error %.3e x bound" % float((err / (tol + 1e-300)).max())


def check_all(got, ref, G, dtype, dx_rows=None, dv_rows=None):
    """Compare every gradient; dv_rows / dx_rows restrict dV / dX to sampled
    rows (ref then holds only those rows)."""
    gmax = float(np.abs(_np(G)).max())
    dV = _np(got["dV"]) if dv_rows is None else _np(got["dV"])[:, dv_rows]
    errV = float(np.abs(dV - ref["dV"]).max())
    assert errV <= DV_TOL[dtype] * gmax, "dV error %.3e > %.3e" % (errV, DV_TOL[dtype] * gmax)
    tol_dzs = check_dzs(got["dzs"], ref["dzs"])
    check_dz(got["dz"], ref["dz"], ref["zs"], ref["dzs"], tol_dzs)
    errW = np.abs(_np(got["dWA"]) - ref["dWA"])
    assert (errW <= _grad_bound(ref["dWA"], DWA_TOL, dtype)).all(), \
        "dW_A error %.3e (max|ref| %.3e)" % (errW.max(), np.abs(ref["dWA"]).max())
    dX = _np(got["dX"]) if dx_rows is None else _np(got["dX"])[:, dx_rows]
    errX = np.abs(dX - ref["dX"])
    assert (errX <= _grad_bound(ref["dX"], DX_TOL, dtype)).all(), \
        "dX error %.3e (max|ref| %.3e)" % (errX.max(), np.abs(ref["dX"]).max())
    return errV / gmax


def parity_bw(B, N, D, H, dtype, seed=0, wa_scale=1.0, mode="auto"):
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=seed, wa_scale=wa_scale)
    G = synth.make_grad(B, N, D, dtype, seed=seed)
    got = run_bw(X, WA, V, G, dtype)
    ref = oracle.backward(X, WA, V, G, mode=mode)
    err = check_all(got, ref, G, dtype)
    return err, got["desc"]


# Shapes covering every forward path the dV product takes (block FFT,
# square-length register kernel, generic four-step, fast four-step with
# N2 = 32 and 64) and both correlation layouts (whole rows up to 4096,
# four-step split above), odd head widths, prime and tiny N, and both
# kernels of the dense gradients (FP32, tensor cores).
SHAPES = [
    (1, 1, 4, 2, "f32"),
    (1, 2, 4, 1, "f32"),
    (2, 7, 6, 3, "f32"),
    (1, 10, 9, 3, "f32"),
    (2, 64, 16, 2, "f32"),
    (1, 64, 16, 2, "bf16"),
    (1, 196, 24, 2, "f32"),
    (1, 256, 64, 2, "f32"),
    (2, 1000, 10, 2, "f32"),
    (1, 1024, 32, 1, "bf16"),
    (1, 4096, 8, 2, "f32"),
    (1, 6000, 8, 2, "f32"),
    (1, 16384, 8, 2, "f32"),
    (1, 20000, 4, 2, "f32"),
    (1, 16384, 128, 2, "bf16"),
    (1, 32768, 64, 1, "f32"),
    # bf16 with D a multiple of 64 (the tensor-core dW_A and dX): a column
    # group past D, an odd head count, token tiles across batch rows and a
    # ragged last tile.
    (3, 1000, 192, 3, "bf16"),
    (2, 4096, 320, 5, "bf16"),
    # The fast path's correlation chunks with dV from their own transform of
    # dO: chunks of 3 rows in half slots (6 heads), and 10 heads in chunks of
    # 4 with a last chunk of 2.
    (1, 16384, 384, 6, "bf16"),
    (1, 16384, 640, 10, "bf16"),
]


@pytest.mark.parametrize("B,N,D,H,dtype", SHAPES)
def test_backward_shapes(B, N, D, H, dtype):
    err, desc = parity_bw(B, N, D, H, dtype, seed=N % 97)
    print("B%d N%d D%d H%d %s: max|ddV|/max|dO| = %.2e  [%s]" % (B, N, D, H, dtype, err, desc))


WORKLOADS = {
    "tiny": dict(B=1, N=256, D=64, H=2, dtype="f32"),
    "vit196": dict(B=64, N=196, D=384, H=6, dtype="f32"),
    "gpt2_f32": dict(B=16, N=1024, D=768, H=12, dtype="f32"),
    "gpt2_bf16": dict(B=16, N=1024, D=768, H=12, dtype="bf16"),
    "gpt2_peaked": dict(B=16, N=1024, D=768, H=12, dtype="f32", wa_scale=8.0),
}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_backward_workloads(name):
    err, _ = parity_bw(**WORKLOADS[name])
    print("%s: max|ddV|/max|dO| = %.2e" % (name, err))


@pytest.mark.parametrize("name,nrows", [("long16k", 24), ("long128k", 8)])
def test_backward_long_sampled(name, nrows):
    """Full-size long-sequence workloads: dz*, dz and dW_A in full (the
    oracle's FFT correlation), dV and dX at sampled rows (the O(N) per-row
    definition; dX from the oracle's dz)."""
    c = synth.CONFIGS[name]
    B, N, D, H, dtype = c["B"], c["N"], c["D"], c["H"], c["dtype"]
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=0)
    G = synth.make_grad(B, N, D, dtype, seed=0)
    got = run_bw(X, WA, V, G, dtype)
    rng = np.random.default_rng(3)
    rows = sorted({0, 1, N // 2, N - 1} | {int(r) for r in rng.choice(N, nrows, replace=False)})
    zs = oracle.zstar(X, WA)
    dzs = oracle.corr_fft(G, V, H)
    dz = oracle.softmax_backward(zs, dzs)
    ref = dict(zs=zs, dzs=dzs, dz=dz, dWA=oracle.grad_wa(X, dz),
               dX=oracle.grad_x(np.ascontiguousarray(dz[:, :, rows]), WA),
               dV=oracle.circ_transpose_direct_rows(zs, G, rows))
    err = check_all(got, ref, G, dtype, dx_rows=rows, dv_rows=rows)
    print("%s: max|ddV|/max|dO| = %.2e over %d rows" % (name, err, len(rows)))


def test_backward_adjoint_on_device():
    """<CAT(X, W_A, V), dO> = <V, dV> with both sides from the CUDA path (a
    property of the pair forward/backward that holds at any size)."""
    B, N, D, H = 2, 16384, 128, 2
    X, WA, V = synth.make_inputs(B, N, D, H, "f32", seed=4)
    G = synth.make_grad(B, N, D, "f32", seed=4)
    Xd, Wd, Vd, Gd = to_dev(X, WA, V, G)
    with cat.Plan(B, N, D, H, "f32") as plan:
        O = plan.forward(Xd, Wd, Vd)
        _, _, dV = plan.backward(Xd, Wd, Vd, Gd)
        plan.sync()
    lhs = float((O.double() * Gd.double()).sum())
    rhs = float((Vd.double() * dV.double()).sum())
    scale = float((O.double() * Gd.double()).abs().sum())
    assert abs(lhs - rhs) <= 1e-5 * scale


def test_backward_repeatable_and_forward_unaffected():
    """Two backward calls give bit-identical gradients, and a forward after a
    backward (which reverses the plan's scores) is the same as before it."""
    B, N, D, H, dtype = 1, 16384, 128, 2, "bf16"
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=6)
    G = synth.make_grad(B, N, D, dtype, seed=6)
    Xd, Wd, Vd, Gd = to_dev(X, WA, V, G)
    with cat.Plan(B, N, D, H, dtype) as plan:
        O1 = plan.forward(Xd, Wd, Vd).clone()
        a = [t.clone() for t in plan.backward(Xd, Wd, Vd, Gd)]
        b = [t.clone() for t in plan.backward(Xd, Wd, Vd, Gd)]
        O2 = plan.forward(Xd, Wd, Vd).clone()
        plan.sync()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(O1, O2)


def test_backward_graph_follows_pointers(monkeypatch):
    """The fast path replays its backward as a CUDA graph while the call's
    pointers stay the same and re-captures it when they change: new output
    buffers, then new inputs, give exactly what the schedule launched
    directly (CAT_GRAPH=0) gives."""
    B, N, D, H, dtype = 1, 16384, 128, 2, "bf16"
    ins = []
    for seed in (7, 8):
        X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=seed)
        G = synth.make_grad(B, N, D, dtype, seed=seed)
        ins.append(to_dev(X, WA, V, G))
    ref = []
    monkeypatch.setenv("CAT_GRAPH", "0")
    with cat.Plan(B, N, D, H, dtype) as plan:
        assert "graph=0" in plan.describe()
        for args in ins:
            ref.append([t.clone() for t in plan.backward(*args)])
        plan.sync()
    monkeypatch.delenv("CAT_GRAPH")
    with cat.Plan(B, N, D, H, dtype) as plan:
        assert "graph=1" in plan.describe()
        first = [t.clone() for t in plan.backward(*ins[0])]           # capture
        again = [t.clone() for t in plan.backward(*ins[0])]           # new outputs: update
        outs = plan.backward(*ins[1])                                  # new inputs and outputs
        other = [t.clone() for t in outs]
        replay = [t.clone() for t in plan.backward(*ins[1], *outs)]   # same pointers: replay
        plan.sync()
        assert "graph=1" in plan.describe()
    for got in (first, again):
        for x, y in zip(got, ref[0]):
            assert torch.equal(x, y)
    for got in (other, replay):
        for x, y in zip(got, ref[1]):
            assert torch.equal(x, y)


def test_backward_argument_errors():
    B, N, D, H = 1, 64, 16, 2
    X, WA, V = to_dev(*synth.make_inputs(B, N, D, H, "f32"))
    G = to_dev(synth.make_grad(B, N, D, "f32"))[0]
    with cat.Plan(B, N, D, H, "f32") as plan:
        h = plan.handle
        dX, dWA, dV = torch.empty_like(X), torch.empty_like(WA), torch.empty_like(V)
        L = cat.lib()
        p = lambda t: t.data_ptr()
        args = (B, N, D, H, cat.CAT_F32)
        assert L.cat_backward(h, p(X), p(WA), p(V), p(G), p(dX), p(dWA), p(dV), *args) == cat.CAT_OK
        # output aliasing an input, or another output
        assert L.cat_backward(h, p(X), p(WA), p(V), p(G), p(G), p(dWA), p(dV), *args) == cat.CAT_ERR_ALIAS
        assert L.cat_backward(h, p(X), p(WA), p(V), p(G), p(dX), p(dWA), p(dX), *args) == cat.CAT_ERR_ALIAS
        # misaligned, null, wrong shape
        assert L.cat_backward(h, p(X) + 4, p(WA), p(V), p(G), p(dX), p(dWA), p(dV), *args) == \
            cat.CAT_ERR_MISALIGNED
        assert L.cat_backward(h, p(X), p(WA), p(V), None, p(dX), p(dWA), p(dV), *args) == \
            cat.CAT_ERR_INVALID_ARG
        assert L.cat_backward(h, p(X), p(WA), p(V), p(G), p(dX), p(dWA), p(dV), B, N, D, H,
                              cat.CAT_BF16) == cat.CAT_ERR_PLAN_MISMATCH
        plan.sync()


def test_backward_empty_batch():
    with cat.Plan(0, 64, 16, 2, "f32") as plan:
        e = torch.empty((0, 64, 16), device="cuda:0")
        w = torch.zeros((16, 2), device="cuda:0")
        assert cat.lib().cat_backward(plan.handle, e.data_ptr(), w.data_ptr(), e.data_ptr(),
                                      e.data_ptr(), e.data_ptr(), w.data_ptr(), e.data_ptr(),
                                      0, 64, 16, 2, cat.CAT_F32) == cat.CAT_OK
        plan.sync()


@pytest.mark.parametrize("B,N,D,H,dtype", [(2, 64, 32, 2, "f32"), (4, 196, 384, 6, "f32"),
                                           (1, 256, 64, 2, "f32"), (2, 1024, 768, 12, "bf16"),
                                           (3, 196, 30, 2, "bf16"), (1, 1024, 75, 5, "f32")])
def test_register_correlation_matches_block_passes(B, N, D, H, dtype, monkeypatch):
    """For N = M² the correlation dz* runs in the register kernel (at
    N = 1024 split over 4 CTAs a row, their partial spectra added, inverted
    and turned into dz by a finishing kernel; head width 15 leaves three of
    the four CTAs without pairs); it agrees with the block-FFT passes
    (CAT_BW_REG=0) and the oracle within the dz* and dz bounds."""
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=N + 3)
    G = synth.make_grad(B, N, D, dtype, seed=N + 3)
    Xd, Wd, Vd, Gd = to_dev(X, WA, V, G)
    got = {}
    for reg in ("1", "0"):
        monkeypatch.setenv("CAT_BW_REG", reg)
        with cat.Plan(B, N, D, H, dtype) as plan:
            dzs, dz = plan.backward_dz(Xd, Wd, Vd, Gd)
            plan.sync()
        got[reg] = (dzs.double().cpu().numpy(), dz.double().cpu().numpy())
    full = oracle.backward(X, WA, V, G, mode="direct" if B * N * N * D <= 2e9 else "fft")
    ref = full["dzs"]
    tol = DZS_TOL * np.abs(ref).max(axis=-1, keepdims=True)
    for reg in ("1", "0"):
        assert (np.abs(got[reg][0] - ref) <= tol).all(), reg
        check_dz(got[reg][1], full["dz"], full["zs"], ref, tol)
