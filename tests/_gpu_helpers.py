"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on seeded inputs and compare with the fp64 oracle under the stated
tolerances."""
import numpy as np
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth

# Tolerances on the output, as fractions of max|V| over the whole tensor:
# fp32 storage 2e-5, bf16 storage 8e-3 (fp32 arithmetic in both cases).
# z*: elementwise relative error 1e-5; entries whose oracle value is below
# 1e-30 are held to an absolute 1e-5·max z* instead.
O_TOL = {"f32": 2e-5, "bf16": 8e-3}
Z_TOL = 1e-5
Z_TINY = 1e-30


def to_dev(*ts):
    return [t.to("cuda:0").contiguous() for t in ts]


def run_gpu(X, WA, V, dtype, want_zstar=True):
    """CAT forward on cuda:0 through libcat; returns (O, z*) as CPU tensors."""
    B, N, D = V.shape
    H = WA.shape[1]
    Xd, Wd, Vd = to_dev(X, WA, V)
    with cat.Plan(B, N, D, H, dtype) as plan:
        O = plan.forward(Xd, Wd, Vd)
        zs = plan.zstar(Xd, Wd) if want_zstar else None
        plan.sync()
    torch.cuda.synchronize()
    return O.cpu(), (zs.cpu() if zs is not None else None)


def check_zstar(zs_gpu, zs_ref):
    g = zs_gpu.double().numpy() if hasattr(zs_gpu, "numpy") else zs_gpu
    ref = np.asarray(zs_ref)
    big = ref >= Z_TINY
    rel = np.abs(g[big] - ref[big]) / ref[big]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= Z_TOL, "z* relative error %.3e > %.1e" % (worst, Z_TOL)
    if (~big).any():
        ab = float(np.abs(g[~big] - ref[~big]).max())
        assert ab <= Z_TOL * ref.max(), "tiny z* abs error %.3e" % ab
    return worst


def check_out(O_gpu, O_ref, V, dtype):
    vmax = float(np.abs(V.double().numpy()).max())
    err = float(np.abs(O_gpu.double().numpy() - O_ref).max())
    bound = O_TOL[dtype] * vmax
    assert err <= bound, "max|O - O_ref| = %.3e > %.3e" % (err, bound)
    return err / vmax


def parity(B, N, D, H, dtype, seed=0, wa_scale=1.0, mode="auto"):
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=seed, wa_scale=wa_scale)
    O, zs = run_gpu(X, WA, V, dtype)
    O_ref, zs_ref = oracle.forward(X, WA, V, mode=mode)
    return check_out(O, O_ref, V, dtype), check_zstar(zs, zs_ref)
