"""cat_forward_noalloc, the plan-free forward for callers that cannot
allocate device memory (their device memory belongs to a caching or pooled
allocator, or they cannot absorb the synchronisation cudaMalloc implies).

Its output must match the plan entry point cat_forward, through the C ABI,
within the parity tolerances (2e-5·max|V| for fp32 storage, 8e-3·max|V| for
bf16), on two calls in a row — the second call finds the fixed workspace
holding the first call's data — and the fp64 oracle within the same bounds.
The bf16 cases cover all three score kernels the entry point can take: the
tensor-copy (TMA) kernel (D a multiple of 64), the register-fed MMA kernel
(D a multiple of 32) and the CUDA-core kernel.  This file is collected last
on purpose.
"""
import numpy as np
import pytest
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-5, "bf16": 8e-3}


@pytest.fixture(autouse=True)
def _built(cuda_device):
    from fft_circulant_attention_gb300 import build
    build.build()
    cat.lib()
    yield


def _dev(*ts):
    return [t.to("cuda:0").contiguous() for t in ts]


def _plan_forward(X, WA, V, dtype):
    B, N, D = V.shape
    H = WA.shape[1]
    with cat.Plan(B, N, D, H, dtype) as p:
        O = p.forward(X, WA, V)
        p.sync()
    return O


@pytest.mark.parametrize("B,N,D,H,dtype", [
    (2, 1024, 64, 4, "f32"),
    (3, 196, 48, 6, "bf16"),        # CUDA-core score
    (1, 16384, 16, 1, "f32"),
    (4, 100, 18, 3, "bf16"),        # CUDA-core score, ragged D
    (2, 256, 64, 1, "bf16"),        # TMA score (D % 64 == 0)
    (2, 1024, 128, 2, "bf16"),      # TMA score, head width 64
    (2, 512, 96, 3, "bf16"),        # register-fed MMA score (D % 32 == 0)
    (1, 1024, 768, 12, "bf16"),     # GPT-2-small width, TMA score
    (16, 1024, 768, 12, "bf16"),    # the whole GPT-2-small bf16 workload
])
def test_noalloc_matches_plan_entry(B, N, D, H, dtype):
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=N + D)
    Xd, Wd, Vd = _dev(X, WA, V)
    ref = _plan_forward(Xd, Wd, Vd, dtype)
    bound = TOL[dtype] * float(V.double().abs().max())
    O_or, _ = oracle.forward(X, WA, V, mode="direct" if B * N * N * D <= 2e9 else "fft")
    stream = torch.cuda.current_stream()
    for _ in range(2):
        O = torch.full_like(Vd, float("nan"))
        cat.cat_forward_noalloc(Xd, Wd, Vd, O, B, N, D, H, dtype, stream)
        torch.cuda.synchronize()
        err = float((O.double() - ref.double()).abs().max())
        assert err <= bound, (err, bound)
        err_or = float(np.abs(O.double().cpu().numpy() - O_or).max())
        assert err_or <= bound, (err_or, bound)


def test_noalloc_alternating_lengths():
    """Calls of different N in a row re-fill the shared twiddle region."""
    cases = [(2, 256, 32, 2, "f32"), (1, 1000, 32, 2, "f32"), (2, 256, 32, 2, "f32")]
    stream = torch.cuda.current_stream()
    for B, N, D, H, dtype in cases:
        X, WA, V = _dev(*synth.make_inputs(B, N, D, H, dtype, seed=N))
        ref = _plan_forward(X, WA, V, dtype)
        O = torch.empty_like(V)
        cat.cat_forward_noalloc(X, WA, V, O, B, N, D, H, dtype, stream)
        torch.cuda.synchronize()
        assert float((O - ref).abs().max()) <= TOL[dtype] * float(V.abs().max())


def test_noalloc_rejected_call_does_not_poison_the_next():
    """A call refused by the host checks leaves the shared workspace (its
    twiddle length in particular) as it was: the next call is correct."""
    stream = torch.cuda.current_stream()
    B, N, D, H, dtype = 2, 1000, 32, 2, "f32"
    X, WA, V = _dev(*synth.make_inputs(B, N, D, H, dtype, seed=7))
    ref = _plan_forward(X, WA, V, dtype)
    X5, V5 = X[:, :500].contiguous(), V[:, :500].contiguous()
    bad = torch.empty(V5.numel() + 4, device="cuda:0")[1:1 + V5.numel()].view_as(V5)
    with pytest.raises(cat.CatError) as e:      # misaligned output, other length
        cat.cat_forward_noalloc(X5, WA, V5, bad, B, 500, D, H, dtype, stream)
    assert e.value.status == cat.CAT_ERR_MISALIGNED
    O = torch.empty_like(V)
    cat.cat_forward_noalloc(X, WA, V, O, B, N, D, H, dtype, stream)
    torch.cuda.synchronize()
    assert float((O - ref).abs().max()) <= TOL[dtype] * float(V.abs().max())


def test_noalloc_rejects_sizes_beyond_its_workspace():
    X = torch.empty(16, device="cuda:0")
    with pytest.raises(cat.CatError) as e:      # B·H·N above the fixed workspace
        cat.cat_forward_noalloc(X, X, X, X, 64, 8192, 64, 1, "f32")
    assert e.value.status == cat.CAT_ERR_TOO_LARGE
    with pytest.raises(cat.CatError) as e:      # N above the single-CTA path
        cat.cat_forward_noalloc(X, X, X, X, 1, 32768, 8, 1, "f32")
    assert e.value.status == cat.CAT_ERR_TOO_LARGE
