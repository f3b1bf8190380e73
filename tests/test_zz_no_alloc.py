"""cat_forward_noalloc, the plan-free forward for callers that cannot
allocate device memory (their device memory belongs to a caching or pooled
allocator, or they cannot absorb the synchronisation cudaMalloc implies).

Its output must match the plan entry point cat_forward, through the C ABI,
within the parity tolerances (2e-5·max|V| for fp32 storage, 8e-3·max|V| for
bf16), on two calls in a row — the second call finds the fixed workspace
holding the first call's data.  This file is collected last on purpose.
"""
import pytest
import torch

import fft_circulant_attention_gb300 as cat
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
    (3, 196, 48, 6, "bf16"),
    (1, 16384, 16, 1, "f32"),
    (4, 100, 18, 3, "bf16"),
])
def test_noalloc_matches_plan_entry(B, N, D, H, dtype):
    X, WA, V = _dev(*synth.make_inputs(B, N, D, H, dtype, seed=N + D))
    ref = _plan_forward(X, WA, V, dtype)
    bound = TOL[dtype] * float(V.double().abs().max())
    stream = torch.cuda.current_stream()
    for _ in range(2):
        O = torch.full_like(V, float("nan"))
        cat.cat_forward_noalloc(X, WA, V, O, B, N, D, H, dtype, stream)
        torch.cuda.synchronize()
        err = float((O.double() - ref.double()).abs().max())
        assert err <= bound, (err, bound)


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


def test_noalloc_rejects_sizes_beyond_its_workspace():
    X = torch.empty(16, device="cuda:0")
    with pytest.raises(cat.CatError) as e:      # B·H·N above the fixed workspace
        cat.cat_forward_noalloc(X, X, X, X, 64, 8192, 64, 1, "f32")
    assert e.value.status == cat.CAT_ERR_TOO_LARGE
    with pytest.raises(cat.CatError) as e:      # N above the single-CTA path
        cat.cat_forward_noalloc(X, X, X, X, 1, 32768, 8, 1, "f32")
    assert e.value.status == cat.CAT_ERR_TOO_LARGE
