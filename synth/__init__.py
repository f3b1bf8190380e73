"""Seeded synthetic inputs for the CAT forward pass.

This module holds no arithmetic of the method: it only draws random numbers
and rounds them to the run's storage type.  Both the fp64 oracle and the CUDA
path consume exactly the arrays it returns.

Recipe (the workloads of the CAT notes page — ViT patch tokens and GPT-2
masked-LM tokens — have no public inputs here, so i.i.d. Gaussians stand in):
  * numpy ``Generator(PCG64(seed))``, draws in the order X, W_A, V, each drawn
    as float32 standard normals;
  * X, V ~ N(0, 1) of shape [B, N, D];  W_A ~ N(0, 1/D) · wa_scale, [D, H];
  * the backward pass's upstream gradient dO ~ N(0, 1), [B, N, D], from a
    second, independent stream (``make_grad``);
  * the 2-D circulant attention's Q, K, V ~ N(0, 1), [B, h·w, D], from a
    third stream (``make_qkv``);
  * the value projection's W_V ~ N(0, 1/D), [D, D], from a fourth stream
    (``make_wv``);
  * then rounded to the storage dtype (float32 as drawn; bfloat16 by torch's
    round-to-nearest-even conversion).
"""
import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}

# The configurations the benchmark and parity tests use: (B, N, D, H, dtype).
CONFIGS = {
    "tiny": dict(B=1, N=256, D=64, H=2, dtype="f32"),
    "vit196": dict(B=64, N=196, D=384, H=6, dtype="f32"),
    "gpt2_f32": dict(B=16, N=1024, D=768, H=12, dtype="f32"),
    "gpt2_bf16": dict(B=16, N=1024, D=768, H=12, dtype="bf16"),
    "long16k": dict(B=4, N=16384, D=1024, H=16, dtype="bf16"),
    "long128k": dict(B=1, N=131072, D=1024, H=16, dtype="bf16"),
}


def make_inputs(B, N, D, H, dtype="f32", seed=0, wa_scale=1.0):
    """Return CPU torch tensors (X [B,N,D], W_A [D,H], V [B,N,D]) in ``dtype``."""
    if dtype not in DTYPES:
        raise ValueError("dtype must be one of %s" % sorted(DTYPES))
    rng = np.random.Generator(np.random.PCG64(seed))
    X = rng.standard_normal((B, N, D), dtype=np.float32)
    WA = rng.standard_normal((D, H), dtype=np.float32)
    WA *= np.float32(wa_scale / np.sqrt(D)) if D > 0 else np.float32(0)
    V = rng.standard_normal((B, N, D), dtype=np.float32)
    tdt = DTYPES[dtype]
    return (torch.from_numpy(X).to(tdt), torch.from_numpy(WA).to(tdt),
            torch.from_numpy(V).to(tdt))


def make_grad(B, N, D, dtype="f32", seed=0):
    """Upstream gradient dO [B, N, D] for the backward pass: float32 standard
    normals from the stream ``PCG64([seed, 1])`` (independent of the stream
    ``make_inputs`` draws X, W_A, V from), rounded to ``dtype``."""
    if dtype not in DTYPES:
        raise ValueError("dtype must be one of %s" % sorted(DTYPES))
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    G = rng.standard_normal((B, N, D), dtype=np.float32)
    return torch.from_numpy(G).to(DTYPES[dtype])


# 2-D circulant attention workloads (token grids): ViT-S/16 at 224 px (14 x 14
# patches) and at 1536 px (96 x 96 patches, the page's high-resolution
# comparison), DeiT-S width 384 with 6 heads.
GRID_CONFIGS = {
    "ca_vit196": dict(B=64, h=14, w=14, D=384, H=6, dtype="f32"),
    "ca_deit1536": dict(B=1, h=96, w=96, D=384, H=6, dtype="bf16"),
}


def make_qkv(B, N, D, dtype="f32", seed=0):
    """Q, K, V [B, N, D] for the 2-D circulant attention: float32 standard
    normals from the stream ``PCG64([seed, 2])``, drawn Q, K, V, rounded to
    ``dtype``."""
    if dtype not in DTYPES:
        raise ValueError("dtype must be one of %s" % sorted(DTYPES))
    rng = np.random.Generator(np.random.PCG64([seed, 2]))
    out = [rng.standard_normal((B, N, D), dtype=np.float32) for _ in range(3)]
    return tuple(torch.from_numpy(a).to(DTYPES[dtype]) for a in out)


def make_wv(D, dtype="f32", seed=0):
    """Value-projection weights W_V [D, D] ~ N(0, 1/D): float32 normals from
    the stream ``PCG64([seed, 3])`` (independent of the other draws), scaled,
    rounded to ``dtype``."""
    if dtype not in DTYPES:
        raise ValueError("dtype must be one of %s" % sorted(DTYPES))
    rng = np.random.Generator(np.random.PCG64([seed, 3]))
    W = rng.standard_normal((D, D), dtype=np.float32)
    W *= np.float32(1.0 / np.sqrt(D)) if D > 0 else np.float32(0)
    return torch.from_numpy(W).to(DTYPES[dtype])


def make_config(name, seed=0, wa_scale=1.0):
    c = CONFIGS[name]
    return make_inputs(c["B"], c["N"], c["D"], c["H"], c["dtype"], seed, wa_scale)
