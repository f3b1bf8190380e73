"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every case draws seeded synthetic inputs, runs cat_forward on cuda:0 and
compares element by element with the oracle (the plain definitions of the
CAT notes page, section 方法详解: score, softmax over tokens, circulant
product).  Bounds: O within 2e-5·max|V| (fp32 storage) or 8e-3·max|V|
(bf16 storage); z* within 1e-5 relative.
"""
import os

import numpy as np
import pytest
import torch

import fft_circulant_attention_gb300 as cat
import oracle
import synth
from _gpu_helpers import check_out, check_zstar, parity, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _needs_gpu(cuda_device):
    from fft_circulant_attention_gb300 import build
    build.build()
    yield


# ---------------------------------------------------------------- workloads

SMALL_CONFIGS = {
    "tiny": dict(B=1, N=256, D=64, H=2, dtype="f32"),
    "vit196": dict(B=64, N=196, D=384, H=6, dtype="f32"),
    "gpt2_f32": dict(B=16, N=1024, D=768, H=12, dtype="f32"),
    "gpt2_bf16": dict(B=16, N=1024, D=768, H=12, dtype="bf16"),
    "gpt2_peaked": dict(B=16, N=1024, D=768, H=12, dtype="f32", wa_scale=8.0),
    "gpt2_peaked_bf16": dict(B=16, N=1024, D=768, H=12, dtype="bf16", wa_scale=8.0),
}


@pytest.mark.parametrize("name", list(SMALL_CONFIGS))
def test_workload_parity(name):
    cfg = dict(SMALL_CONFIGS[name])
    errO, errZ = parity(**cfg)
    print("%s: max|dO|/max|V| = %.2e, max rel dz* = %.2e" % (name, errO, errZ))


def _sampled_rows(N, k, seed):
    rng = np.random.default_rng(seed)
    rows = {0, 1, N // 2, N - 1}
    rows.update(int(r) for r in rng.choice(N, size=k, replace=False))
    return sorted(rows)


# Output rows compared with the definition at the full-size long workloads:
# i = 32·r (4096 rows at N = 131072, 512 at N = 16384), every batch and
# column, plus the last row and a few random ones off that grid.
ROW_STEP = 32


def _slice_rows(N):
    rows = set(range(0, N, ROW_STEP))
    rows.update(_sampled_rows(N, 8, 1))
    return sorted(rows)


@pytest.mark.parametrize("name", ["long16k", "long128k"])
def test_long_workload_sampled(name):
    """Full-size long-sequence workloads in the benchmark's launch shape:
    all of z* against the oracle, and O on a slice of rows i = 32·r (4096 rows
    of the 131072-token workload; every batch and all 1024 columns) against
    the O(N)-per-element definition."""
    c = synth.CONFIGS[name]
    X, WA, V = synth.make_inputs(c["B"], c["N"], c["D"], c["H"], c["dtype"], seed=0)
    O, zs = run_gpu(X, WA, V, c["dtype"])
    zs_ref = oracle.zstar(X, WA)
    errZ = check_zstar(zs, zs_ref)
    rows = _slice_rows(c["N"])
    O_ref = oracle.circ_direct_rows(zs_ref, V, rows)
    errO = check_out(O[:, rows], O_ref, V, c["dtype"])
    # Column sums are kept by a circulant whose columns sum to one.
    Vs = V.double().sum(1).numpy()
    Os = O.double().sum(1).numpy()
    assert np.abs(Os - Vs).max() <= 8e-3 * np.abs(V.double().numpy()).max() * np.sqrt(c["N"])
    print("%s: max|dO|/max|V| = %.2e (%d rows), max rel dz* = %.2e" % (name, errO, len(rows), errZ))


# --------------------------------------------------------- length sweeps

SMEM_NS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 12, 14, 15, 16, 21, 25, 27, 32, 35, 49, 64, 96,
           100, 125, 128, 196, 210, 243, 256, 343, 512, 1000, 1024, 2048, 2401, 4096,
           8192, 15625, 16384]


@pytest.mark.parametrize("N", SMEM_NS)
def test_length_sweep_f32(N):
    mode = "direct" if N <= 4096 else "fft"
    parity(2, N, 8, 2, "f32", seed=N, mode=mode)


@pytest.mark.parametrize("N", [7, 64, 196, 1000, 16384])
def test_length_sweep_bf16(N):
    parity(1, N, 16, 2, "bf16", seed=N, mode="direct" if N <= 4096 else "fft")


FOURSTEP_NS = [32768, 49152, 65536, 3 * 5 * 7 * 512]


@pytest.mark.parametrize("N", FOURSTEP_NS)
def test_fourstep_lengths(N):
    """Lengths above the single-CTA limit take the four-step path."""
    parity(1, N, 8, 2, "f32", seed=N, mode="fft")


@pytest.fixture
def force_fourstep():
    os.environ["CAT_FORCE_PATH"] = "fourstep"
    yield
    del os.environ["CAT_FORCE_PATH"]


@pytest.mark.parametrize("N,D,H,dtype", [
    (4, 8, 2, "f32"), (12, 8, 2, "f32"), (64, 16, 2, "f32"), (196, 24, 3, "f32"),
    (1024, 64, 2, "bf16"), (4096, 16, 4, "f32"), (16384, 8, 1, "f32"),
    (100, 6, 2, "bf16"), (256, 18, 3, "f32"),
])
def test_fourstep_forced(force_fourstep, N, D, H, dtype):
    """The four-step path on short sequences, where the oracle is cheap."""
    with cat.Plan(1, N, D, H, dtype) as p:
        assert "fourstep" in p.describe()
    parity(2, N, D, H, dtype, seed=N + D, mode="direct" if N <= 4096 else "fft")


# ------------------------------------------------------------- edge cases

@pytest.mark.parametrize("B,N,D,H,dtype", [
    (2, 64, 6, 2, "f32"),      # odd head width (a half pair per head)
    (2, 64, 9, 3, "bf16"),     # odd head width, bf16, unaligned pairs
    (1, 128, 64, 32, "f32"),   # more than 16 heads (two score passes)
    (1, 128, 40, 20, "bf16"),
    (3, 50, 6, 1, "f32"),      # D not a multiple of the vector width
    (1, 1, 8, 2, "f32"),       # single token
    (1, 2, 2, 2, "bf16"),      # head width 1
    (5, 96, 256, 1, "bf16"),   # one head owning all columns
])
def test_shapes(B, N, D, H, dtype):
    parity(B, N, D, H, dtype, seed=B * 1000 + N, mode="direct")


def test_single_token_is_identity():
    X, WA, V = synth.make_inputs(3, 1, 16, 4, "f32", seed=3)
    O, zs = run_gpu(X, WA, V, "f32")
    assert torch.equal(zs, torch.ones_like(zs))
    assert torch.equal(O, V)


def test_empty_batch():
    with cat.Plan(0, 64, 8, 2, "f32") as p:
        X = torch.empty((0, 64, 8), device="cuda:0")
        W = torch.empty((8, 2), device="cuda:0")
        O = p.forward(X, W, X.clone())
        p.sync()
    assert O.shape == (0, 64, 8)


def _one_hot_inputs(N, D, H, shifts, dtype):
    _, _, V = synth.make_inputs(1, N, D, H, dtype, seed=11)
    X = torch.zeros((1, N, D))
    WA = torch.zeros((D, H))
    for h, s in enumerate(shifts):
        WA[h, h] = 1.0
        X[0, :, h] = -100.0
        X[0, s, h] = 100.0
    return X.to(V.dtype), WA.to(V.dtype), V


@pytest.mark.parametrize("N,dtype", [(40, "f32"), (196, "bf16"), (4096, "f32"), (32768, "bf16")])
def test_one_hot_is_cyclic_shift(N, dtype):
    """z* one-hot at s_h gives O[i] = V[(i - s_h) mod N] for head h."""
    D, H = 8, 4
    shifts = [0, 1, 7, N - 3]
    X, WA, V = _one_hot_inputs(N, D, H, shifts, dtype)
    O, zs = run_gpu(X, WA, V, dtype)
    dh = D // H
    vmax = float(V.double().abs().max())
    tol = 2e-5 if dtype == "f32" else 8e-3
    for h, s in enumerate(shifts):
        assert float(zs[0, h, s]) == 1.0
        cols = slice(h * dh, (h + 1) * dh)
        ref = torch.roll(V[0, :, cols].double(), s, dims=0)
        assert float((O[0, :, cols].double() - ref).abs().max()) <= tol * vmax


@pytest.mark.parametrize("N,dtype", [(27, "f32"), (1024, "bf16"), (65536, "f32")])
def test_uniform_gives_column_mean(N, dtype):
    X, WA, V = synth.make_inputs(2, N, 12, 3, dtype, seed=12)
    WA = torch.zeros_like(WA)
    O, zs = run_gpu(X, WA, V, dtype)
    assert float((zs.double() - 1.0 / N).abs().max()) <= 1e-5 / N
    ref = V.double().mean(1, keepdim=True).expand_as(O)
    tol = 2e-5 if dtype == "f32" else 8e-3
    assert float((O.double() - ref).abs().max()) <= tol * float(V.double().abs().max())


# ------------------------------------------------------- API behaviour

@pytest.mark.parametrize("B,N,D,H,dtype", [
    (2, 1024, 64, 4, "bf16"),      # two one-batch steps
    (5, 196, 384, 6, "f32"),       # odd step count: both staging slots, last one alone
    (3, 16384, 128, 2, "bf16"),    # the fast path in one-batch sub-plans
    (1, 1000, 16, 2, "f32"),       # one batch: the serial copy, compute, copy
])
def test_host_buffer_entry_matches_device_entry(B, N, D, H, dtype):
    """The host-buffer entry (copies inside the call, overlapped with the
    compute one batch per step) gives the device entry's output bit for bit:
    every (b, h) is computed by the same kernels on the same values."""
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=5)
    Od, _ = run_gpu(X, WA, V, dtype, want_zstar=False)
    Xp, Wp, Vp = (t.pin_memory() for t in (X, WA, V))
    Oh = torch.empty_like(Vp).pin_memory()
    with cat.Plan(B, N, D, H, dtype) as p:
        p.forward_host(Xp, Wp, Vp, Oh)
        Oh.fill_(float("nan"))
        p.forward_host(Xp, Wp, Vp, Oh)   # staging buffers and sub-plans are reused
        p.sync()
    assert torch.equal(Oh, Od)


def test_deterministic():
    X, WA, V = to_dev(*synth.make_inputs(2, 2048, 64, 4, "f32", seed=6))
    with cat.Plan(2, 2048, 64, 4, "f32") as p:
        a = p.forward(X, WA, V).clone()
        for _ in range(3):
            assert torch.equal(p.forward(X, WA, V), a)
        p.sync()


def test_error_paths_leave_context_usable():
    X, WA, V = to_dev(*synth.make_inputs(1, 64, 8, 2, "f32", seed=7))
    with cat.Plan(1, 64, 8, 2, "f32") as p:
        O = torch.empty_like(V)
        raw = torch.empty(V.numel() + 1, device="cuda:0")
        with pytest.raises(cat.CatError) as e:       # misaligned by 4 bytes
            cat.cat_forward(p.handle, X, WA, V, raw.data_ptr() + 4, 1, 64, 8, 2, 0)
        assert e.value.status == cat.CAT_ERR_MISALIGNED
        with pytest.raises(cat.CatError) as e:       # shape differs from the plan
            cat.cat_forward(p.handle, X, WA, V, O, 1, 32, 8, 2, 0)
        assert e.value.status == cat.CAT_ERR_PLAN_MISMATCH
        with pytest.raises(cat.CatError) as e:       # O overlaps V
            cat.cat_forward(p.handle, X, WA, V, V, 1, 64, 8, 2, 0)
        assert e.value.status == cat.CAT_ERR_ALIAS
        with pytest.raises(cat.CatError) as e:
            cat.cat_forward(p.handle, None, WA, V, O, 1, 64, 8, 2, 0)
        assert e.value.status == cat.CAT_ERR_INVALID_ARG
        p.forward(X, WA, V, O)
        p.sync()
    O_ref, _ = oracle.forward(X.cpu(), WA.cpu(), V.cpu(), mode="direct")
    assert float(np.abs(O.cpu().double().numpy() - O_ref).max()) <= 2e-5 * float(V.abs().max())


def test_plan_on_a_side_stream():
    s = torch.cuda.Stream()
    X, WA, V = to_dev(*synth.make_inputs(2, 512, 32, 2, "f32", seed=8))
    with torch.cuda.stream(s):
        with cat.Plan(2, 512, 32, 2, "f32", stream=s) as p:
            O = p.forward(X, WA, V)
            p.sync()
    O_ref, _ = oracle.forward(X.cpu(), WA.cpu(), V.cpu(), mode="direct")
    assert float(np.abs(O.cpu().double().numpy() - O_ref).max()) <= 2e-5 * float(V.abs().max())


def test_plans_of_different_lengths_coexist():
    """Two live plans whose kernels need different shared memory: creating
    the smaller one must not break the larger one's launches."""
    big = synth.make_inputs(1, 16384, 16, 2, "f32", seed=21)
    small = synth.make_inputs(2, 256, 16, 2, "f32", seed=22)
    with cat.Plan(1, 16384, 16, 2, "f32") as pb:
        with cat.Plan(2, 256, 16, 2, "f32") as ps:
            Ob = pb.forward(*to_dev(*big))
            Os = ps.forward(*to_dev(*small))
            pb.sync()
            ps.sync()
    for (X, WA, V), O in ((big, Ob), (small, Os)):
        O_ref, _ = oracle.forward(X, WA, V, mode="fft")
        assert float(np.abs(O.cpu().double().numpy() - O_ref).max()) <= 2e-5 * float(V.abs().max())


@pytest.mark.parametrize("N,B,H,dtype", [
    (16384, 2, 1, "f32"), (16384, 1, 2, "bf16"), (32768, 1, 1, "f32"),
    (65536, 1, 1, "bf16"), (131072, 1, 1, "f32"), (131072, 1, 2, "bf16"),
])
def test_fast_path_lengths(N, B, H, dtype):
    """Head width 64 and N = 512·N2 (N2 = 32..256) take the three-pass fast
    path; checked against the oracle's convolution-theorem evaluation."""
    D = 64 * H
    with cat.Plan(B, N, D, H, dtype) as p:
        assert "path=fast" in p.describe()
    parity(B, N, D, H, dtype, seed=N + H, mode="fft")


def test_fast_path_chunks(monkeypatch):
    """Chunks of 1, 3 (ragged: 3 + 1) and 4 heads per scratch slot, on the
    overlapped two-stream schedule and on the serialised one (stage timing
    on), all give the same result."""
    X, WA, V = to_dev(*synth.make_inputs(3, 16384, 256, 4, "bf16", seed=31))
    outs = []
    for chunk in ("1", "3", "4"):
        monkeypatch.setenv("CAT_CHUNK_BH", chunk)
        with cat.Plan(3, 16384, 256, 4, "bf16") as p:
            assert "chunk_bh=%s" % chunk in p.describe()
            outs.append(p.forward(X, WA, V))
            p.timing(1)
            outs.append(p.forward(X, WA, V))
            p.sync()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    O_ref, _ = oracle.forward(X.cpu(), WA.cpu(), V.cpu(), mode="fft")
    assert float(np.abs(outs[0].cpu().double().numpy() - O_ref).max()) <= 8e-3 * float(V.abs().max())


@pytest.mark.parametrize("score", ["tma", "mma", "cuda"])
@pytest.mark.parametrize("cfg", [dict(B=4, N=1024, D=768, H=12, wa_scale=8.0),
                                 dict(B=2, N=2048, D=1024, H=16, wa_scale=1.0),
                                 dict(B=1, N=512, D=96, H=3, wa_scale=8.0),
                                 dict(B=3, N=100, D=128, H=32, wa_scale=8.0)])
def test_bf16_score_kernels(monkeypatch, score, cfg):
    """All three bf16 score kernels (TMA-fed tensor-core slices, register-fed
    tensor-core slices, CUDA-core runs; each with a double-float total) meet
    the z* bound, peaked case and ragged token tiles included."""
    if score == "tma":
        monkeypatch.delenv("CAT_SCORE", raising=False)
    else:
        monkeypatch.setenv("CAT_SCORE", score)
    errO, errZ = parity(dtype="bf16", seed=41, mode="fft", **cfg)
    print("score=%s %s: dO %.2e, dz* %.2e" % (score, cfg, errO, errZ))


def test_graph_replay_follows_pointers(monkeypatch):
    """The fast path replays a captured CUDA graph while the call's pointers
    stay the same and updates it when they change: alternating between two
    input sets and two outputs gives, every time, what direct launches give."""
    B, N, D, H = 2, 16384, 128, 2
    sets = [to_dev(*synth.make_inputs(B, N, D, H, "bf16", seed=s)) for s in (51, 52)]
    monkeypatch.setenv("CAT_GRAPH", "0")
    with cat.Plan(B, N, D, H, "bf16") as p:
        assert "graph=0" in p.describe()
        want = [p.forward(*xs) for xs in sets]
        p.sync()
    monkeypatch.delenv("CAT_GRAPH")
    outs = [torch.empty_like(sets[0][2]) for _ in range(2)]
    with cat.Plan(B, N, D, H, "bf16") as p:
        assert "graph=1" in p.describe()
        for k in (0, 1, 1, 0, 0, 1):
            outs[k].zero_()
            p.forward(*sets[k], outs[k])
            p.sync()
            assert torch.equal(outs[k], want[k])
        # A new output buffer with the same inputs.
        O2 = torch.empty_like(outs[0])
        p.forward(*sets[0], O2)
        p.sync()
        assert torch.equal(O2, want[0])


@pytest.mark.parametrize("fork", ["start", "score", "spectrum"])
def test_repeated_forwards_are_bit_identical(monkeypatch, fork):
    """Thirty forwards of the 131072-token workload give bit-identical
    outputs with each fork point of the overlapped schedule, including the
    one where the score runs beside the first FFT passes: every stage a
    tensor copy refills was read before the copy rewrites it."""
    monkeypatch.setenv("CAT_FORK", fork)
    B, N, D, H = 1, 131072, 1024, 16
    X, WA, V = to_dev(*synth.make_inputs(B, N, D, H, "bf16", seed=61))
    with cat.Plan(B, N, D, H, "bf16") as p:
        first = p.forward(X, WA, V)
        O = torch.empty_like(first)
        for _ in range(30):
            O.zero_()
            p.forward(X, WA, V, O)
            p.sync()
            assert torch.equal(O, first)


def test_pass_times_cover_the_circulant_product():
    """With timing armed, the fast path records an event after each pass of
    each chunk: one launch of each pass per chunk and call, and the three
    passes' times add up to the circulant-product stage."""
    B, N, D, H = 2, 16384, 256, 4
    X, WA, V = to_dev(*synth.make_inputs(B, N, D, H, "bf16", seed=71))
    with cat.Plan(B, N, D, H, "bf16") as p:
        desc = p.describe()
        chunks = -(-B * H // int(desc.split("chunk_bh=")[1].split()[0]))
        p.timing(3)
        for _ in range(3):
            p.forward(X, WA, V)
        stage, calls = p.stage_times()
        passes, launches = p.pass_times()
        p.timing(0)
    assert calls == 3 and launches == 3 * chunks
    assert all(t > 0 for t in stage) and all(t > 0 for t in passes)
    assert sum(passes) <= stage[2] * 1.001 + 1e-3
    assert sum(passes) >= 0.5 * stage[2]


@pytest.mark.parametrize("N", [64, 196, 256, 1024])
@pytest.mark.parametrize("B,D,H,dtype", [(3, 128, 2, "f32"), (2, 384, 6, "bf16"),
                                         (2, 75, 5, "f32"), (1, 63, 3, "bf16")])
def test_square_lengths_register_kernel(monkeypatch, N, B, D, H, dtype):
    """Square lengths N = M² (M = 8, 14, 16, 32) take the two-step register
    kernel for the circulant product.  Odd head widths (15, 21) put pairs at
    odd columns and a lone last column in every head.  Checked against the
    oracle, and against the block-FFT kernel the lengths otherwise take."""
    with cat.Plan(B, N, D, H, dtype) as p:
        assert "reg_m=%d" % int(round(N ** 0.5)) in p.describe()
    parity(B, N, D, H, dtype, seed=N + D)
    X, WA, V = to_dev(*synth.make_inputs(B, N, D, H, dtype, seed=N + D))
    with cat.Plan(B, N, D, H, dtype) as p:
        O_reg = p.forward(X, WA, V)
        p.sync()
    monkeypatch.setenv("CAT_SMEM_REG", "0")
    with cat.Plan(B, N, D, H, dtype) as p:
        assert "reg_m=0" in p.describe()
        O_blk = p.forward(X, WA, V)
        p.sync()
    scale = float(V.abs().max())
    tol = (8e-3 if dtype == "bf16" else 2e-5) * scale
    assert float((O_reg.float() - O_blk.float()).abs().max()) <= tol


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_longest_sequence(dtype):
    """The longest sequence the ABI accepts (CAT_MAX_N = 2²² tokens) on the
    general four-step path: all of z* against the oracle, O at sampled rows
    against the per-element definition, and the column sums a circulant
    with unit column sums keeps."""
    B, N, D, H = 1, 1 << 22, 4, 2
    X, WA, V = synth.make_inputs(B, N, D, H, dtype, seed=81)
    with cat.Plan(B, N, D, H, dtype) as p:
        assert "path=fourstep" in p.describe()
    O, zs = run_gpu(X, WA, V, dtype)
    zs_ref = oracle.zstar(X, WA)
    check_zstar(zs, zs_ref)
    rows = _sampled_rows(N, 12, 2)
    O_ref = oracle.circ_direct_rows(zs_ref, V, rows)
    check_out(O[:, rows], O_ref, V, dtype)
    Vs = V.double().sum(1).numpy()
    Os = O.double().sum(1).numpy()
    tol = (8e-3 if dtype == "bf16" else 2e-5) * np.abs(V.double().numpy()).max() * np.sqrt(N)
    assert np.abs(Os - Vs).max() <= tol
