"""The C ABI library loads and exports what include/cat.h declares (no GPU).

Only calls that fail validation before touching CUDA are made here: they
must return the documented status codes and never abort.
"""
import ctypes
import os
import re

import pytest

import fft_circulant_attention_gb300 as cat

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cat.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(cat\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from fft_circulant_attention_gb300 import build
    build.build()
    return cat.lib()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("cat_plan_create", "cat_forward", "cat_plan_destroy", "cat_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in cat.SIGNATURES, "binding lacks %s" % name


def test_binding_names_match_header():
    assert sorted(cat.SIGNATURES) == _declared()


def test_status_strings(lib):
    for code, name in cat.STATUS.items():
        assert cat.cat_status_string(code) == name
    assert cat.cat_status_string(12345) == "CAT_ERR_UNKNOWN"


def _create(lib, *args):
    h = ctypes.c_void_p()
    st = lib.cat_plan_create(ctypes.byref(h), *args)
    return st, h.value


@pytest.mark.parametrize("args,code", [
    ((1, 0, 64, 2, 0, None), cat.CAT_ERR_INVALID_ARG),      # N = 0
    ((-1, 16, 64, 2, 0, None), cat.CAT_ERR_INVALID_ARG),    # B < 0
    ((1, 16, 64, 3, 0, None), cat.CAT_ERR_INVALID_ARG),     # D % H != 0
    ((1, 16, 4, 8, 0, None), cat.CAT_ERR_INVALID_ARG),      # H > D
    ((1, 16, 64, 0, 0, None), cat.CAT_ERR_INVALID_ARG),     # H = 0
    ((1, 16, 64, 2, 7, None), cat.CAT_ERR_INVALID_ARG),     # bad dtype
    ((1, 11, 64, 2, 0, None), cat.CAT_ERR_UNSUPPORTED_N),   # prime factor 11
    ((1, 13 * 16, 64, 2, 0, None), cat.CAT_ERR_UNSUPPORTED_N),
    ((1, 1 << 23, 64, 2, 0, None), cat.CAT_ERR_UNSUPPORTED_N),  # above CAT_MAX_N
    ((1, 16, 1 << 15, 2, 0, None), cat.CAT_ERR_INVALID_ARG),    # above CAT_MAX_D
])
def test_create_rejects_bad_shapes(lib, args, code):
    st, h = _create(lib, *args)
    assert st == code
    assert not h


@pytest.mark.parametrize("args,code", [
    ((1, 0, 4, 64, 2, 0, None), cat.CAT_ERR_INVALID_ARG),       # h = 0
    ((1, 4, -1, 64, 2, 0, None), cat.CAT_ERR_INVALID_ARG),      # w < 0
    ((1, 11, 4, 64, 2, 0, None), cat.CAT_ERR_UNSUPPORTED_N),    # prime factor 11
    ((1, 4, 20000, 64, 2, 0, None), cat.CAT_ERR_UNSUPPORTED_N), # side above 16384
    ((1, 4, 4, 64, 3, 0, None), cat.CAT_ERR_INVALID_ARG),       # D % H != 0
    ((1, 4, 4, 64, 2, 9, None), cat.CAT_ERR_INVALID_ARG),       # bad dtype
])
def test_create_2d_rejects_bad_shapes(lib, args, code):
    h = ctypes.c_void_p()
    assert lib.cat_plan_create_2d(ctypes.byref(h), *args) == code
    assert not h.value
    assert lib.cat_plan_create_2d(None, *args) == cat.CAT_ERR_INVALID_ARG


def test_null_out_pointer(lib):
    assert lib.cat_plan_create(None, 1, 16, 64, 2, 0, None) == cat.CAT_ERR_INVALID_ARG


def test_null_plan_calls(lib):
    assert lib.cat_plan_destroy(None) == cat.CAT_OK
    assert lib.cat_forward(None, None, None, None, None, 1, 16, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_forward_zstar(None, None, None, None, 1, 16, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_forward_host(None, None, None, None, None, 1, 16, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_plan_sync(None) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_plan_set_stream(None, None) == cat.CAT_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(16)
    assert lib.cat_plan_describe(None, buf, 16) == cat.CAT_ERR_INVALID_ARG
    ms = (ctypes.c_float * 3)()
    assert lib.cat_plan_stage_times(None, ms, 3, None) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_plan_pass_times(None, ms, 3, None) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_backward(None, None, None, None, None, None, None, None,
                            1, 16, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat_backward_dz(None, None, None, None, None, None, None,
                               1, 16, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat2d_forward(None, None, None, None, None, 1, 4, 4, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG
    assert lib.cat2d_scores(None, None, None, None, 1, 4, 4, 64, 2, 0) == cat.CAT_ERR_INVALID_ARG


def test_python_raises_caterror(lib):
    with pytest.raises(cat.CatError) as e:
        cat.cat_plan_create(1, 11, 64, 2, "f32")
    assert e.value.status == cat.CAT_ERR_UNSUPPORTED_N


def test_dtype_codes():
    import torch
    assert cat.dtype_code(torch.float32) == cat.CAT_F32
    assert cat.dtype_code(torch.bfloat16) == cat.CAT_BF16
    assert cat.dtype_code("bf16") == cat.CAT_BF16
    with pytest.raises(ValueError):
        cat.dtype_code(torch.float16)


# --------------------------------------------------------- host path choice
# cat_plan_query runs the plan constructor's shape validation and path
# selection on the host without a device, so the choice for every workload
# shape is checked here.

@pytest.mark.parametrize("shape,expect", [
    ((1, 256, 64, 2, "f32"), ["path=smem", "reg_m=16", "radices=8x8x4"]),
    ((64, 196, 384, 6, "f32"), ["path=smem", "reg_m=14", "radices=4x7x7"]),
    ((16, 1024, 768, 12, "bf16"), ["path=smem", "reg_m=32"]),
    ((1, 1000, 10, 2, "f32"), ["path=smem", "reg_m=0", "radices=8x5x5x5"]),
    ((1, 16384, 8, 2, "f32"), ["path=smem", "reg_m=0"]),            # head width 4: not fast
    ((4, 16384, 1024, 16, "bf16"), ["path=fast", "N2=32", "chunk_bh=8", "launches=26"]),
    ((1, 131072, 1024, 16, "bf16"), ["path=fast", "N2=256", "chunk_bh=1"]),
    ((2, 32768, 128, 2, "f32"), ["path=fast", "N2=64"]),
    ((1, 20000, 4, 2, "f32"), ["path=fourstep", "N1=160(8x4x5)", "N2=125(5x5x5)"]),
    ((1, 1 << 22, 64, 1, "f32"), ["path=fourstep", "N1=2048", "N2=2048"]),   # 2^22 > 512·256
    # Short lengths without a register FFT kernel take the direct product.
    ((32, 128, 768, 12, "bf16"), ["path=direct", "TR=8", "fused=0", "launches=2"]),
    ((8, 512, 768, 12, "bf16"), ["path=direct", "fused=0"]),
    ((3, 100, 48, 3, "f32"), ["path=direct", "fused=1", "launches=1"]),
    ((1, 1000, 16, 2, "f32"), ["path=smem", "reg_m=0"]),            # N > 512: transforms
    ((4, 64, 384, 6, "f32"), ["path=smem", "reg_m=8"]),             # 8²: register FFT
])
def test_query_path_choice(lib, shape, expect):
    nbytes, desc = cat.cat_plan_query(*shape)
    for e in expect:
        assert e in desc, (e, desc)
    B, N, D, H, dt = shape
    rows = B * H * N
    assert nbytes >= rows * 12 + N * 8           # scores, z*, twiddles at least
    assert ("workspace=%d" % nbytes) in desc


def test_query_matches_between_calls_and_env(lib, monkeypatch):
    a = cat.cat_plan_query(1, 4096, 8, 2, "f32")
    assert a == cat.cat_plan_query(1, 4096, 8, 2, "f32")
    monkeypatch.setenv("CAT_FORCE_PATH", "fourstep")
    assert "path=fourstep" in cat.cat_plan_query(1, 4096, 8, 2, "f32")[1]
    monkeypatch.delenv("CAT_FORCE_PATH")
    monkeypatch.setenv("CAT_SMEM_REG", "0")
    assert "reg_m=0" in cat.cat_plan_query(1, 256, 64, 2, "f32")[1]
    monkeypatch.delenv("CAT_SMEM_REG")
    # CAT_FORCE_PATH=direct wherever the direct product is supported (head
    # width a multiple of 4, at most 128; N <= 1024), =smem never.
    monkeypatch.setenv("CAT_FORCE_PATH", "direct")
    assert "path=direct" in cat.cat_plan_query(1, 256, 64, 2, "f32")[1]
    assert "path=direct" in cat.cat_plan_query(16, 1024, 768, 12, "f32")[1]
    assert "path=smem" in cat.cat_plan_query(1, 256, 10, 2, "f32")[1]      # head width 5
    assert "path=smem" in cat.cat_plan_query(1, 2048, 64, 2, "f32")[1]     # N > 1024
    monkeypatch.setenv("CAT_FORCE_PATH", "smem")
    assert "path=smem" in cat.cat_plan_query(32, 128, 768, 12, "bf16")[1]


@pytest.mark.parametrize("shape,code", [
    ((1, 11, 64, 2, 0), cat.CAT_ERR_UNSUPPORTED_N),
    ((1, 16, 64, 3, 0), cat.CAT_ERR_INVALID_ARG),
    ((1, 16, 64, 2, 5), cat.CAT_ERR_INVALID_ARG),
])
def test_query_rejects_bad_shapes(lib, shape, code):
    assert lib.cat_plan_query(*shape, None, None, 0) == code


def test_no_device_fails_loudly(lib):
    """Without a CUDA device the library has no other way to compute: plan
    creation (1-D and 2-D) reports CAT_ERR_CUDA instead of falling back."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    with pytest.raises(cat.CatError) as e:
        cat.cat_plan_create(1, 256, 64, 2, "f32")
    assert e.value.status == cat.CAT_ERR_CUDA
    with pytest.raises(cat.CatError) as e:
        cat.cat_plan_create_2d(1, 14, 14, 64, 2, "f32")
    assert e.value.status == cat.CAT_ERR_CUDA
