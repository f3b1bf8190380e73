"""Python binding of libcat, the GB300 CAT library (include/cat.h): the
forward pass and its backward pass.

CAT (circular-convolutional attention), from the notes page "CAT:
Circular-Convolutional Attention for Sub-Quadratic Transformers", section
方法详解: per batch b and head h, z = X·W_A[:, h], z* = softmax over the N
tokens, and O_h = circ(z*)·V_h = IFFT(FFT(z*) ⊙ FFT(V_h)).

This module only marshals arguments (tensor -> device pointer, stream ->
handle, status -> exception).  Every step of the computation runs in the
CUDA kernels of ``libcat.so``; there is no other implementation behind it,
and importing it fails loudly when the library has not been built.

The functions carry the C names: ``cat_plan_create``, ``cat_forward``,
``cat_forward_zstar``, ``cat_forward_host``, ``cat_forward_fused``,
``cat_project``, ``cat_forward_noalloc``, ``cat_backward``,
``cat_backward_dz``, ``cat_plan_create_2d``, ``cat2d_forward``, ``cat2d_scores``,
``cat_plan_query``,
``cat_plan_sync``,
``cat_plan_timing``, ``cat_plan_stage_times``, ``cat_plan_pass_times``,
``cat_plan_describe``, ``cat_plan_set_stream``, ``cat_plan_destroy`` and
``cat_status_string``.  ``Plan`` (1-D) and ``Plan2D`` (token grid) wrap them
for convenience.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcat.so")

CAT_F32, CAT_BF16 = 0, 1
CAT_OK = 0
STATUS = {
    0: "CAT_OK", -1: "CAT_ERR_INVALID_ARG", -2: "CAT_ERR_UNSUPPORTED_N",
    -3: "CAT_ERR_MISALIGNED", -4: "CAT_ERR_PLAN_MISMATCH", -5: "CAT_ERR_ALLOC",
    -6: "CAT_ERR_CUDA", -7: "CAT_ERR_DEVICE_STATUS", -8: "CAT_ERR_ALIAS",
    -9: "CAT_ERR_TOO_LARGE",
}
for _code, _name in STATUS.items():
    globals()[_name] = _code

# Every symbol include/cat.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "cat_plan_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _I, _P]),
    "cat_plan_destroy": (_I, [_P]),
    "cat_plan_set_stream": (_I, [_P, _P]),
    "cat_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_forward_zstar": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_forward_fused": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_project": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_forward_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_plan_sync": (_I, [_P]),
    "cat_plan_describe": (_I, [_P, ctypes.c_char_p, _I]),
    "cat_plan_timing": (_I, [_P, _I]),
    "cat_plan_stage_times": (_I, [_P, ctypes.POINTER(ctypes.c_float), _I,
                                  ctypes.POINTER(_I)]),
    "cat_plan_pass_times": (_I, [_P, ctypes.POINTER(ctypes.c_float), _I,
                                 ctypes.POINTER(_I)]),
    "cat_forward_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "cat_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_backward_dz": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I]),
    "cat_plan_create_2d": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _I, _I, _P]),
    "cat_plan_query": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t), ctypes.c_char_p,
                            _I]),
    "cat2d_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I]),
    "cat2d_scores": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I]),
    "cat_probe_dft32": (_I, [_P, _P, _I, _I, _I, _P]),
    "cat_status_string": (ctypes.c_char_p, [_I]),
}

_LIB = None


class CatError(RuntimeError):
    """A libcat call returned a non-zero status."""

    def __init__(self, status, where=""):
        self.status = status
        super().__init__("%s%s (%d)" % (where + ": " if where else "",
                                        STATUS.get(status, "CAT_ERR_UNKNOWN"), status))


def lib():
    """The loaded libcat.so (ctypes.CDLL).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libcat.so is missing at %s: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _ptr(x):
    """Device or host address of a tensor / numpy array / int (None -> 0)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError("cannot take the address of %r" % type(x))


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st, where):
    if st != CAT_OK:
        raise CatError(st, where)


def dtype_code(dtype):
    """CAT_F32 / CAT_BF16 from a code, a name or a torch dtype."""
    if isinstance(dtype, int):
        return dtype
    name = str(dtype).replace("torch.", "")
    if name in ("float32", "f32", "float"):
        return CAT_F32
    if name in ("bfloat16", "bf16"):
        return CAT_BF16
    raise ValueError("unsupported dtype %r" % (dtype,))


def cat_probe_dft32(x, y, nsig, mode, rounds, stream=None):
    """Measurement probe: one DFT-32 stage `rounds` times on `nsig` signals
    (mode 0 FP32 pipe, 1 / 2 tensor cores with 2 / 3 bf16 terms)."""
    _check(lib().cat_probe_dft32(_ptr(x), _ptr(y), nsig, mode, rounds, _stream(stream)),
           "cat_probe_dft32")


def cat_status_string(status):
    return lib().cat_status_string(status).decode()


def cat_plan_create(B, N, D, H, dtype, stream=None):
    """Create a plan; returns its handle (an int).  Raises CatError."""
    h = ctypes.c_void_p()
    _check(lib().cat_plan_create(ctypes.byref(h), B, N, D, H, dtype_code(dtype),
                                 _stream(stream)), "cat_plan_create")
    return h.value


def cat_plan_query(B, N, D, H, dtype):
    """(device workspace bytes, description) of the plan cat_plan_create would
    build for this shape, computed on the host without a device."""
    nbytes = ctypes.c_size_t(0)
    buf = ctypes.create_string_buffer(512)
    _check(lib().cat_plan_query(B, N, D, H, dtype_code(dtype), ctypes.byref(nbytes), buf, 512),
           "cat_plan_query")
    return nbytes.value, buf.value.decode()


def cat_plan_destroy(plan):
    _check(lib().cat_plan_destroy(plan), "cat_plan_destroy")


def cat_plan_set_stream(plan, stream):
    _check(lib().cat_plan_set_stream(plan, _stream(stream)), "cat_plan_set_stream")


def cat_forward(plan, X, W_A, V, O, B, N, D, H, dtype):
    _check(lib().cat_forward(plan, _ptr(X), _ptr(W_A), _ptr(V), _ptr(O), B, N, D, H,
                             dtype_code(dtype)), "cat_forward")


def cat_forward_zstar(plan, X, W_A, zstar, B, N, D, H, dtype):
    _check(lib().cat_forward_zstar(plan, _ptr(X), _ptr(W_A), _ptr(zstar), B, N, D, H,
                                   dtype_code(dtype)), "cat_forward_zstar")


def cat_forward_host(plan, X, W_A, V, O, B, N, D, H, dtype):
    _check(lib().cat_forward_host(plan, _ptr(X), _ptr(W_A), _ptr(V), _ptr(O), B, N, D, H,
                                  dtype_code(dtype)), "cat_forward_host")


def cat_forward_fused(plan, X, W_V, W_A, V, O, B, N, D, H, dtype):
    _check(lib().cat_forward_fused(plan, _ptr(X), _ptr(W_V), _ptr(W_A), _ptr(V), _ptr(O), B, N, D,
                                   H, dtype_code(dtype)), "cat_forward_fused")


def cat_project(plan, X, W_V, W_A, V, zstar, B, N, D, H, dtype):
    _check(lib().cat_project(plan, _ptr(X), _ptr(W_V), _ptr(W_A), _ptr(V), _ptr(zstar), B, N, D,
                             H, dtype_code(dtype)), "cat_project")


def cat_forward_noalloc(X, W_A, V, O, B, N, D, H, dtype, stream=None):
    """The forward without a plan or any allocation (fixed device workspace;
    B·H·N and N bounded).  Enqueued on `stream` (default: the legacy default
    stream)."""
    _check(lib().cat_forward_noalloc(_ptr(X), _ptr(W_A), _ptr(V), _ptr(O), B, N, D, H,
                                     dtype_code(dtype), _stream(stream)), "cat_forward_noalloc")


def cat_backward(plan, X, W_A, V, dO, dX, dW_A, dV, B, N, D, H, dtype):
    _check(lib().cat_backward(plan, _ptr(X), _ptr(W_A), _ptr(V), _ptr(dO), _ptr(dX), _ptr(dW_A),
                              _ptr(dV), B, N, D, H, dtype_code(dtype)), "cat_backward")


def cat_backward_dz(plan, X, W_A, V, dO, dzstar, dz, B, N, D, H, dtype):
    _check(lib().cat_backward_dz(plan, _ptr(X), _ptr(W_A), _ptr(V), _ptr(dO), _ptr(dzstar),
                                 _ptr(dz), B, N, D, H, dtype_code(dtype)), "cat_backward_dz")


def cat_plan_create_2d(B, h, w, D, H, dtype, stream=None):
    """Create a 2-D (h x w token grid) plan; returns its handle."""
    hd = ctypes.c_void_p()
    _check(lib().cat_plan_create_2d(ctypes.byref(hd), B, h, w, D, H, dtype_code(dtype),
                                    _stream(stream)), "cat_plan_create_2d")
    return hd.value


def cat2d_forward(plan, Q, K, V, O, B, h, w, D, H, dtype):
    _check(lib().cat2d_forward(plan, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), B, h, w, D, H,
                               dtype_code(dtype)), "cat2d_forward")


def cat2d_scores(plan, Q, K, a, B, h, w, D, H, dtype):
    _check(lib().cat2d_scores(plan, _ptr(Q), _ptr(K), _ptr(a), B, h, w, D, H,
                              dtype_code(dtype)), "cat2d_scores")


def cat_plan_sync(plan):
    _check(lib().cat_plan_sync(plan), "cat_plan_sync")


def cat_plan_timing(plan, max_calls):
    _check(lib().cat_plan_timing(plan, max_calls), "cat_plan_timing")


def cat_plan_stage_times(plan):
    """(ms per stage [score, softmax/spectrum, circulant product], calls)."""
    ms = (ctypes.c_float * 3)()
    n = ctypes.c_int(0)
    _check(lib().cat_plan_stage_times(plan, ms, 3, ctypes.byref(n)), "cat_plan_stage_times")
    return [float(v) for v in ms], n.value


def cat_plan_pass_times(plan):
    """(ms of passes A, B, C summed over recorded chunks, launches of each)."""
    ms = (ctypes.c_float * 3)()
    n = ctypes.c_int(0)
    _check(lib().cat_plan_pass_times(plan, ms, 3, ctypes.byref(n)), "cat_plan_pass_times")
    return [float(v) for v in ms], n.value


def cat_plan_describe(plan):
    buf = ctypes.create_string_buffer(512)
    _check(lib().cat_plan_describe(plan, buf, 512), "cat_plan_describe")
    return buf.value.decode()


class Plan:
    """Owns one libcat plan for a fixed (B, N, D, H, dtype).

    ``forward(X, W_A, V, O=None)`` takes CUDA tensors of the plan's dtype
    (X, V, O: [B, N, D]; W_A: [D, H]) and enqueues the forward on the plan's
    stream (torch's current stream when the plan was made, unless given).
    """

    def __init__(self, B, N, D, H, dtype, stream=None):
        import torch
        self.B, self.N, self.D, self.H = B, N, D, H
        self.dtype = dtype_code(dtype)
        self.torch_dtype = torch.bfloat16 if self.dtype == CAT_BF16 else torch.float32
        if stream is None and torch.cuda.is_available():
            stream = torch.cuda.current_stream()
        self.handle = cat_plan_create(B, N, D, H, self.dtype, stream)

    def _shape(self):
        return (self.B, self.N, self.D, self.H, self.dtype)

    def forward(self, X, W_A, V, O=None):
        import torch
        if O is None:
            O = torch.empty_like(V)
        for t in (X, W_A, V, O):
            if not t.is_contiguous() or t.dtype != self.torch_dtype:
                raise ValueError("tensors must be contiguous %s" % self.torch_dtype)
        cat_forward(self.handle, X, W_A, V, O, *self._shape())
        return O

    def forward_fused(self, X, W_V, W_A, V=None, O=None):
        """V = X·W_V and the scores from one pass over X (tensor cores), then
        the forward; returns (V, O)."""
        import torch
        V = torch.empty_like(X) if V is None else V
        O = torch.empty_like(X) if O is None else O
        for t in (X, W_V, W_A, V, O):
            if not t.is_contiguous() or t.dtype != self.torch_dtype:
                raise ValueError("tensors must be contiguous %s" % self.torch_dtype)
        cat_forward_fused(self.handle, X, W_V, W_A, V, O, *self._shape())
        return V, O

    def project(self, X, W_V, W_A):
        """The fused projection alone: returns (V, z*)."""
        import torch
        V = torch.empty_like(X)
        zs = torch.empty((self.B, self.H, self.N), dtype=torch.float32, device=X.device)
        cat_project(self.handle, X, W_V, W_A, V, zs, *self._shape())
        return V, zs

    def zstar(self, X, W_A, out=None):
        import torch
        if out is None:
            out = torch.empty((self.B, self.H, self.N), dtype=torch.float32, device=X.device)
        cat_forward_zstar(self.handle, X, W_A, out, *self._shape())
        return out

    def backward(self, X, W_A, V, dO, dX=None, dW_A=None, dV=None):
        """Gradients (dX, dW_A, dV) for the upstream gradient dO = dL/dO."""
        import torch
        dX = torch.empty_like(X) if dX is None else dX
        dW_A = torch.empty_like(W_A) if dW_A is None else dW_A
        dV = torch.empty_like(V) if dV is None else dV
        for t in (X, W_A, V, dO, dX, dW_A, dV):
            if not t.is_contiguous() or t.dtype != self.torch_dtype:
                raise ValueError("tensors must be contiguous %s" % self.torch_dtype)
        cat_backward(self.handle, X, W_A, V, dO, dX, dW_A, dV, *self._shape())
        return dX, dW_A, dV

    def backward_dz(self, X, W_A, V, dO):
        """(dL/dz*, dL/dz), each fp32 [B, H, N]."""
        import torch
        shape = (self.B, self.H, self.N)
        dzs = torch.empty(shape, dtype=torch.float32, device=X.device)
        dz = torch.empty(shape, dtype=torch.float32, device=X.device)
        cat_backward_dz(self.handle, X, W_A, V, dO, dzs, dz, *self._shape())
        return dzs, dz

    def forward_host(self, X, W_A, V, O):
        cat_forward_host(self.handle, X, W_A, V, O, *self._shape())
        return O

    def sync(self):
        cat_plan_sync(self.handle)

    def describe(self):
        return cat_plan_describe(self.handle)

    def timing(self, max_calls):
        cat_plan_timing(self.handle, max_calls)

    def stage_times(self):
        return cat_plan_stage_times(self.handle)

    def pass_times(self):
        return cat_plan_pass_times(self.handle)

    def close(self):
        if self.handle:
            cat_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Plan2D:
    """Owns one 2-D circulant-attention plan for a fixed (B, h, w, D, H, dtype):
    ``forward(Q, K, V, O=None)`` with CUDA tensors [B, h·w, D] of the plan's
    dtype; ``scores(Q, K)`` returns the fp32 scores a [B, H, h·w]."""

    def __init__(self, B, h, w, D, H, dtype, stream=None):
        import torch
        self.B, self.h, self.w, self.D, self.H = B, h, w, D, H
        self.dtype = dtype_code(dtype)
        self.torch_dtype = torch.bfloat16 if self.dtype == CAT_BF16 else torch.float32
        if stream is None and torch.cuda.is_available():
            stream = torch.cuda.current_stream()
        self.handle = cat_plan_create_2d(B, h, w, D, H, self.dtype, stream)

    def _shape(self):
        return (self.B, self.h, self.w, self.D, self.H, self.dtype)

    def forward(self, Q, K, V, O=None):
        import torch
        if O is None:
            O = torch.empty_like(V)
        for t in (Q, K, V, O):
            if not t.is_contiguous() or t.dtype != self.torch_dtype:
                raise ValueError("tensors must be contiguous %s" % self.torch_dtype)
        cat2d_forward(self.handle, Q, K, V, O, *self._shape())
        return O

    def scores(self, Q, K):
        import torch
        a = torch.empty((self.B, self.H, self.h * self.w), dtype=torch.float32, device=Q.device)
        cat2d_scores(self.handle, Q, K, a, *self._shape())
        return a

    def sync(self):
        cat_plan_sync(self.handle)

    def describe(self):
        return cat_plan_describe(self.handle)

    def close(self):
        if self.handle:
            cat_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


__all__ = ["CatError", "Plan", "Plan2D", "lib", "dtype_code", "cat_plan_create", "cat_plan_destroy",
           "cat_plan_set_stream", "cat_forward", "cat_forward_zstar", "cat_forward_host",
           "cat_plan_sync", "cat_plan_describe", "cat_plan_timing", "cat_plan_stage_times",
           "cat_plan_pass_times", "cat_forward_noalloc", "cat_backward", "cat_backward_dz",
           "cat_plan_create_2d", "cat2d_forward", "cat2d_scores", "cat_plan_query",
           "cat_status_string", "CAT_F32", "CAT_BF16",
           "SIGNATURES", "LIB_PATH"]
