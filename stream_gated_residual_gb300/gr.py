"""Python binding of libgr_gb300.so: argument marshalling only.

Every step of the Gated Residual read/write runs in the library's CUDA kernels; this module
checks tensor devices, dtypes and contiguity, takes ``data_ptr()`` and the current CUDA stream,
calls the C entry point of the same name and raises ``GRError`` on a non-zero status. PyTorch
supplies device memory and streams. There is no fallback: if the library is missing, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

GR_F32, GR_BF16, GR_FP8 = 0, 1, 2
GR_PARAMS_TAG = 0x47523330304B5031

_DTYPES = {torch.float32: GR_F32, torch.bfloat16: GR_BF16}
# The FP8 branch state is named by torch's e4m3 dtype in shapes and parameter packing; the state
# itself is a pair of uint8 tensors (codes [N,4,D], block exponents [N,4,D/32]).
FP8 = torch.float8_e4m3fn
_SHAPE_DTYPES = {**_DTYPES, FP8: GR_FP8}


class GRError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


class Shape(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("d_model", ctypes.c_int32),
                ("n_branch", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32), ("eps", ctypes.c_float)]


class ParamsStruct(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("d_model", ctypes.c_int32),
                ("n_branch", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("state_dtype", ctypes.c_int32), ("tag", ctypes.c_uint64)]


_LIB = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgr_gb300.so (built by ``__graft_entry__.build()``); raise if it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"{_build.LIB} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(_build.LIB)
    P, S, V = ctypes.POINTER(ParamsStruct), ctypes.POINTER(Shape), ctypes.c_void_p
    sz = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "gr_api_version": ([], ctypes.c_int),
        "gr_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "gr_kernel_path": ([S], ctypes.c_char_p),
        "gr_packed_size": ([S, sz], ctypes.c_int),
        "gr_pack_params": ([S, V, V, V, V, V, ctypes.c_size_t, P, V], ctypes.c_int),
        "gr_read": ([S, V, P, V, V, V], ctypes.c_int),
        "gr_read_ws": ([S, V, P, V, V, V, ctypes.c_size_t, V], ctypes.c_int),
        "gr_step_workspace_size": ([S, sz], ctypes.c_int),
        "gr_write_then_read_ws": ([S, V, V, V, P, V, V, V, ctypes.c_size_t, V], ctypes.c_int),
        "gr_write": ([S, V, V, V, V], ctypes.c_int),
        "gr_write_then_read": ([S, V, V, V, P, V, V, V], ctypes.c_int),
        "gr_read_fixed_gates": ([S, V, V, V, V, V], ctypes.c_int),
        "gr_residual_add_ref": ([ctypes.c_int64, ctypes.c_int32, V, V, V], ctypes.c_int),
        "gr_host_workspace_size": ([S, sz], ctypes.c_int),
        "gr_device_status": ([ctypes.c_int], ctypes.c_int),
        "gr_write_then_read_host": ([S, V, V, V, P, V, V, V, ctypes.c_size_t, V], ctypes.c_int),
        "gr_write_then_read_host_static": ([S, V, V, V, P, V, V, V], ctypes.c_int),
        "gr_selftest_bounded_wait": ([ctypes.c_int64, V], ctypes.c_int),
        "gr_read_backward_workspace_size": ([S, sz], ctypes.c_int),
        "gr_read_backward": ([S] + [V] * 13 + [ctypes.c_size_t, V], ctypes.c_int),
        "gr_write_backward": ([S, V, V, V, V, V, V, V], ctypes.c_int),
        "gr_decompose": ([S, V, V, V, V, V, ctypes.c_int32, V, V, V, V, V, V, V, V],
                         ctypes.c_int),
        "gr_fp8_encode": ([S, V, ctypes.c_int32, V, V, V], ctypes.c_int),
        "gr_fp8_decode": ([S, V, V, V, ctypes.c_int32, V], ctypes.c_int),
        "gr_read_fp8": ([S, V, V, P, V, V, V], ctypes.c_int),
        "gr_write_fp8": ([S, V, V, V, V, V], ctypes.c_int),
        "gr_write_then_read_fp8": ([S, V, V, V, V, P, V, V, V], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _LIB = L
    return L


def status_string(status: int) -> str:
    return load().gr_status_string(int(status)).decode()


def kernel_path(n_tokens: int, d_model: int, rank: int, dtype: torch.dtype) -> str:
    """Which kernel a read or fused step of this shape runs ("fused_bf16",
    "fused_bf16+tiled_bf16", "tiled_bf16", "tc_bf16" (the large-rank path), "tiled_fp8" for
    dtype FP8, or "generic")."""
    return load().gr_kernel_path(ctypes.byref(make_shape(n_tokens, d_model, rank, dtype))).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise GRError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def _dev(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_shape(n_tokens: int, d_model: int, rank: int, dtype: torch.dtype,
               eps: float = 1e-6) -> Shape:
    if dtype not in _SHAPE_DTYPES:
        raise ValueError(f"state dtype must be float32, bfloat16 or FP8, got {dtype}")
    return Shape(int(n_tokens), int(d_model), 4, int(rank), _SHAPE_DTYPES[dtype], float(eps))


class Params:
    """One GR module's packed parameters: the device buffer and its ``gr_params`` record."""

    def __init__(self, buf: torch.Tensor, st: ParamsStruct, dtype: torch.dtype, eps: float):
        self.buffer = buf
        self.struct = st
        self.dtype = dtype
        self.eps = eps
        self.d_model = st.d_model
        self.rank = st.rank

    def ref(self):
        return ctypes.byref(self.struct)


def packed_size(d_model: int, rank: int, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gr_packed_size(ctypes.byref(make_shape(0, d_model, rank, dtype)),
                                 ctypes.byref(n)), "gr_packed_size")
    return n.value


def pack_params(gamma: torch.Tensor, w_down: torch.Tensor, w_up: torch.Tensor,
                w_write: torch.Tensor, dtype: torch.dtype, eps: float = 1e-6,
                stream=None) -> Params:
    """gr_pack_params: fp32 CUDA tensors gamma [4,D], W_d [r,4D], W_u [4D,r], W_w [4,4D]."""
    for t, n in ((gamma, "gamma"), (w_down, "w_down"), (w_up, "w_up"), (w_write, "w_write")):
        _dev(t, n)
        if t.dtype != torch.float32:
            raise ValueError(f"{n} must be float32")
    r, K = w_down.shape
    D = K // 4
    if tuple(gamma.shape) != (4, D) or tuple(w_up.shape) != (K, r) or \
            tuple(w_write.shape) != (4, K):
        raise ValueError("parameter shapes must be gamma [4,D], W_d [r,4D], W_u [4D,r], "
                         "W_w [4,4D]")
    shape = make_shape(0, D, r, dtype, eps)
    nbytes = packed_size(D, r, dtype)
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=gamma.device)
    off = (-buf.data_ptr()) % 256
    view = buf[off:off + nbytes]
    st = ParamsStruct()
    _check(load().gr_pack_params(ctypes.byref(shape), _ptr(gamma), _ptr(w_down), _ptr(w_up),
                                 _ptr(w_write), _ptr(view), nbytes, ctypes.byref(st),
                                 _stream(stream)), "gr_pack_params")
    p = Params(view, st, dtype, eps)
    p._keep = buf
    return p


def _state_shape(R: torch.Tensor, params_or_rank, eps: float) -> Shape:
    _dev(R, "R")
    if R.dim() != 3 or R.shape[1] != 4:
        raise ValueError("R must have shape [N, 4, D]")
    rank = params_or_rank.rank if isinstance(params_or_rank, Params) else int(params_or_rank)
    return make_shape(R.shape[0], R.shape[2], rank, R.dtype, eps)


def step_workspace_size(n_tokens: int, d_model: int, rank: int, dtype: torch.dtype) -> int:
    """gr_step_workspace_size: device bytes a read or fused step of this shape needs (0 except on
    the large-rank path)."""
    need = ctypes.c_size_t(0)
    shape = make_shape(n_tokens, d_model, rank, dtype)
    _check(load().gr_step_workspace_size(ctypes.byref(shape), ctypes.byref(need)),
           "gr_step_workspace_size")
    return need.value


def _step_ws(shape: Shape, device, workspace):
    """(pointer, bytes) of the step's workspace: the caller's, else a fresh 256-byte aligned
    buffer when the shape needs one."""
    need = ctypes.c_size_t(0)
    _check(load().gr_step_workspace_size(ctypes.byref(shape), ctypes.byref(need)),
           "gr_step_workspace_size")
    if workspace is not None:
        _dev(workspace, "workspace")
        return _ptr(workspace), workspace.numel() * workspace.element_size(), workspace
    if need.value == 0:
        return ctypes.c_void_p(None), 0, None
    buf = torch.empty(need.value + 256, dtype=torch.uint8, device=device)
    view = buf[(-buf.data_ptr()) % 256:][:need.value]
    return _ptr(view), need.value, buf


def read(R: torch.Tensor, params: Params, x: torch.Tensor | None = None,
         s: torch.Tensor | None = None, stream=None, workspace: torch.Tensor | None = None):
    """gr_read (through gr_read_ws): R [N,4,D] -> (x [N,D], s [N,4] fp32). The large-rank path
    needs a device workspace: the caller's (256-byte aligned), else one allocated here."""
    shape = _state_shape(R, params, params.eps)
    N, _, D = R.shape
    x = torch.empty((N, D), dtype=R.dtype, device=R.device) if x is None else x
    s = torch.empty((N, 4), dtype=torch.float32, device=R.device) if s is None else s
    _dev(x, "x")
    _dev(s, "s")
    wp, wn, keep = _step_ws(shape, R.device, workspace)
    _check(load().gr_read_ws(ctypes.byref(shape), _ptr(R), params.ref(), _ptr(x), _ptr(s), wp,
                             wn, _stream(stream)), "gr_read")
    if keep is not None and stream is not None:
        keep.record_stream(stream)   # the allocator may hand it out again only after `stream`
    return x, s


def write(R: torch.Tensor, y: torch.Tensor, s: torch.Tensor, stream=None) -> torch.Tensor:
    """gr_write: R += s_i y in place; returns R."""
    shape = _state_shape(R, 1, 1e-6)
    _dev(y, "y")
    _dev(s, "s")
    _check(load().gr_write(ctypes.byref(shape), _ptr(R), _ptr(y), _ptr(s), _stream(stream)),
           "gr_write")
    return R


def write_then_read(R: torch.Tensor, y: torch.Tensor, s_prev: torch.Tensor, params: Params,
                    x: torch.Tensor | None = None, s_next: torch.Tensor | None = None,
                    stream=None, workspace: torch.Tensor | None = None):
    """gr_write_then_read (through gr_write_then_read_ws): R += s_prev_i y in place, then
    (x, s_next) = read(R, params). Workspace as for read()."""
    shape = _state_shape(R, params, params.eps)
    N, _, D = R.shape
    x = torch.empty((N, D), dtype=R.dtype, device=R.device) if x is None else x
    s_next = torch.empty((N, 4), dtype=torch.float32, device=R.device) if s_next is None \
        else s_next
    for t, n in ((y, "y"), (s_prev, "s_prev"), (x, "x"), (s_next, "s_next")):
        _dev(t, n)
    wp, wn, keep = _step_ws(shape, R.device, workspace)
    _check(load().gr_write_then_read_ws(ctypes.byref(shape), _ptr(R), _ptr(y), _ptr(s_prev),
                                        params.ref(), _ptr(x), _ptr(s_next), wp, wn,
                                        _stream(stream)), "gr_write_then_read")
    if keep is not None and stream is not None:
        keep.record_stream(stream)
    return x, s_next


def read_fixed_gates(R: torch.Tensor, gamma: torch.Tensor, G: torch.Tensor, eps: float = 1e-6,
                     x: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gr_read_fixed_gates: x = (1/4) sum_i G_i * RMSNorm(R_i; gamma_i)."""
    shape = _state_shape(R, 1, eps)
    N, _, D = R.shape
    x = torch.empty((N, D), dtype=R.dtype, device=R.device) if x is None else x
    for t, n in ((gamma, "gamma"), (G, "G"), (x, "x")):
        _dev(t, n)
    _check(load().gr_read_fixed_gates(ctypes.byref(shape), _ptr(R), _ptr(gamma), _ptr(G),
                                      _ptr(x), _stream(stream)), "gr_read_fixed_gates")
    return x


def residual_add_ref(x: torch.Tensor, y: torch.Tensor, stream=None) -> torch.Tensor:
    """gr_residual_add_ref: x += y (single stream), in place."""
    _dev(x, "x")
    _dev(y, "y")
    if x.dtype not in _DTYPES or y.dtype != x.dtype or x.numel() != y.numel():
        raise ValueError("x and y must have the same size and dtype (float32 or bfloat16)")
    _check(load().gr_residual_add_ref(x.numel(), _DTYPES[x.dtype], _ptr(y), _ptr(x),
                                      _stream(stream)), "gr_residual_add_ref")
    return x


def device_status(clear: bool = False) -> int:
    """gr_device_status: 0, or the status code of a bounded device-side wait that ran out."""
    return int(load().gr_device_status(1 if clear else 0))


def selftest_bounded_wait(limit_cycles: int, stream=None) -> None:
    """gr_selftest_bounded_wait: one device-side wait that nothing satisfies gives up after
    limit_cycles and sets the status that device_status() reports."""
    _check(load().gr_selftest_bounded_wait(int(limit_cycles), _stream(stream)),
           "gr_selftest_bounded_wait")


def host_workspace_size(n_tokens: int, d_model: int, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gr_host_workspace_size(ctypes.byref(make_shape(n_tokens, d_model, 1, dtype)),
                                         ctypes.byref(n)), "gr_host_workspace_size")
    return n.value


def write_then_read_host(R: torch.Tensor, y: torch.Tensor, s_prev: torch.Tensor,
                         params: Params, x: torch.Tensor, s_next: torch.Tensor,
                         workspace: torch.Tensor, stream=None):
    """gr_write_then_read_host on CPU tensors (pinned for asynchronous copies); `workspace` is
    a CUDA uint8 tensor of at least host_workspace_size() bytes, 256-byte aligned."""
    for t, n in ((R, "R"), (y, "y"), (s_prev, "s_prev"), (x, "x"), (s_next, "s_next")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    N, _, D = R.shape
    shape = make_shape(N, D, params.rank, R.dtype, params.eps)
    _check(load().gr_write_then_read_host(
        ctypes.byref(shape), _ptr(R), _ptr(y), _ptr(s_prev), params.ref(), _ptr(x), _ptr(s_next),
        _ptr(workspace), workspace.numel(), _stream(stream)), "gr_write_then_read_host")
    return x, s_next


def write_then_read_host_static(R: torch.Tensor, y: torch.Tensor, s_prev: torch.Tensor,
                                params: Params, x: torch.Tensor, s_next: torch.Tensor,
                                stream=None):
    """gr_write_then_read_host_static on CPU tensors (pinned for asynchronous copies), staged
    through the library's fixed 32 MiB device workspace (GR_STATIC_WORKSPACE_BYTES), for callers
    that cannot allocate device memory: a host program without a device allocator, a process
    whose device memory a pool already holds, or a decode loop that cannot afford the device-wide
    synchronisation of cudaFree. Nothing is allocated; shapes that need more than the workspace
    raise GR_E_SIZE, and calls must not overlap in time (they share the workspace)."""
    for t, n in ((R, "R"), (y, "y"), (s_prev, "s_prev"), (x, "x"), (s_next, "s_next")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    N, _, D = R.shape
    shape = make_shape(N, D, params.rank, R.dtype, params.eps)
    _check(load().gr_write_then_read_host_static(
        ctypes.byref(shape), _ptr(R), _ptr(y), _ptr(s_prev), params.ref(), _ptr(x), _ptr(s_next),
        _stream(stream)), "gr_write_then_read_host_static")
    return x, s_next


# ---- backward (training) ------------------------------------------------------------------------

def read_backward(R: torch.Tensor, gamma: torch.Tensor, w_down: torch.Tensor, w_up: torch.Tensor,
                  w_write: torch.Tensor, dx: torch.Tensor, ds: torch.Tensor, eps: float = 1e-6,
                  workspace: torch.Tensor | None = None, stream=None):
    """gr_read_backward: dL/dR [N,4,D] fp32 and the parameter gradients (dict like the
    parameters: gamma, w_down, w_up, w_write; fp32) given dL/dx [N,D] and dL/ds [N,4] (fp32).
    The parameters are the fp32 tensors (not the packed buffer)."""
    _dev(R, "R")
    N, _, D = R.shape
    r = w_down.shape[0]
    shape = make_shape(N, D, r, R.dtype, eps)
    for t, n in ((gamma, "gamma"), (w_down, "w_down"), (w_up, "w_up"), (w_write, "w_write"),
                 (dx, "dx"), (ds, "ds")):
        _dev(t, n)
        if t.dtype != torch.float32:
            raise ValueError(f"{n} must be float32")
    need = ctypes.c_size_t(0)
    _check(load().gr_read_backward_workspace_size(ctypes.byref(shape), ctypes.byref(need)),
           "gr_read_backward_workspace_size")
    if workspace is None:
        buf = torch.empty(need.value + 256, dtype=torch.uint8, device=R.device)
        workspace = buf[(-buf.data_ptr()) % 256:][:need.value]
    dev = R.device
    dR = torch.empty((N, 4, D), dtype=torch.float32, device=dev)
    g = {"gamma": torch.empty_like(gamma), "w_down": torch.empty_like(w_down),
         "w_up": torch.empty_like(w_up), "w_write": torch.empty_like(w_write)}
    _check(load().gr_read_backward(
        ctypes.byref(shape), _ptr(R), _ptr(gamma), _ptr(w_down), _ptr(w_up), _ptr(w_write),
        _ptr(dx), _ptr(ds), _ptr(dR), _ptr(g["gamma"]), _ptr(g["w_down"]), _ptr(g["w_up"]),
        _ptr(g["w_write"]), _ptr(workspace), workspace.numel(), _stream(stream)),
        "gr_read_backward")
    return dR, g


def write_backward(dR_next: torch.Tensor, y: torch.Tensor, s: torch.Tensor, stream=None):
    """gr_write_backward: (dR, dy, ds) from dL/dR' [N,4,D] fp32, y [N,D] (state dtype), s [N,4]."""
    for t, n in ((dR_next, "dR_next"), (y, "y"), (s, "s")):
        _dev(t, n)
    N, _, D = dR_next.shape
    shape = make_shape(N, D, 1, y.dtype)
    dR = torch.empty_like(dR_next)
    dy = torch.empty((N, D), dtype=torch.float32, device=dR_next.device)
    ds = torch.empty((N, 4), dtype=torch.float32, device=dR_next.device)
    _check(load().gr_write_backward(ctypes.byref(shape), _ptr(dR_next), _ptr(y), _ptr(s),
                                    _ptr(dR), _ptr(dy), _ptr(ds), _stream(stream)),
           "gr_write_backward")
    return dR, dy, ds


# ---- contribution decomposition ---------------------------------------------------------------

def decompose(R: torch.Tensor, gamma: torch.Tensor, w_down: torch.Tensor, w_up: torch.Tensor,
              w_write: torch.Tensor, y: torch.Tensor | None, s: torch.Tensor | None,
              R0: torch.Tensor | None = None, eps: float = 1e-6, branch_norm: bool = True,
              pi: bool = True, stream=None) -> dict:
    """gr_decompose at one reader: R [N,4,D] the state it reads, its fp32 parameters, the
    writers' outputs y [U,N,D] (state dtype) and write strengths s [U,N,4] (fp32), optionally
    the initial state R0 [N,4,D]. Returns fp32 tensors: norm [N,U], branch_norm [N,U,4] and pi
    [N,U] (when asked), a0_norm [N] (with R0)."""
    _dev(R, "R")
    N, _, D = R.shape
    r = w_down.shape[0]
    shape = make_shape(N, D, r, R.dtype, eps)
    for t, n in ((gamma, "gamma"), (w_down, "w_down"), (w_up, "w_up"), (w_write, "w_write")):
        _dev(t, n)
        if t.dtype != torch.float32:
            raise ValueError(f"{n} must be float32")
    U = 0 if y is None else y.shape[0]
    if U:
        _dev(y, "y")
        _dev(s, "s")
        if y.dtype != R.dtype or tuple(y.shape) != (U, N, D) or tuple(s.shape) != (U, N, 4) \
                or s.dtype != torch.float32:
            raise ValueError("y must be [U, N, D] in the state dtype and s [U, N, 4] float32")
    if R0 is not None:
        _dev(R0, "R0")
        if R0.dtype != R.dtype or R0.shape != R.shape:
            raise ValueError("R0 must match R")
    dev = R.device
    out = {"norm": torch.empty((N, U), dtype=torch.float32, device=dev)}
    if branch_norm:
        out["branch_norm"] = torch.empty((N, U, 4), dtype=torch.float32, device=dev)
    if pi:
        out["pi"] = torch.empty((N, U), dtype=torch.float32, device=dev)
    if R0 is not None:
        out["a0_norm"] = torch.empty((N,), dtype=torch.float32, device=dev)

    def p(k):
        t = out.get(k)
        return _ptr(t) if t is not None and t.numel() else None

    _check(load().gr_decompose(
        ctypes.byref(shape), _ptr(R), _ptr(gamma), _ptr(w_down), _ptr(w_up), _ptr(w_write), U,
        _ptr(y) if U else None, _ptr(s) if U else None, _ptr(R0) if R0 is not None else None,
        p("norm"), p("branch_norm"), p("pi"), p("a0_norm"), _stream(stream)), "gr_decompose")
    return out


# ---- FP8 branch state (e4m3 codes, one power-of-two exponent per 32-channel block) ------------

def _fp8_state(codes: torch.Tensor, scales: torch.Tensor):
    _dev(codes, "codes")
    _dev(scales, "scales")
    if codes.dtype != torch.uint8 or scales.dtype != torch.uint8:
        raise ValueError("codes and scales must be uint8")
    if codes.dim() != 3 or codes.shape[1] != 4 or codes.shape[2] % 32:
        raise ValueError("codes must have shape [N, 4, D] with D a multiple of 32")
    N, _, D = codes.shape
    if tuple(scales.shape) != (N, 4, D // 32):
        raise ValueError("scales must have shape [N, 4, D/32]")
    return N, D


def fp8_encode(R: torch.Tensor, codes: torch.Tensor | None = None,
               scales: torch.Tensor | None = None, stream=None):
    """gr_fp8_encode: a bf16 or fp32 state R [N,4,D] -> (codes [N,4,D], scales [N,4,D/32])."""
    _dev(R, "R")
    if R.dtype not in _DTYPES or R.dim() != 3 or R.shape[1] != 4:
        raise ValueError("R must be a float32 or bfloat16 tensor of shape [N, 4, D]")
    N, _, D = R.shape
    codes = torch.empty((N, 4, D), dtype=torch.uint8, device=R.device) if codes is None else codes
    scales = torch.empty((N, 4, D // 32), dtype=torch.uint8, device=R.device) if scales is None \
        else scales
    _fp8_state(codes, scales)
    shape = make_shape(N, D, 1, FP8)
    _check(load().gr_fp8_encode(ctypes.byref(shape), _ptr(R), _DTYPES[R.dtype], _ptr(codes),
                                _ptr(scales), _stream(stream)), "gr_fp8_encode")
    return codes, scales


def fp8_decode(codes: torch.Tensor, scales: torch.Tensor, dtype: torch.dtype = torch.float32,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gr_fp8_decode: (codes, scales) -> the state's values [N,4,D] in float32 or bfloat16."""
    N, D = _fp8_state(codes, scales)
    if dtype not in _DTYPES:
        raise ValueError("dtype must be float32 or bfloat16")
    out = torch.empty((N, 4, D), dtype=dtype, device=codes.device) if out is None else out
    _dev(out, "out")
    shape = make_shape(N, D, 1, FP8)
    _check(load().gr_fp8_decode(ctypes.byref(shape), _ptr(codes), _ptr(scales), _ptr(out),
                                _DTYPES[dtype], _stream(stream)), "gr_fp8_decode")
    return out


def read_fp8(codes: torch.Tensor, scales: torch.Tensor, params: Params,
             x: torch.Tensor | None = None, s: torch.Tensor | None = None, stream=None):
    """gr_read_fp8: FP8 state -> (x [N,D] bf16, s [N,4] fp32)."""
    N, D = _fp8_state(codes, scales)
    shape = make_shape(N, D, params.rank, FP8, params.eps)
    x = torch.empty((N, D), dtype=torch.bfloat16, device=codes.device) if x is None else x
    s = torch.empty((N, 4), dtype=torch.float32, device=codes.device) if s is None else s
    _dev(x, "x")
    _dev(s, "s")
    _check(load().gr_read_fp8(ctypes.byref(shape), _ptr(codes), _ptr(scales), params.ref(),
                              _ptr(x), _ptr(s), _stream(stream)), "gr_read_fp8")
    return x, s


def write_fp8(codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor, s: torch.Tensor,
              stream=None):
    """gr_write_fp8: R += s_i y on the FP8 state (y bf16 [N,D]), in place."""
    N, D = _fp8_state(codes, scales)
    _dev(y, "y")
    _dev(s, "s")
    shape = make_shape(N, D, 1, FP8)
    _check(load().gr_write_fp8(ctypes.byref(shape), _ptr(codes), _ptr(scales), _ptr(y), _ptr(s),
                               _stream(stream)), "gr_write_fp8")
    return codes, scales


def write_then_read_fp8(codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor,
                        s_prev: torch.Tensor, params: Params, x: torch.Tensor | None = None,
                        s_next: torch.Tensor | None = None, stream=None):
    """gr_write_then_read_fp8: the write in place on the FP8 state, then the read with
    `params` -> (x [N,D] bf16, s_next [N,4] fp32)."""
    N, D = _fp8_state(codes, scales)
    shape = make_shape(N, D, params.rank, FP8, params.eps)
    x = torch.empty((N, D), dtype=torch.bfloat16, device=codes.device) if x is None else x
    s_next = torch.empty((N, 4), dtype=torch.float32, device=codes.device) if s_next is None \
        else s_next
    for t, n in ((y, "y"), (s_prev, "s_prev"), (x, "x"), (s_next, "s_next")):
        _dev(t, n)
    _check(load().gr_write_then_read_fp8(ctypes.byref(shape), _ptr(codes), _ptr(scales), _ptr(y),
                                         _ptr(s_prev), params.ref(), _ptr(x), _ptr(s_next),
                                         _stream(stream)), "gr_write_then_read_fp8")
    return x, s_next

