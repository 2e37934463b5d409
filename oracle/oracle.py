"""ctypes binding of the fp64 C oracle (gr_oracle.c). Test infrastructure only."""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gr_oracle.c")
_SO = os.path.join(_HERE, "libgr_oracle.so")
_LOCK = threading.Lock()
_LIB = None


def _stamp() -> str:
    import hashlib
    import platform
    h = hashlib.sha256(platform.machine().encode())
    with open(_SRC, "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile gr_oracle.c into a shared library beside it (gcc, OpenMP, no fast-math). A
    library built from other sources or on another machine is rebuilt."""
    stamp = _SO + ".stamp"
    fresh = (os.path.exists(_SO) and os.path.exists(stamp)
             and open(stamp).read().strip() == _stamp())
    if force or not fresh:
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
        with open(stamp, "w") as f:
            f.write(_stamp() + "\n")
    return _SO


def _load(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    P = ctypes.POINTER(ctypes.c_double)
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    L.gro_read.argtypes = [i64, i32, i32, i32, f64, P, P, P, P, P, P, P, P, P]
    L.gro_write.argtypes = [i64, i32, i32, P, P, P, P]
    L.gro_write_then_read.argtypes = [i64, i32, i32, i32, f64, P, P, P, P, P, P, P, P, P, P]
    L.gro_read_fixed_gates.argtypes = [i64, i32, i32, f64, P, P, P, P]
    L.gro_residual_add.argtypes = [i64, P, P]
    L.gro_round_significand.argtypes = [i64, i32, P]
    L.gro_num_threads.argtypes = []
    L.gro_set_num_threads.argtypes = [i32]
    L.gro_set_num_threads.restype = None
    U = ctypes.POINTER(ctypes.c_uint8)
    L.gro_read_backward.argtypes = [i64, i32, i32, i32, f64] + [P] * 12
    L.gro_write_backward.argtypes = [i64, i32, i32, P, P, P, P, P, P]
    L.gro_fp8_encode.argtypes = [i64, i32, P, U, U]
    L.gro_fp8_decode.argtypes = [i64, i32, U, U, P]
    L.gro_fp8_code_values.argtypes = [P]
    L.gro_fp8_round_codes.argtypes = [i64, P, U]
    L.gro_decompose.argtypes = [i64, i32, i32, i32, f64, P, P, P, P, P, i32, P, P, P, P, P, P,
                                P, P, P]
    for f in ("gro_read", "gro_write", "gro_write_then_read", "gro_read_fixed_gates",
              "gro_residual_add", "gro_num_threads", "gro_round_significand", "gro_fp8_encode",
              "gro_read_backward", "gro_write_backward", "gro_decompose",
              "gro_fp8_decode", "gro_fp8_code_values", "gro_fp8_round_codes"):
        getattr(L, f).restype = ctypes.c_int
    return L


def lib() -> ctypes.CDLL:
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            _LIB = _load(_SO)
    return _LIB


@contextlib.contextmanager
def use_library(path: str):
    """Run the functions of this module against another build of the oracle source (the
    tests use it to check that deliberately broken copies fail the pins)."""
    global _LIB
    old = lib()
    _LIB = _load(path)
    try:
        yield
    finally:
        _LIB = old


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _pu8(a: np.ndarray):
    assert a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _check(st: int, what: str) -> None:
    if st != 0:
        raise RuntimeError(f"oracle {what} failed with status {st}")


def num_threads() -> int:
    return int(lib().gro_num_threads())


def set_num_threads(k: int) -> None:
    lib().gro_set_num_threads(int(k))


def read(R, gamma, w_down, w_up, w_write, eps: float = 1e-6, return_internals: bool = False):
    """gr_read. R [n, nb, D] -> x [n, D], s [n, nb] (and G [n, nb, D], inv [n, nb])."""
    R = _f64(R)
    n, nb, D = R.shape
    Wd = _f64(w_down)
    r = Wd.shape[0]
    gamma, Wu, Ww = _f64(gamma), _f64(w_up), _f64(w_write)
    assert gamma.shape == (nb, D) and Wd.shape == (r, nb * D)
    assert Wu.shape == (nb * D, r) and Ww.shape == (nb, nb * D)
    x = np.empty((n, D))
    s = np.empty((n, nb))
    G = np.empty((n, nb, D)) if return_internals else None
    inv = np.empty((n, nb)) if return_internals else None
    _check(lib().gro_read(n, nb, D, r, float(eps), _p(R), _p(gamma), _p(Wd), _p(Wu), _p(Ww),
                          _p(x), _p(s), _p(G), _p(inv)), "read")
    if return_internals:
        return x, s, G, inv
    return x, s


def write(R, y, s):
    """gr_write. R' = R + s_i y for every branch i."""
    R, y, s = _f64(R), _f64(y), _f64(s)
    n, nb, D = R.shape
    assert y.shape == (n, D) and s.shape == (n, nb)
    out = np.empty_like(R)
    _check(lib().gro_write(n, nb, D, _p(R), _p(y), _p(s), _p(out)), "write")
    return out


_STORE_BITS = {"bf16": 8, "f32": 24}


def round_to_storage(a, dtype: str):
    """Nearest value representable in the storage format (bf16: 8 significant bits, f32: 24),
    ties to even, as a new float64 array."""
    out = _f64(a).copy()
    _check(lib().gro_round_significand(out.size, _STORE_BITS[dtype], _p(out)), "round")
    return out


def write_then_read(R, y, s_prev, params: dict, eps: float = 1e-6, store: str | None = None):
    """Fused step: the write with s_prev, then the read with ``params`` (keys gamma, w_down,
    w_up, w_write). Returns (R', x, s_next).

    store=None keeps R' in fp64 and reads it as is (the plain definition). store="bf16" or
    "f32" models the library's storage: the sum R + s·y is formed in fp32 (one rounding, as a
    fused multiply-add does), stored in that format (a second rounding for bf16), and the read
    sees the stored value."""
    R, y, s_prev = _f64(R), _f64(y), _f64(s_prev)
    n, nb, D = R.shape
    gamma, Wd, Wu, Ww = (_f64(params[k]) for k in ("gamma", "w_down", "w_up", "w_write"))
    r = Wd.shape[0]
    if store is not None:
        Rw = round_to_storage(round_to_storage(write(R, y, s_prev), "f32"), store)
        x, s = read(Rw, gamma, Wd, Wu, Ww, eps)
        return Rw, x, s
    R_out = np.empty_like(R)
    x = np.empty((n, D))
    s = np.empty((n, nb))
    _check(lib().gro_write_then_read(n, nb, D, r, float(eps), _p(R), _p(y), _p(s_prev),
                                     _p(gamma), _p(Wd), _p(Wu), _p(Ww), _p(R_out), _p(x), _p(s)),
           "write_then_read")
    return R_out, x, s


# ---- backward ---------------------------------------------------------------------------------

def read_backward(R, params: dict, dx, ds, eps: float = 1e-6):
    """Gradients of the read given dL/dx [n, D] and dL/ds [n, nb]: returns dR [n, nb, D] and a
    dict of parameter gradients (gamma, w_down, w_up, w_write), summed over the tokens."""
    R = _f64(R)
    n, nb, D = R.shape
    gamma, Wd, Wu, Ww = (_f64(params[k]) for k in ("gamma", "w_down", "w_up", "w_write"))
    r = Wd.shape[0]
    dx, ds = _f64(dx), _f64(ds)
    assert dx.shape == (n, D) and ds.shape == (n, nb)
    dR = np.empty_like(R)
    out = {"gamma": np.empty((nb, D)), "w_down": np.empty((r, nb * D)),
           "w_up": np.empty((nb * D, r)), "w_write": np.empty((nb, nb * D))}
    _check(lib().gro_read_backward(n, nb, D, r, float(eps), _p(R), _p(gamma), _p(Wd), _p(Wu),
                                   _p(Ww), _p(dx), _p(ds), _p(dR), _p(out["gamma"]),
                                   _p(out["w_down"]), _p(out["w_up"]), _p(out["w_write"])),
           "read_backward")
    return dR, out


def write_backward(dRp, y, s):
    """Gradients of the write R' = R + s_i y given dL/dR': returns (dR, dy, ds)."""
    dRp, y, s = _f64(dRp), _f64(y), _f64(s)
    n, nb, D = dRp.shape
    dR, dy, ds = np.empty_like(dRp), np.empty((n, D)), np.empty((n, nb))
    _check(lib().gro_write_backward(n, nb, D, _p(dRp), _p(y), _p(s), _p(dR), _p(dy), _p(ds)),
           "write_backward")
    return dR, dy, ds


# ---- contribution decomposition ---------------------------------------------------------------

def decompose(R, params: dict, ys, ss, eps: float = 1e-6, R0=None, vectors: bool = False):
    """eq auv at reader v: R [n, nb, D] the state the reader reads, ``params`` its parameters,
    ys [U, n, D] and ss [U, n, nb] the writers' outputs and write strengths, R0 [n, nb, D] the
    initial state (optional). Returns a dict with norm [n, U] (‖a_{u→v}‖ per token), bnorm
    [n, U, nb] (per branch), pi [n, U], and with R0 a0_norm [n]; with ``vectors`` also A
    [n, U, D] (the vectors a_{u→v}) and, with R0, A0 [n, D]."""
    R = _f64(R)
    n, nb, D = R.shape
    gamma, Wd, Wu, Ww = (_f64(params[k]) for k in ("gamma", "w_down", "w_up", "w_write"))
    r = Wd.shape[0]
    ys = _f64(ys).reshape(-1, n, D)
    ss = _f64(ss).reshape(-1, n, nb)
    U = ys.shape[0]
    assert ss.shape[0] == U
    R0 = None if R0 is None else _f64(R0)
    assert R0 is None or R0.shape == R.shape
    out = {"norm": np.empty((n, U)), "bnorm": np.empty((n, U, nb)), "pi": np.empty((n, U))}
    if R0 is not None:
        out["a0_norm"] = np.empty(n)
    if vectors:
        out["A"] = np.empty((n, U, D))
        if R0 is not None:
            out["A0"] = np.empty((n, D))
    _check(lib().gro_decompose(n, nb, D, r, float(eps), _p(R), _p(gamma), _p(Wd), _p(Wu),
                               _p(Ww), U, _p(ys) if U else None, _p(ss) if U else None,
                               _p(R0), _p(out["norm"]), _p(out["bnorm"]), _p(out["pi"]),
                               _p(out.get("a0_norm")), _p(out.get("A")), _p(out.get("A0"))),
           "decompose")
    return out


# ---- FP8 state: e4m3 codes with one power-of-two scale per 32-channel block -----------------

def fp8_encode(V):
    """Encode a state [..., D] (D a multiple of 32; exact fp32 values) into e4m3 codes
    (uint8, same shape) and biased block exponents (uint8, [..., D/32]; scale 2^(b-127))."""
    V = _f64(V)
    D = V.shape[-1]
    rows = V.size // D if D else 0
    codes = np.empty(V.shape, dtype=np.uint8)
    scales = np.empty(V.shape[:-1] + (D // 32,), dtype=np.uint8)
    _check(lib().gro_fp8_encode(rows, D, _p(V), _pu8(codes), _pu8(scales)), "fp8_encode")
    return codes, scales


def fp8_decode(codes, scales):
    """Values of an FP8 state (codes [..., D], block exponents [..., D/32]) as float64."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    D = codes.shape[-1]
    assert scales.shape == codes.shape[:-1] + (D // 32,)
    out = np.empty(codes.shape, dtype=np.float64)
    _check(lib().gro_fp8_decode(codes.size // D if D else 0, D, _pu8(codes), _pu8(scales),
                                _p(out)), "fp8_decode")
    return out


def fp8_code_values():
    """The value of every e4m3 code 0..255 (NaN for 0x7F and 0xFF)."""
    out = np.empty(256)
    _check(lib().gro_fp8_code_values(_p(out)), "fp8_code_values")
    return out


def fp8_round_codes(w):
    """Nearest e4m3 code of each value (no block scale; |w| <= 448, ties to even)."""
    w = _f64(w)
    codes = np.empty(w.shape, dtype=np.uint8)
    _check(lib().gro_fp8_round_codes(w.size, _p(w), _pu8(codes)), "fp8_round_codes")
    return codes


def write_then_read_fp8(codes, scales, y, s_prev, params: dict, eps: float = 1e-6):
    """Fused step on an FP8 state, modelling the storage: the write decodes R, forms R + s·y
    with one fp32 rounding (as a fused multiply-add does), encodes the result block by block,
    and the read sees the decoded stored values. Returns (codes', scales', x, s_next)."""
    R = fp8_decode(codes, scales)
    W = round_to_storage(write(R, y, s_prev), "f32")
    c2, b2 = fp8_encode(W)
    p = params
    x, s = read(fp8_decode(c2, b2), p["gamma"], p["w_down"], p["w_up"], p["w_write"], eps)
    return c2, b2, x, s


def read_fixed_gates(R, gamma, G, eps: float = 1e-6):
    """x = (1/nb) sum_i G_i * RMSNorm(R_i; gamma_i) with given gates G [nb, D]."""
    R, gamma, G = _f64(R), _f64(gamma), _f64(G)
    n, nb, D = R.shape
    assert gamma.shape == (nb, D) and G.shape == (nb, D)
    x = np.empty((n, D))
    _check(lib().gro_read_fixed_gates(n, nb, D, float(eps), _p(R), _p(gamma), _p(G), _p(x)),
           "read_fixed_gates")
    return x


def residual_add(x, y):
    """Single-stream x + y."""
    x = _f64(x).copy()
    y = _f64(y)
    assert x.shape == y.shape
    _check(lib().gro_residual_add(x.size, _p(y), _p(x)), "residual_add")
    return x


def chain(R0, ys, params_list, eps: float = 1e-6):
    """A stack of sublayers: read with params_list[0], then for l = 1..L-1 the fused write of
    y_{l-1} with s_{l-1} followed by the read with params_list[l], then the final write of
    y_{L-1}. Returns the states before every read and after the last write (L+1 states,
    fp64), the block inputs x_l and the write strengths s_l."""
    L = len(params_list)
    assert len(ys) == L
    states = [_f64(R0)]
    xs, ss = [], []
    p0 = params_list[0]
    x, s = read(states[0], p0["gamma"], p0["w_down"], p0["w_up"], p0["w_write"], eps)
    xs.append(x)
    ss.append(s)
    for l in range(1, L):
        R, x, s = write_then_read(states[-1], ys[l - 1], ss[-1], params_list[l], eps)
        states.append(R)
        xs.append(x)
        ss.append(s)
    states.append(write(states[-1], ys[L - 1], ss[-1]))
    return states, xs, ss
