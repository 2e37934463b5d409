"""Seeded synthetic inputs for the Gated Residual read/write.

This module only draws random numbers and rounds them to the storage dtype; it holds none of the
method's arithmetic. The CPU oracle and the CUDA path receive the same bytes from it.

Storage conventions of the returned arrays:
  * state-dtype arrays (R, y, x) are numpy ``uint16`` bf16 bit patterns for ``dtype == "bf16"``
    and ``float32`` for ``dtype == "f32"``; ``to_f64`` converts either exactly to float64;
  * parameters (gamma, W_d, W_u, W_w) and write strengths s are ``float32``. On bf16 workloads
    the weights are rounded to bf16-representable values, so packing them to bf16 is exact;
  * on FP8-state workloads (``dtype == "fp8"``) the state's values come as ``float32`` (the
    consumer encodes them into the FP8 state format), y is bf16 and the weights are
    bf16-representable, as on the bf16 path.

Shapes follow the library: R ``[N, 4, D]``, y ``[N, D]``, s ``[N, 4]``, gamma ``[4, D]``,
W_d ``[r, 4D]``, W_u ``[4D, r]``, W_w ``[4, 4D]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os

import numpy as np

N_BRANCH = 4

# independent random streams per array kind: default_rng([seed, kind, layer(, chunk)])
_K_STATE, _K_Y, _K_PARAMS, _K_S, _K_OUTLIER = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_tokens: int
    d_model: int
    rank: int
    dtype: str  # "f32", "bf16" or "fp8" (FP8 branch state; y and x bf16)
    y_std: float
    y_kind: str = "normal"  # "normal" or "t3" (Student-t with 3 degrees of freedom)
    branch_scales: tuple = (1.0, 1.0, 1.0, 1.0)
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    weight_std: float = 0.02
    n_sublayers: int = 1
    eps: float = 1e-6
    seed: int = 0

    @property
    def n_branch(self) -> int:
        return N_BRANCH

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def state_bytes_per_elem(self) -> int:
        return {"f32": 4, "bf16": 2, "fp8": 1}[self.dtype]

    @property
    def state_storage(self) -> str:
        """Storage of make_state's arrays: the FP8 state's source values come as fp32."""
        return "f32" if self.dtype == "fp8" else self.dtype

    @property
    def io_storage(self) -> str:
        """Storage of y and x: bf16 on the FP8 path."""
        return "bf16" if self.dtype == "fp8" else self.dtype


WORKLOADS = {
    # one read + one write of a small state, fp32 end to end
    "tiny_fp32": Workload("tiny_fp32", 64, 256, 8, "f32", y_std=1.0),
    # decode: batch 128, one token each
    "decode": Workload("decode", 128, 4096, 16, "bf16", y_std=0.5),
    # prefill: B=4, S=4096 flattened to N=16384 rows
    "prefill": Workload("prefill", 16384, 4096, 16, "bf16", y_std=0.5),
    # 48 layers x (token mixer, MLP) = 96 chained sublayers
    "deep_stack": Workload("deep_stack", 8192, 2048, 16, "bf16", y_std=0.1, n_sublayers=96),
    # prefill with the FP8 branch state (e4m3 codes + per-32-channel exponents; y, x bf16)
    "prefill_fp8": Workload("prefill_fp8", 16384, 4096, 16, "fp8", y_std=0.5),
    # the pages' own rank: d = 2560 with r = d/8 = 320 (Digest §二.4), prefill-sized batch
    "paper_rank": Workload("paper_rank", 16384, 2560, 320, "bf16", y_std=0.5),
    # skewed branch scales, 1% outlier channels x50, heavy-tailed y
    "large_skewed": Workload("large_skewed", 65536, 7168, 32, "bf16", y_std=0.5, y_kind="t3",
                             branch_scales=(0.1, 1.0, 10.0, 100.0), outlier_frac=0.01,
                             outlier_mult=50.0),
}


# ---------------------------------------------------------------------------------------------
# dtype helpers (bit manipulation only)

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16, nearest-even; returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 value, returned as float32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(a))


def to_storage(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(a32)
    raise ValueError(dtype)


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact float64 copy of a storage array (bf16 bits or float32)."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------------------------
# generators

CHUNK_ROWS = 1024  # rows per independent random stream (part of the recipe)


def _rng(w: Workload, kind: int, layer: int = 0, chunk: int | None = None):
    key = [w.seed, kind, layer] if chunk is None else [w.seed, kind, layer, chunk]
    return np.random.default_rng(key)


def _draw_rows(w: Workload, kind: int, layer: int, n_rows: int, row_shape: tuple, fill,
               dtype: str) -> np.ndarray:
    """Draw an [n_rows, *row_shape] array chunk by chunk: chunk q (rows q*CHUNK_ROWS ...) comes
    from its own stream default_rng([seed, kind, layer, q]) through ``fill(rng, rows)``
    (float32), then is rounded to the storage dtype. Chunks run on a thread pool; the result
    does not depend on the thread count, and the first n rows do not depend on n_rows."""
    itemsize = 2 if dtype == "bf16" else 4
    out = np.empty((n_rows,) + tuple(row_shape), dtype=np.uint16 if itemsize == 2 else np.float32)

    def one(q):
        a = q * CHUNK_ROWS
        b = min(n_rows, a + CHUNK_ROWS)
        vals = fill(_rng(w, kind, layer, q), b - a)
        out[a:b] = to_storage(vals, dtype)

    nchunks = (n_rows + CHUNK_ROWS - 1) // CHUNK_ROWS
    if nchunks <= 1:
        for q in range(nchunks):
            one(q)
    else:
        workers = min(nchunks, os.cpu_count() or 1, 32)
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(one, range(nchunks)))
    return out


def outlier_channels(w: Workload) -> np.ndarray:
    """The seeded fixed set of ceil(outlier_frac * D) channels scaled by outlier_mult."""
    k = int(math.ceil(w.outlier_frac * w.d_model)) if w.outlier_frac > 0 else 0
    if k == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(w, _K_OUTLIER).choice(w.d_model, size=k, replace=False))


def make_state(w: Workload, n_tokens: int | None = None) -> np.ndarray:
    """Initial residual state R [N, 4, D] in storage dtype: N(0,1) per branch, times the
    branch scale, times outlier_mult on the outlier channels (all tokens and branches)."""
    n = w.n_tokens if n_tokens is None else n_tokens
    scales = np.asarray(w.branch_scales, dtype=np.float32)
    ch = outlier_channels(w)

    def fill(rng, rows):
        R = rng.standard_normal((rows, N_BRANCH, w.d_model), dtype=np.float32)
        if np.any(scales != 1.0):
            R *= scales[None, :, None]
        if ch.size:
            R[:, :, ch] *= np.float32(w.outlier_mult)
        return R

    return _draw_rows(w, _K_STATE, 0, n, (N_BRANCH, w.d_model), fill, w.state_storage)


def make_y(w: Workload, layer: int = 0, n_tokens: int | None = None) -> np.ndarray:
    """Sublayer output y [N, D] in storage dtype: y_std * N(0,1), or y_std * Student-t(3)."""
    n = w.n_tokens if n_tokens is None else n_tokens
    if w.y_kind not in ("normal", "t3"):
        raise ValueError(w.y_kind)

    def fill(rng, rows):
        if w.y_kind == "normal":
            return rng.standard_normal((rows, w.d_model), dtype=np.float32) * np.float32(w.y_std)
        return (w.y_std * rng.standard_t(3, size=(rows, w.d_model))).astype(np.float32)

    return _draw_rows(w, _K_Y, layer, n, (w.d_model,), fill, w.io_storage)


def make_params(w: Workload, layer: int = 0, weight_mult: float = 1.0) -> dict:
    """Per-sublayer parameters: gains 1 (the workloads' branch scales act on the state, see
    make_state), W_d, W_u, W_w ~ N(0, weight_std) * weight_mult.
    On bf16 workloads the weights are rounded to bf16-representable float32 values."""
    rng = _rng(w, _K_PARAMS, layer)
    K = N_BRANCH * w.d_model
    std = w.weight_std * weight_mult
    Wd = (std * rng.standard_normal((w.rank, K))).astype(np.float32)
    Wu = (std * rng.standard_normal((K, w.rank))).astype(np.float32)
    Ww = (std * rng.standard_normal((N_BRANCH, K))).astype(np.float32)
    if w.dtype in ("bf16", "fp8"):
        Wd, Wu, Ww = round_to_bf16(Wd), round_to_bf16(Wu), round_to_bf16(Ww)
    gamma = np.ones((N_BRANCH, w.d_model), dtype=np.float32)
    return {"gamma": gamma, "w_down": Wd, "w_up": Wu, "w_write": Ww}


def make_random_gamma(w: Workload, layer: int = 0) -> np.ndarray:
    """Non-trivial gains (for tests): 1 + 0.25 N(0,1), bf16-representable."""
    rng = np.random.default_rng([w.seed, 17, layer])
    g = (1.0 + 0.25 * rng.standard_normal((N_BRANCH, w.d_model))).astype(np.float32)
    return round_to_bf16(g)


def make_s_prev(w: Workload, n_tokens: int | None = None) -> np.ndarray:
    """Write strengths of the previous sublayer, float32 [N, 4], uniform on (0.25, 1.75)
    (inside the (0, 2) range that 2·sigmoid produces)."""
    n = w.n_tokens if n_tokens is None else n_tokens
    rng = _rng(w, _K_S)
    return rng.uniform(0.25, 1.75, size=(n, N_BRANCH)).astype(np.float32)
