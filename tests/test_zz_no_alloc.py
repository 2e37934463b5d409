"""gr_write_then_read_host_static (the host-buffer step staged through the library's fixed device
workspace, for callers that cannot allocate device memory: a host program with no device
allocator, a process whose memory a pool already holds, a decode loop that cannot take
cudaFree's device-wide synchronisation) against gr_write_then_read_host (caller-provided
workspace): two fused steps in a
row, each fed with the previous step's R' and s, give bit-identical results. On a shape that
gr_write_then_read_host splits between the cluster kernel and the two-pass kernel, the static
entry runs the cluster kernel alone: R' is still bit-identical, x and s agree within the bf16
tolerance. The file is
collected last on purpose, so the static entry also runs after every other test has used the
library in the same process. Beside the comparison with the other host entry, the static entry's
two chained steps are checked directly against the fp64 oracle's chain of the same two steps
(per-row relative L2 within 1e-5 on the fp32 path, 2e-2 on bf16 states)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gr_testlib import TOL, params_to_torch, rel_rows, to_torch
from stream_gated_residual_gb300 import build as gbuild
from stream_gated_residual_gb300 import gr
from stream_gated_residual_gb300 import workloads as wl

TDT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _pinned(a):
    return to_torch(a, "cpu").pin_memory()


def _two_steps(entry, w, R0, y0, y1, s0, P):
    """Two chained host-buffer steps; returns (R, x, s) after each."""
    tdt = TDT[w.dtype]
    R = _pinned(R0)
    s = torch.from_numpy(s0).pin_memory()
    outs = []
    for y in (y0, y1):
        x = torch.empty((w.n_tokens, w.d_model), dtype=tdt).pin_memory()
        s_next = torch.empty((w.n_tokens, 4), dtype=torch.float32).pin_memory()
        entry(R, _pinned(y), s, P, x, s_next)
        outs.append((R.clone(), x.clone(), s_next.clone()))
        s = s_next
    return outs


def _compare(N, D, r, dtype):
    w = wl.Workload("noalloc", N, D, r, dtype, y_std=0.5, seed=23)
    R0, s0 = wl.make_state(w), wl.make_s_prev(w)
    y0, y1 = wl.make_y(w, 0), wl.make_y(w, 1)
    t = params_to_torch(wl.make_params(w, 1))
    P = gr.pack_params(t["gamma"], t["w_down"], t["w_up"], t["w_write"], TDT[dtype], w.eps)
    nws = gr.host_workspace_size(N, D, TDT[dtype])
    buf = torch.empty(nws + 256, dtype=torch.uint8, device="cuda")
    ws = buf[(-buf.data_ptr()) % 256:][:nws]

    def with_workspace(R, y, s, P, x, sn):
        gr.write_then_read_host(R, y, s, P, x, sn, ws)

    def static(R, y, s, P, x, sn):
        gr.write_then_read_host_static(R, y, s, P, x, sn)

    split = gr.kernel_path(N, D, r, TDT[dtype]) == "fused_bf16+tiled_bf16"
    ref = _two_steps(with_workspace, w, R0, y0, y1, s0, P)
    got = _two_steps(static, w, R0, y0, y1, s0, P)
    for i, ((Ra, xa, sa), (Rb, xb, sb)) in enumerate(zip(ref, got)):
        if split and i > 0:
            # the second write uses each entry's own s from the first step
            assert rel_rows(Rb.float().numpy(), Ra.float().numpy()) <= TOL[dtype]
        else:
            assert torch.equal(Ra, Rb)
        if split:
            assert rel_rows(xb.float().numpy(), xa.float().numpy()) <= TOL[dtype]
            assert rel_rows(sb.numpy(), sa.numpy()) <= TOL[dtype]
        else:
            assert torch.equal(xa, xb) and torch.equal(sa, sb)
    assert gr.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,r,dtype", [(128, 4096, 16, "bf16"), (64, 256, 8, "f32"),
                                         (1500, 1024, 16, "bf16")])
def test_static_workspace_entry_matches_the_oracle(N, D, r, dtype):
    """Two calls in a row of the static entry against the oracle's chain of the same two fused
    steps: the oracle's first step gives R' and s for its second step, so no expected value
    comes from the GPU."""
    w = wl.Workload("noalloc_oracle", N, D, r, dtype, y_std=0.5, seed=29)
    R0, s0 = wl.make_state(w), wl.make_s_prev(w)
    y0, y1 = wl.make_y(w, 0), wl.make_y(w, 1)
    p = wl.make_params(w, 1)
    t = params_to_torch(p)
    P = gr.pack_params(t["gamma"], t["w_down"], t["w_up"], t["w_write"], TDT[dtype], w.eps)

    def static(R, y, s, P, x, sn):
        gr.write_then_read_host_static(R, y, s, P, x, sn)

    got = _two_steps(static, w, R0, y0, y1, s0, P)
    Ro, s_o = wl.to_f64(R0), s0
    for (Rg, xg, sg), y in zip(got, (y0, y1)):
        Ro, xo, s_o = oracle.write_then_read(Ro, wl.to_f64(y), s_o, p, w.eps)
        assert rel_rows(Rg.double().numpy(), Ro) <= TOL[dtype]
        assert rel_rows(xg.double().numpy(), xo) <= TOL[dtype]
        assert rel_rows(sg.double().numpy(), s_o) <= TOL[dtype]
    assert gr.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,r,dtype", [(128, 4096, 16, "bf16"), (64, 256, 8, "f32"),
                                         (333, 1024, 12, "bf16")])
def test_static_workspace_entry_matches_workspace_entry(N, D, r, dtype):
    _compare(N, D, r, dtype)


@pytest.mark.gpu
def test_static_workspace_entry_past_the_split_threshold():
    """1500 tokens at D = 1024 (18.5 MB of workspace), past the split's first token bound at that
    width (800). On a GB300 the split's time model keeps this shape, like every cluster-kernel
    shape that fits the 32 MiB workspace, on the cluster kernel alone, so the results are
    bit-identical; where the host entry does split, the static entry still runs the cluster
    kernel alone, and x and s agree within the bf16 tolerance."""
    _compare(1500, 1024, 16, "bf16")


def test_static_workspace_entry_rejects_oversize_before_any_cuda_call():
    """683 tokens at D = 4096 in bf16 need 33,592,832 bytes, more than the 32 MiB workspace:
    GR_E_SIZE, checked on the host before any copy or launch (no GPU needed)."""
    gbuild.build()
    L = gr.load()
    shape = gr.Shape(683, 4096, 4, 16, gr.GR_BF16, 1e-6)
    need = ctypes.c_size_t(0)
    assert L.gr_host_workspace_size(ctypes.byref(shape), ctypes.byref(need)) == 0
    assert need.value == 33_592_832 > (32 << 20)
    p = gr.ParamsStruct()
    p.tag, p.packed = gr.GR_PARAMS_TAG, 0x1000
    p.d_model, p.n_branch, p.rank, p.state_dtype = 4096, 4, 16, gr.GR_BF16
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(5)]
    st = L.gr_write_then_read_host_static(ctypes.byref(shape), fake[0], fake[1], fake[2],
                                          ctypes.byref(p), fake[3], fake[4], None)
    assert st == -7  # GR_E_SIZE
    shape.n_tokens = 682
    assert L.gr_host_workspace_size(ctypes.byref(shape), ctypes.byref(need)) == 0
    assert need.value <= (32 << 20)


def test_static_workspace_entry_validates_on_the_host():
    """Missing pointers, overlapping host buffers and the large-rank shapes (device entries only)
    are rejected before any CUDA call; an empty batch returns at once (no GPU needed)."""
    gbuild.build()
    L = gr.load()
    shape = gr.Shape(64, 1024, 4, 16, gr.GR_BF16, 1e-6)
    p = gr.ParamsStruct()
    p.tag, p.packed = gr.GR_PARAMS_TAG, 0x1000
    p.d_model, p.n_branch, p.rank, p.state_dtype = 1024, 4, 16, gr.GR_BF16
    fake = [ctypes.c_void_p(0x1000000 * (i + 1)) for i in range(5)]

    def call(sh, ptrs):
        return L.gr_write_then_read_host_static(ctypes.byref(sh), ptrs[0], ptrs[1], ptrs[2],
                                                ctypes.byref(p), ptrs[3], ptrs[4], None)

    assert call(shape, [fake[0], None, fake[2], fake[3], fake[4]]) == -1       # GR_E_NULL
    assert call(shape, [fake[0], fake[1], fake[2], fake[0], fake[4]]) == -8    # GR_E_ALIAS: x on R
    assert call(shape, [fake[0], fake[1], fake[2], fake[1], fake[4]]) == -8    # x on y
    assert call(shape, [fake[0], fake[1], fake[2], fake[3], fake[2]]) == -8    # s_next on s_prev
    p.rank = 8
    assert call(shape, fake) == -6                                             # GR_E_PARAMS
    tc = gr.Shape(64, 2560, 4, 320, gr.GR_BF16, 1e-6)
    p.d_model, p.rank = 2560, 320
    assert call(tc, fake) == -5                                                # GR_E_RANK
    empty = gr.Shape(0, 1024, 4, 16, gr.GR_BF16, 1e-6)
    p.d_model, p.rank = 1024, 16
    assert call(empty, [None] * 5) == 0
