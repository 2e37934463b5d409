"""Failure detection without a GPU fault: a device-side bounded wait that nothing satisfies
gives up after its limit, records the status word and returns; the host reads GR_E_TIMEOUT
through gr_device_status, clears it, and the library keeps working."""
import ctypes

import pytest
import torch

from gr_testlib import params_to_torch, to_torch
from stream_gated_residual_gb300 import build as gbuild
from stream_gated_residual_gb300 import gr
from stream_gated_residual_gb300 import workloads as wl

GR_E_SIZE, GR_E_TIMEOUT = -7, -12


def test_selftest_rejects_bad_limits_on_the_host():
    gbuild.build()
    L = gr.load()
    for bad in (0, -5, 4_000_000_001):
        assert L.gr_selftest_bounded_wait(bad, None) == GR_E_SIZE


@pytest.mark.gpu
def test_bounded_wait_times_out_and_is_reported():
    gr.device_status(clear=True)
    assert gr.device_status() == 0
    gr.selftest_bounded_wait(200_000)          # about 0.1 ms at 2 GHz
    assert gr.device_status() == GR_E_TIMEOUT  # sticky until cleared
    assert gr.device_status(clear=True) == GR_E_TIMEOUT
    assert gr.device_status() == 0
    # the context is still usable: a fused step runs and reports no timeout
    w = wl.Workload("after", 64, 1024, 16, "bf16", y_std=0.5, seed=5)
    t = params_to_torch(wl.make_params(w, 1))
    P = gr.pack_params(t["gamma"], t["w_down"], t["w_up"], t["w_write"], torch.bfloat16, w.eps)
    R = to_torch(wl.make_state(w))
    x, s = gr.write_then_read(R, to_torch(wl.make_y(w)),
                              torch.from_numpy(wl.make_s_prev(w)).cuda(), P)
    torch.cuda.synchronize()
    assert torch.isfinite(x.float()).all() and torch.isfinite(s).all()
    assert gr.device_status() == 0
