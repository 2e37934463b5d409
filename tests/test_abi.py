"""The C-ABI library loads on the CPU host and exports every symbol include/gr.h declares; the
host-side validation rejects bad arguments before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from stream_gated_residual_gb300 import build as gbuild
from stream_gated_residual_gb300 import gr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gr.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gr.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(gr_\w+)\s*\(", text, re.M)))


def header_constant(name):
    text = open(HEADER).read()
    m = re.search(rf"{name}\s*=\s*(-?\d+)", text) or re.search(rf"#define {name}\s+(\w+)", text)
    return int(m.group(1), 0)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gr.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.gr_api_version() == header_constant("GR_API_VERSION")
    for code in range(0, -14, -1):
        s = gr.status_string(code)
        assert s and s != "unknown status", code
    assert gr.status_string(-99) == "unknown status"


def _shape(n=4, d=64, nb=4, r=8, dt=gr.GR_BF16, eps=1e-6):
    return gr.Shape(n, d, nb, r, dt, eps)


FAKE = ctypes.c_void_p(0x10000)          # 16-byte aligned, never dereferenced on the host
FAKE2 = ctypes.c_void_p(0x20000000)
FAKE3 = ctypes.c_void_p(0x40000000)
FAKE4 = ctypes.c_void_p(0x60000000)
FAKE5 = ctypes.c_void_p(0x70000000)


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), "GR_E_SHAPE"), (dict(d=12), "GR_E_SHAPE"), (dict(d=0), "GR_E_SHAPE"),
    (dict(d=12296), "GR_E_SHAPE"), (dict(nb=3), "GR_E_SHAPE"), (dict(r=0), "GR_E_RANK"),
    (dict(r=65), "GR_E_RANK"), (dict(dt=7), "GR_E_DTYPE"), (dict(eps=-1.0), "GR_E_EPS"),
    (dict(eps=float("inf")), "GR_E_EPS")])
def test_packed_size_rejects_bad_shapes(lib, kw, code):
    n = ctypes.c_size_t(0)
    st = lib.gr_packed_size(ctypes.byref(_shape(**kw)), ctypes.byref(n))
    assert st == header_constant(code)


def test_packed_size_grows_with_shape(lib):
    def size(d, r, dt):
        n = ctypes.c_size_t(0)
        assert lib.gr_packed_size(ctypes.byref(_shape(d=d, r=r, dt=dt)), ctypes.byref(n)) == 0
        return n.value
    assert size(256, 8, gr.GR_F32) > 0 and size(256, 8, gr.GR_BF16) > 0
    assert size(264, 8, gr.GR_F32) > size(264, 8, gr.GR_BF16)  # no fragment section at D=264
    assert size(512, 8, gr.GR_BF16) > size(256, 8, gr.GR_BF16)
    assert size(256, 16, gr.GR_BF16) > size(256, 8, gr.GR_BF16)
    assert size(256, 8, gr.GR_BF16) % 256 == 0


def test_calls_validate_before_any_launch(lib):
    sh = ctypes.byref(_shape())
    null = ctypes.c_void_p(None)
    E = header_constant
    p = gr.ParamsStruct()
    # params never packed
    assert lib.gr_read(sh, FAKE, ctypes.byref(p), FAKE2, FAKE3, null) == E("GR_E_PARAMS")
    p.tag = gr.GR_PARAMS_TAG
    p.packed = 0x1000
    p.d_model, p.n_branch, p.rank, p.state_dtype = 64, 4, 8, gr.GR_BF16
    pr = ctypes.byref(p)
    assert lib.gr_read(None, FAKE, pr, FAKE2, FAKE3, null) == E("GR_E_NULL")
    assert lib.gr_read(sh, null, pr, FAKE2, FAKE3, null) == E("GR_E_NULL")
    assert lib.gr_read(sh, ctypes.c_void_p(0x10008), pr, FAKE2, FAKE3, null) == E("GR_E_ALIGN")
    assert lib.gr_read(sh, FAKE, pr, FAKE, FAKE3, null) == E("GR_E_ALIAS")
    # params packed for another shape
    p.rank = 16
    assert lib.gr_read(sh, FAKE, pr, FAKE2, FAKE3, null) == E("GR_E_PARAMS")
    p.rank = 8
    assert lib.gr_write(sh, FAKE, FAKE, FAKE3, null) == E("GR_E_ALIAS")
    assert lib.gr_write(sh, null, FAKE2, FAKE3, null) == E("GR_E_NULL")
    # x may equal y; x may not overlap R
    assert lib.gr_write_then_read(sh, FAKE, FAKE2, FAKE3, pr, FAKE, FAKE4, null) == E("GR_E_ALIAS")
    assert lib.gr_write_then_read(sh, FAKE, FAKE2, FAKE3, pr, FAKE4, FAKE2, null) == \
        E("GR_E_ALIAS")
    # pack: misaligned packed buffer, too small a buffer
    out = gr.ParamsStruct()
    assert lib.gr_pack_params(sh, FAKE, FAKE2, FAKE3, FAKE4, ctypes.c_void_p(0x70000010), 1 << 30,
                              ctypes.byref(out), null) == E("GR_E_ALIGN")
    assert lib.gr_pack_params(sh, FAKE, FAKE2, FAKE3, FAKE4, FAKE5, 16, ctypes.byref(out),
                              null) == E("GR_E_SIZE")
    assert out.tag == 0  # untouched on error
    assert lib.gr_residual_add_ref(-1, gr.GR_BF16, FAKE, FAKE2, null) == E("GR_E_SHAPE")
    assert lib.gr_residual_add_ref(16, 5, FAKE, FAKE2, null) == E("GR_E_DTYPE")
    assert lib.gr_residual_add_ref(64, gr.GR_BF16, FAKE, FAKE, null) == E("GR_E_ALIAS")
    ws = ctypes.c_size_t(0)
    assert lib.gr_host_workspace_size(sh, ctypes.byref(ws)) == 0 and ws.value > 0
    assert lib.gr_write_then_read_host(sh, FAKE, FAKE2, FAKE3, pr, FAKE4, FAKE5, FAKE, 16,
                                       null) == E("GR_E_SIZE")


@pytest.mark.parametrize("D,r,dtype,path", [
    (4096, 16, gr.GR_BF16, "fused_bf16"), (2048, 16, gr.GR_BF16, "fused_bf16"),
    (256, 8, gr.GR_BF16, "fused_bf16"), (512, 1, gr.GR_BF16, "fused_bf16"),
    (1024, 12, gr.GR_BF16, "fused_bf16"), (7168, 32, gr.GR_BF16, "tiled_bf16"),
    (4096, 32, gr.GR_BF16, "tiled_bf16"), (4104, 16, gr.GR_BF16, "generic"),
    (768, 16, gr.GR_BF16, "tiled_bf16"), (8192, 16, gr.GR_BF16, "tiled_bf16"),
    (64, 1, gr.GR_BF16, "tiled_bf16"), (4096, 33, gr.GR_BF16, "generic"),
    (4096, 16, gr.GR_F32, "generic"), (8, 4, gr.GR_BF16, "generic"),
    (2560, 320, gr.GR_BF16, "tc_bf16"), (4096, 64, gr.GR_BF16, "tc_bf16"),
    (1024, 448, gr.GR_BF16, "tc_bf16"), (4104, 64, gr.GR_BF16, "generic"),
    (4096, 60, gr.GR_BF16, "generic"), (4096, 64, gr.GR_F32, "generic")])
def test_kernel_path_selection(lib, D, r, dtype, path):
    """The cluster tensor-core kernel takes bf16 shapes whose width splits into 1..16 CTAs of 256
    channels (a power of two) with rank <= 16; the two-pass tensor-core kernel takes the other
    bf16 shapes with D a multiple of 64 and rank <= 32; every other valid shape (fp32 states
    included) runs the generic kernel; bf16 shapes with D a multiple of 64 and a rank of 64 … 448
    (a multiple of 8) run the large-rank tensor-core path."""
    sh = _shape(n=100, d=D, r=r, dt=dtype)
    assert lib.gr_kernel_path(ctypes.byref(sh)).decode() == path
    assert lib.gr_kernel_path(ctypes.byref(_shape(d=12))).decode() == "invalid"


def test_fp8_calls_validate_before_any_launch(lib):
    """The FP8-state entries: dtype, width, rank, NULL, alignment and aliasing are checked on
    the host first; valid arguments get as far as the device check (no GPU here)."""
    E = header_constant
    null = ctypes.c_void_p(None)
    P = gr.ParamsStruct()
    P.tag, P.packed = gr.GR_PARAMS_TAG, 0x1000
    P.d_model, P.n_branch, P.rank, P.state_dtype = 4096, 4, 16, gr.GR_FP8
    sh = _shape(n=64, d=4096, r=16, dt=gr.GR_FP8)
    pr = ctypes.byref(P)
    # encode / decode
    assert lib.gr_fp8_encode(ctypes.byref(_shape(d=4096, dt=gr.GR_BF16)), FAKE, gr.GR_BF16,
                             FAKE2, FAKE3, null) == E("GR_E_DTYPE")
    assert lib.gr_fp8_encode(sh, FAKE, 7, FAKE2, FAKE3, null) == E("GR_E_DTYPE")
    assert lib.gr_fp8_encode(ctypes.byref(_shape(d=48, dt=gr.GR_FP8)), FAKE, gr.GR_BF16, FAKE2,
                             FAKE3, null) == E("GR_E_SHAPE")
    assert lib.gr_fp8_encode(ctypes.byref(_shape(n=0, d=4096, dt=gr.GR_FP8)), null, gr.GR_BF16,
                             null, null, null) == 0
    assert lib.gr_fp8_encode(sh, null, gr.GR_BF16, FAKE2, FAKE3, null) == E("GR_E_NULL")
    assert lib.gr_fp8_encode(sh, ctypes.c_void_p(0x10008), gr.GR_BF16, FAKE2, FAKE3,
                             null) == E("GR_E_ALIGN")
    assert lib.gr_fp8_encode(sh, FAKE, gr.GR_BF16, FAKE2, ctypes.c_void_p(0x20000000 + 4096),
                             null) == E("GR_E_ALIAS")
    assert lib.gr_fp8_encode(sh, FAKE, gr.GR_BF16, FAKE2, FAKE3, null) == E("GR_E_DEVICE")
    assert lib.gr_fp8_decode(sh, FAKE2, FAKE3, FAKE, 3, null) == E("GR_E_DTYPE")
    assert lib.gr_fp8_decode(sh, FAKE2, FAKE3, FAKE, gr.GR_F32, null) == E("GR_E_DEVICE")
    # the read calls need the two-pass kernel's shapes
    for d, code in ((160, "GR_E_SHAPE"), (8320, "GR_E_SHAPE"), (4096, "GR_E_DEVICE")):
        P.d_model = d
        s2 = _shape(n=64, d=d, r=16, dt=gr.GR_FP8)
        assert lib.gr_read_fp8(ctypes.byref(s2), FAKE2, FAKE3, pr, FAKE4, FAKE5,
                               null) == E(code), d
    P.rank = 33
    assert lib.gr_read_fp8(ctypes.byref(_shape(n=64, d=4096, r=33, dt=gr.GR_FP8)), FAKE2, FAKE3,
                           pr, FAKE4, FAKE5, null) == E("GR_E_RANK")
    P.rank, P.state_dtype = 16, gr.GR_BF16
    assert lib.gr_read_fp8(sh, FAKE2, FAKE3, pr, FAKE4, FAKE5, null) == E("GR_E_PARAMS")
    P.state_dtype = gr.GR_FP8
    # x overlapping the codes is refused; x == y (F's in/out buffer) is allowed
    assert lib.gr_write_then_read_fp8(sh, FAKE2, FAKE3, FAKE, FAKE5, pr, FAKE2, FAKE4,
                                      null) == E("GR_E_ALIAS")
    assert lib.gr_write_then_read_fp8(sh, FAKE2, FAKE3, FAKE, FAKE5, pr, FAKE, FAKE4,
                                      null) == E("GR_E_DEVICE")
    assert lib.gr_write_fp8(sh, FAKE2, FAKE2, FAKE, FAKE5, null) == E("GR_E_ALIAS")
    assert lib.gr_write_fp8(sh, FAKE2, FAKE3, FAKE, FAKE5, null) == E("GR_E_DEVICE")
    # the bf16/fp32 entries do not take an FP8 shape
    assert lib.gr_read(sh, FAKE, pr, FAKE2, FAKE3, null) == E("GR_E_DTYPE")
    assert lib.gr_write(sh, FAKE, FAKE2, FAKE3, null) == E("GR_E_DTYPE")


def test_fp8_kernel_path_and_packing(lib):
    def path(d, r):
        return lib.gr_kernel_path(ctypes.byref(_shape(n=100, d=d, r=r, dt=gr.GR_FP8))).decode()
    assert path(4096, 16) == "tiled_fp8" and path(7168, 32) == "tiled_fp8"
    assert path(128, 1) == "tiled_fp8" and path(8192, 8) == "tiled_fp8"
    assert path(160, 8) == "invalid" and path(8320, 8) == "invalid" and path(4096, 33) == "invalid"
    n = ctypes.c_size_t(0)
    assert lib.gr_packed_size(ctypes.byref(_shape(d=4096, r=16, dt=gr.GR_FP8)),
                              ctypes.byref(n)) == 0 and n.value > 0


def test_backward_calls_validate_before_any_launch(lib):
    E = header_constant
    null = ctypes.c_void_p(None)
    sh = _shape(n=64, d=256, r=16, dt=gr.GR_BF16)
    need = ctypes.c_size_t(0)
    assert lib.gr_read_backward_workspace_size(ctypes.byref(sh), ctypes.byref(need)) == 0
    assert need.value >= 3 * 64 * 4 * 256 * 4
    # R, gamma, W_d, W_u, W_w, dx, ds, then dR, dgamma, dW_d, dW_u, dW_w
    ptrs = [ctypes.c_void_p(0x100000 * (k + 1)) for k in range(12)]
    ws = ctypes.c_void_p(0x7000000000)
    args = lambda p, w=ws, nb=need.value: (ctypes.byref(sh), *p, w, nb, null)
    assert lib.gr_read_backward(*args(ptrs)) == E("GR_E_DEVICE")
    assert lib.gr_read_backward(*args(ptrs, nb=need.value - 1)) == E("GR_E_SIZE")
    assert lib.gr_read_backward(*args(ptrs[:3] + [null] + ptrs[4:])) == E("GR_E_NULL")
    assert lib.gr_read_backward(*args(ptrs, w=ctypes.c_void_p(0x7000000010))) == E("GR_E_ALIGN")
    aliased = ptrs[:7] + [ptrs[0]] + ptrs[8:]          # dR on top of R
    assert lib.gr_read_backward(*args(aliased)) == E("GR_E_ALIAS")
    fp8 = _shape(n=64, d=256, r=16, dt=gr.GR_FP8)
    assert lib.gr_read_backward(ctypes.byref(fp8), *ptrs, ws, need.value, null) == E("GR_E_DTYPE")
    assert lib.gr_read_backward(ctypes.byref(_shape(n=0, d=256, r=16)), *[null] * 12, null, 0,
                                null) == 0
    # write backward: dR may be dR_next itself; dy on top of dR_next is refused
    assert lib.gr_write_backward(ctypes.byref(sh), FAKE, FAKE2, FAKE3, FAKE, FAKE4, FAKE5,
                                 null) == E("GR_E_DEVICE")
    assert lib.gr_write_backward(ctypes.byref(sh), FAKE, FAKE2, FAKE3, FAKE4, FAKE, FAKE5,
                                 null) == E("GR_E_ALIAS")


def test_decompose_validates_before_any_launch(lib):
    E = header_constant
    null = ctypes.c_void_p(None)
    sh = _shape(n=64, d=256, r=16, dt=gr.GR_BF16)
    # R, gamma, W_d, W_u, W_w, then (after U) y, s, R0, norm, branch_norm, pi, a0_norm
    p = [ctypes.c_void_p(0x1000000 * (k + 1)) for k in range(12)]
    call = lambda q, U=5, shape=sh: lib.gr_decompose(ctypes.byref(shape), *q[:5], U, *q[5:],
                                                     null)
    assert call(p) == E("GR_E_DEVICE")
    assert call(p, U=-1) == E("GR_E_SHAPE")
    assert call(p, U=E("GR_MAX_WRITERS") + 1) == E("GR_E_SHAPE")
    assert call(p[:5] + [null] + p[6:]) == E("GR_E_NULL")                 # y
    assert call(p[:8] + [null] + p[9:]) == E("GR_E_NULL")                 # norm
    assert call(p[:11] + [null]) == E("GR_E_NULL")                        # R0 without a0_norm
    assert call(p[:5] + [ctypes.c_void_p(0x6000008)] + p[6:]) == E("GR_E_ALIGN")
    assert call(p[:8] + [p[5]] + p[9:]) == E("GR_E_ALIAS")                # norm on y
    assert call(p[:9] + [p[8]] + p[10:]) == E("GR_E_ALIAS")               # branch_norm on norm
    # optional outputs may be absent; no writers and no initial state: nothing to do
    assert call(p[:9] + [null, null] + p[11:]) == E("GR_E_DEVICE")
    assert call(p[:5] + [null] * 7, U=0) == 0
    assert call(p, shape=_shape(n=64, d=256, r=16, dt=gr.GR_FP8)) == E("GR_E_DTYPE")


def test_large_rank_validation(lib):
    """Ranks above 64 exist only on the large-rank path (bf16, D % 64 == 0, r % 8 == 0,
    r <= 448); its shapes need a step workspace: the workspace-free entries refuse them with
    GR_E_SIZE, the host-buffer entries with GR_E_RANK, before any CUDA call."""
    E = header_constant
    null = ctypes.c_void_p(None)
    assert E("GR_MAX_RANK_TC") == 448
    need = ctypes.c_size_t(0)
    tc = _shape(n=300, d=2560, r=320, dt=gr.GR_BF16)
    assert lib.gr_step_workspace_size(ctypes.byref(tc), ctypes.byref(need)) == 0
    a256 = lambda n: (n + 255) // 256 * 256
    # 1/rms | h (bf16, r rounded up to 64) | the r + 4 projections of each branch (fp32) | ssq
    assert need.value == a256(300 * 16) + a256(300 * 320 * 2) + a256(300 * 16 * 324) + a256(300 * 16)
    small = _shape(n=300, d=4096, r=16, dt=gr.GR_BF16)
    assert lib.gr_step_workspace_size(ctypes.byref(small), ctypes.byref(need)) == 0
    assert need.value == 0
    for d, r, dt in ((2560, 512, gr.GR_BF16), (2560, 456, gr.GR_BF16), (2560, 100, gr.GR_BF16),
                     (2568, 128, gr.GR_BF16), (2560, 128, gr.GR_F32), (2560, 128, gr.GR_FP8)):
        bad = _shape(n=4, d=d, r=r, dt=dt)
        assert lib.gr_step_workspace_size(ctypes.byref(bad), ctypes.byref(need)) in (
            E("GR_E_RANK"), E("GR_E_SHAPE"), E("GR_E_DTYPE")), (d, r, dt)
    # a packed-parameter struct for the shape (never dereferenced on the host)
    st = gr.ParamsStruct()
    st.tag, st.packed, st.d_model, st.n_branch, st.rank, st.state_dtype = (
        gr.GR_PARAMS_TAG, FAKE.value, 2560, 4, 320, gr.GR_BF16)
    R, x, s = (ctypes.c_void_p(0x1000000), ctypes.c_void_p(0x4000000), ctypes.c_void_p(0x5000000))
    ws = ctypes.c_void_p(0x6000000)
    assert lib.gr_read(ctypes.byref(tc), R, ctypes.byref(st), x, s, null) == E("GR_E_SIZE")
    assert lib.gr_read_ws(ctypes.byref(tc), R, ctypes.byref(st), x, s, ws, 10**7,
                          null) == E("GR_E_DEVICE")
    assert lib.gr_read_ws(ctypes.byref(tc), R, ctypes.byref(st), x, s, ws, 100,
                          null) == E("GR_E_SIZE")
    assert lib.gr_read_ws(ctypes.byref(tc), R, ctypes.byref(st), x, s,
                          ctypes.c_void_p(0x6000010), 10**7, null) == E("GR_E_ALIGN")
    assert lib.gr_read_ws(ctypes.byref(tc), R, ctypes.byref(st), x, s, R, 10**7,
                          null) == E("GR_E_ALIAS")
    y = ctypes.c_void_p(0x3000000)
    assert lib.gr_write_then_read(ctypes.byref(tc), R, y, s, ctypes.byref(st), x,
                                  ctypes.c_void_p(0x5100000), null) == E("GR_E_SIZE")
    assert lib.gr_write_then_read_ws(ctypes.byref(tc), R, y, s, ctypes.byref(st), x,
                                     ctypes.c_void_p(0x5100000), ws, 10**7,
                                     null) == E("GR_E_DEVICE")
    assert lib.gr_write_then_read_host(ctypes.byref(tc), R, y, s, ctypes.byref(st), x,
                                       ctypes.c_void_p(0x5100000), ws, 10**9,
                                       null) == E("GR_E_RANK")
    # the CUDA-core backward and decomposition stop at rank 64
    assert lib.gr_read_backward_workspace_size(ctypes.byref(tc), ctypes.byref(need)) == \
        E("GR_E_RANK")
