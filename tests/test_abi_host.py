"""Host-side checks of the C ABI and the Python binding (no GPU needed):
the library loads, exports every symbol the header declares, and rejects
invalid problems with the pages' exception types before touching the GPU."""

import ctypes
import os
import re

import pytest
import torch

import mamba_mimo_chunked_gb300 as mm
import synthetic_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", n) for n in ("mamba_mimo_bwd_fwd.h", "mamba_mimo_bwd_bwd.h")]


@pytest.fixture(scope="module")
def lib():
    mm.build()
    return mm.load_library()


def declared_functions():
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"\b(mamba_mimo_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mamba_mimo_bwd_fwd" in names and "mamba_mimo_bwd_fwd_workspace_size" in names
    assert "mamba_mimo_bwd_bwd" in names and "mamba_mimo_bwd_bwd_workspace_size" in names
    for name in names:
        assert hasattr(lib, name), name
    assert lib.mamba_mimo_abi_version() == 1


def dims(**kw):
    base = dict(B=1, S=8192, H=16, G=1, R=4, N=64, P=64)
    base.update(kw)
    return mm._Dims(*[base[k] for k in ("B", "S", "H", "G", "R", "N", "P")])


def ws(lib, d, C=16, div=4, reduced=1, has_z=1):
    n = ctypes.c_size_t(0)
    st = lib.mamba_mimo_bwd_fwd_workspace_size(ctypes.byref(d), C, div, reduced, has_z, ctypes.byref(n))
    return st, n.value, lib.mamba_mimo_last_error().decode()


def test_workspace_query_and_shape_errors(lib):
    st, n, _ = ws(lib, dims())
    assert st == 0 and n > 0
    cases = [
        (dims(B=0), 16, 4, 1, "B, S, R and G must be positive"),
        (dims(R=0), 16, 4, 1, "B, S, R and G must be positive"),
        (dims(), 33, 4, 1, "chunk_size * R must be in [1, 128]"),
        (dims(), 0, 4, 1, "chunk_size * R must be in [1, 128]"),
        (dims(), 16, 3, 1, "rotary_dim_divisor must be 2 or 4"),
        (dims(N=66), 16, 4, 1, "N must be even and divisible"),
        (dims(N=256), 16, 4, 1, "N greater than 128"),
        (dims(H=6, G=4), 16, 4, 1, "H must be divisible by G"),
        (dims(P=129), 16, 4, 1, "P greater than 128"),
        (dims(R=32), 4, 4, 3, "outside this build's envelope"),
    ]
    for d, C, div, code, msg in cases:
        st, _, err = ws(lib, d, C, div)
        assert st == code and msg in err, (st, err)


def test_entry_point_rejects_bad_pointer_patterns_without_gpu(lib):
    d = dims(S=64, H=2, R=2, N=16, P=16)
    fake = ctypes.c_void_p(0x1000)
    null = None
    args = [fake] * 17
    # z given, mimo_z missing
    args[9] = null
    st = lib.mamba_mimo_bwd_fwd(ctypes.byref(d), *args, 16, 4, fake, fake, fake, fake, fake, fake,
                                1 << 30, None)
    assert st == 2 and "mimo_z is required" in lib.mamba_mimo_last_error().decode()
    # misaligned input
    args = [fake] * 17
    args[2] = ctypes.c_void_p(0x1002)
    st = lib.mamba_mimo_bwd_fwd(ctypes.byref(d), *args, 16, 4, fake, fake, fake, fake, fake, fake,
                                1 << 30, None)
    assert st == 4
    # workspace too small
    args = [fake] * 17
    st = lib.mamba_mimo_bwd_fwd(ctypes.byref(d), *args, 16, 4, fake, fake, fake, fake, fake, fake,
                                16, None)
    assert st == 5 and "workspace needs" in lib.mamba_mimo_last_error().decode()
    # dmimo_o requested without mimo_o
    args = [fake] * 17
    args[7] = null
    st = lib.mamba_mimo_bwd_fwd(ctypes.byref(d), *args, 16, 4, fake, fake, fake, fake, fake, fake,
                                1 << 30, None)
    assert st == 2


def _unit_args(**kw):
    inp = si.make_inputs(B=1, S=16, H=1, G=1, R=4, N=64, P=64, C=16, recipe="unit", **kw)
    return list(si.args_of(inp))


def test_python_binding_invalid_q_shape():
    args = _unit_args()
    args[1] = torch.randn((1, 16, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="q must have shape"):
        mm.mamba_mimo_bwd_fwd(*args)


def test_python_binding_invalid_empty_batch():
    args = _unit_args()
    args[1] = torch.zeros((0, 16, 4, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="B, S, R and G must be positive"):
        mm.mamba_mimo_bwd_fwd(*args)


def test_python_binding_invalid_q_dtype():
    args = _unit_args()
    args[1] = args[1].to(torch.float16)
    with pytest.raises(TypeError, match="torch.bfloat16"):
        mm.mamba_mimo_bwd_fwd(*args)


def test_python_binding_requires_cuda_tensors():
    with pytest.raises(ValueError, match="CUDA tensors"):
        mm.mamba_mimo_bwd_fwd(*_unit_args())


def test_device_status_without_a_call_is_ok(lib):
    # nothing enqueued on this thread yet: no stream is touched
    import threading
    res = []
    t = threading.Thread(target=lambda: res.append(lib.mamba_mimo_device_status(None)))
    t.start()
    t.join()
    assert res == [0]


# ---- second backward stage: host-side validation (nothing reaches a GPU)

def bb_ws(lib, d, C=16, div=4):
    n = ctypes.c_size_t(0)
    st = lib.mamba_mimo_bwd_bwd_workspace_size(ctypes.byref(d), C, div, ctypes.byref(n))
    return st, n.value, lib.mamba_mimo_last_error().decode()


def test_bwd_bwd_workspace_query_and_envelope(lib):
    st, n, _ = bb_ws(lib, dims())
    # dstates [BH][nc][N][P] + decays + DMIMO_V and DD partials, FP32
    nc = 8192 // 16
    assert st == 0 and n >= 16 * nc * (64 * 64 + 1 + 4 * 64 + 1) * 4
    for d, C, div, code, msg in [
        (dims(B=0), 16, 4, 1, "must be positive"),
        (dims(H=6, G=4), 16, 4, 1, "multiple of G"),
        (dims(), 16, 3, 1, "rotary_dim_divisor"),
        (dims(N=66), 16, 4, 1, "N must be even"),
        (dims(N=512), 16, 4, 3, "N <= 256, P, C*R <= 128"),
        (dims(P=192), 16, 4, 3, "N <= 256, P, C*R <= 128"),
        (dims(), 64, 4, 3, "N <= 256, P, C*R <= 128"),
        (dims(R=32, N=16, P=16), 2, 4, 3, "R <= 16"),
    ]:
        st, _, err = bb_ws(lib, d, C, div)
        assert st == code and msg in err, (st, err)


def test_bwd_bwd_wide_shapes_add_the_gradient_scratch(lib):
    # above 64 in N, P or C*R the gradient kernel keeps its FP32 tiles in a
    # per-CTA scratch (152 persistent CTAs), sized from the padded extents
    def need(**kw):
        C = kw.pop("C", 16)
        st, n, _ = bb_ws(lib, dims(**kw), C, 4)
        assert st == 0
        return n

    base = need()
    for kw, (CR16, LN, LP, N16, C, W, R, P) in [
        (dict(N=128, P=128), (64, 128, 128, 128, 16, 32, 4, 128)),
        (dict(C=32), (128, 64, 64, 64, 32, 16, 4, 64)),
        (dict(N=256, P=72, R=1, C=128), (128, 256, 80, 256, 128, 64, 1, 72)),
    ]:
        n = need(**kw)
        S, H = 8192, 16
        nc = (S + C - 1) // C
        Np = kw.get("N", 64)
        plain = sum((x + 255) // 256 * 256 for x in (H * nc * Np * P * 4, H * nc * 4, H * nc * R * P * 4, H * nc * 4))
        cc = CR16 * CR16
        m1 = -(-max(cc, 2 * C * W + R * P) // 64) * 64
        m2 = -(-max(cc, C * P) // 64) * 64
        scr = -(-(4 * CR16 * LN + 3 * CR16 * LP + 2 * N16 * LP + m1 + m2) // 64) * 64
        assert n == plain + (152 * scr * 4 + 255) // 256 * 256, kw
    assert base < need(N=128, P=128)


def test_bwd_bwd_rejects_bad_pointer_patterns_without_gpu(lib):
    d = dims(S=64, H=2, R=2, N=16, P=16)
    fake = ctypes.c_void_p(0x1000)

    def call(ins, outs, ws_bytes=1 << 30, ws_ptr=fake, dtype=0, act=1):
        return lib.mamba_mimo_bwd_bwd(ctypes.byref(d), *ins, 16, 4, act, dtype, *outs, ws_ptr, ws_bytes, None)

    ins = [fake] * 17
    outs = [fake] * 12
    # DD without d
    ins2 = list(ins)
    ins2[16] = None
    assert call(ins2, outs) == 2 and "DD must be given" in lib.mamba_mimo_last_error().decode()
    # a required input missing
    ins2 = list(ins)
    ins2[7] = None
    assert call(ins2, outs) == 2
    # misaligned pointer
    ins2 = list(ins)
    ins2[3] = ctypes.c_void_p(0x1002)
    assert call(ins2, outs) == 4
    # workspace too small / misaligned
    assert call(ins, outs, ws_bytes=16) == 5
    assert call(ins, outs, ws_ptr=ctypes.c_void_p(0x1010)) == 4
    # an unknown DQ / DK / DV dtype
    assert call(ins, outs, dtype=3) == 2 and "dqkv_dtype" in lib.mamba_mimo_last_error().decode()
    assert call(ins, outs, act=-1) == 2 and "act_dtype" in lib.mamba_mimo_last_error().decode()
