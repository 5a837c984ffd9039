"""C-ABI checks that need no GPU: the library builds and loads, exports every entry point the
header declares, sizes its buffers, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from linear_lsh_sketch_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "race_attn.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    import linear_lsh_sketch_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(race_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("race_attn_fwd", "race_attn_bwd", "race_attn_workspace_bytes", "race_attn_state_bytes",
              "race_attn_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.library_path)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def shape(lib, B=1, H=2, N=100, d=64, dtype=1):
    return lib.make_shape(B, H, N, d, dtype)


def test_sizes(lib):
    s = shape(lib)
    for causal in (0, 1):
        f = lib.race_attn_workspace_bytes(s, 3, 3, causal, 0)
        b = lib.race_attn_workspace_bytes(s, 3, 3, causal, 1)
        st = lib.race_attn_state_bytes(s, 3, 3, causal)
        assert 0 < f <= b
        assert st >= 2 * 24 * 65 * 4  # at least one [A | B] per (b, h)
    # the saved sketch is one [LR, d+1] float32 block per (b, h) when non-causal
    assert lib.race_attn_state_bytes(s, 3, 3, 0) == 2 * 24 * 65 * 4
    # causal float32: whole segment sketches only; causal bf16 (tcgen05 path): the segment
    # sketches, then every key's bucket features (bf16, L R = 24 per token) at a 256-byte offset,
    # then every key's 1 / |k| (float32), again at a 256-byte offset
    assert lib.race_attn_state_bytes(shape(lib, dtype=0), 3, 3, 1) % (24 * 65 * 4) == 0
    sk = lib.race_attn_state_bytes(s, 3, 3, 1) - 2 * 100 * 4 - (2 * 100 * 24 * 2 + 255) // 256 * 256
    nseg = sk // (2 * 24 * 65 * 4)
    assert sk % 256 == 0 and nseg >= 1 and sk - 256 < nseg * 2 * 24 * 65 * 4 <= sk
    # sizes depend on the shape only
    assert lib.race_attn_state_bytes(s, 3, 3, 1) == lib.race_attn_state_bytes(shape(lib), 3, 3, 1)


@pytest.mark.parametrize("bad", [
    dict(d=65), dict(d=0), dict(d=136), dict(N=0), dict(B=0), dict(dtype=7),
    dict(P=0), dict(P=9), dict(L=0), dict(L=17), dict(P=7, L=4),
])
def test_invalid_sizes_report_zero(lib, bad):
    P, L = bad.pop("P", 3), bad.pop("L", 3)
    s = shape(lib, **bad)
    assert lib.race_attn_workspace_bytes(s, L, P, 0, 1) == 0
    assert lib.race_attn_state_bytes(s, L, P, 1) == 0


def _raw(lib):
    return lib.load_library()


def test_fwd_rejects_before_launch(lib):
    """Argument errors return a status without touching the GPU (safe on a machine without one)."""
    L = _raw(lib)
    s = shape(lib)
    p = ctypes.c_void_p(4096)  # an aligned, never-dereferenced address
    ws = lib.race_attn_workspace_bytes(s, 3, 3, 0, 0)
    fwd = lambda *a: L.race_attn_fwd(*a)
    assert fwd(None, p, p, p, p, 10.0, 3, 3, 0, p, None, p, ws, None) == -1
    assert fwd(ctypes.byref(s), None, p, p, p, 10.0, 3, 3, 0, p, None, p, ws, None) == -1
    assert fwd(ctypes.byref(s), p, p, p, p, float("nan"), 3, 3, 0, p, None, p, ws, None) == -1
    assert fwd(ctypes.byref(s), p, p, p, p, -1.0, 3, 3, 0, p, None, p, ws, None) == -1
    assert fwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 9, 0, p, None, p, ws, None) == -1
    assert fwd(ctypes.byref(s), ctypes.c_void_p(4097), p, p, p, 10.0, 3, 3, 0, p, None, p, ws, None) == -5
    assert fwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 0, p, None, p, ws - 1, None) == -3


def test_bwd_rejects_before_launch(lib):
    L = _raw(lib)
    s = shape(lib)
    p = ctypes.c_void_p(4096)
    ws = lib.race_attn_workspace_bytes(s, 3, 3, 1, 1)
    bwd = lambda *a: L.race_attn_bwd(*a)
    assert bwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 1, None, None, p, p, p, None, None, None, p, ws, None) == -1
    assert bwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 1, None, p, p, p, p, None, None, None, p, ws - 256,
               None) == -3
    assert bwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 1, None, p, p, ctypes.c_void_p(4104), p, None, None, None, p,
               ws, None) == -5
    # d(loss)/d(beta) and d(loss)/d(W) outputs: float32, so 4-byte alignment is required
    assert bwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 1, None, p, p, p, p, ctypes.c_void_p(4098), None, None, p,
               ws, None) == -5
    assert bwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 1, None, p, p, p, p, None, ctypes.c_void_p(4098), None, p,
               ws, None) == -5
    # d(loss)/d(W) needs the larger workspace (is_bwd = 2): the backward's plus the dz rows
    ws_dw = lib.race_attn_workspace_bytes(s, 3, 3, 1, 2)
    assert ws_dw > ws
    assert bwd(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, 1, None, p, p, p, p, None, p, None, p, ws, None) == -3


def test_decode_rejects_before_launch(lib):
    """The decode step takes one token per (b, h): N must be 1; null, misaligned or out-of-range
    arguments are refused without a launch."""
    L = _raw(lib)
    s = shape(lib)  # N > 1
    one = lib.make_shape(s.B, s.H, 1, s.d, s.dtype)
    p = ctypes.c_void_p(4096)
    dec = lambda *a: L.race_attn_decode(*a)
    assert dec(ctypes.byref(s), p, p, p, p, 10.0, 3, 3, p, p, None) == -1
    assert dec(ctypes.byref(one), p, None, p, p, 10.0, 3, 3, p, p, None) == -1
    assert dec(ctypes.byref(one), p, p, p, p, float("nan"), 3, 3, p, p, None) == -1
    assert dec(ctypes.byref(one), p, p, p, p, -1.0, 3, 3, p, p, None) == -1
    assert dec(ctypes.byref(one), p, p, p, p, 10.0, 3, 3, ctypes.c_void_p(4100), p, None) == -5
    assert dec(None, p, p, p, p, 10.0, 3, 3, p, p, None) == -1


def test_strerror(lib):
    assert lib.race_attn_strerror(0) == "ok"
    for rc in (-1, -2, -3, -4, -5, -6, -7, -8, -9):
        assert lib.race_attn_strerror(rc) not in ("ok", "unknown status")
    assert lib.race_attn_strerror(-99) == "unknown status"


def test_instrumentation_defaults(lib):
    assert lib.race_attn_launch_count() >= 0
    lib.race_attn_profile_reset()
    assert lib.race_attn_profile_read() == {}


def test_per_head_w_layout(lib):
    """race_shape.per_head_w selects W [H, L, P, d]: it changes no buffer size, takes only 0 or 1,
    and the binding picks it from W's shape (checked before any call)."""
    import torch
    s = shape(lib)
    ph = lib.make_shape(s.B, s.H, s.N, s.d, s.dtype, per_head_w=True)
    assert ctypes.sizeof(type(s)) == 40
    for causal in (0, 1):
        for is_bwd in (0, 1):
            assert lib.race_attn_workspace_bytes(ph, 3, 3, causal, is_bwd) == \
                lib.race_attn_workspace_bytes(s, 3, 3, causal, is_bwd)
    s.per_head_w = 2
    assert lib.race_attn_workspace_bytes(s, 3, 3, 0, 1) == 0
    Q = torch.zeros((2, 4, 8, 64), dtype=torch.bfloat16)
    assert lib._shape_of(Q, torch.zeros((3, 2, 64)), 3, 2).per_head_w == 0
    assert lib._shape_of(Q, torch.zeros((4, 3, 2, 64)), 3, 2).per_head_w == 1
    for bad in ((2, 3, 2, 64), (3, 2, 32), (4, 3, 2)):
        with pytest.raises(ValueError):
            lib._shape_of(Q, torch.zeros(bad), 3, 2)
    with pytest.raises(ValueError):
        lib._shape_of(Q, torch.zeros((3, 2, 64), dtype=torch.float64), 3, 2)


def test_beta_domain(lib):
    """beta >= 0, finite or +inf (hard hashing); NaN and negatives are refused before any launch.
    A short workspace makes an accepted beta stop at the workspace check instead."""
    L = _raw(lib)
    s = shape(lib)
    p = ctypes.c_void_p(4096)
    ws = lib.race_attn_workspace_bytes(s, 3, 3, 0, 0)
    fwd = lambda b: L.race_attn_fwd(ctypes.byref(s), p, p, p, p, b, 3, 3, 0, p, None, p, ws - 256, None)
    assert fwd(float("nan")) == -1
    assert fwd(-0.5) == -1
    assert fwd(float("-inf")) == -1
    assert fwd(float("inf")) == -3
    assert fwd(0.0) == -3


def test_angular_rejects_before_launch(lib):
    """race_attn_angular: gamma finite >= 0, non-null 16-byte aligned tensors, valid shape."""
    L = _raw(lib)
    s = shape(lib)
    p = ctypes.c_void_p(4096)
    ang = lambda sh, q, g, o: L.race_attn_angular(ctypes.byref(sh) if sh is not None else None, q, p, p, g, 0, o,
                                                   None)
    for g in (float("nan"), float("inf"), -1.0):
        assert ang(s, p, g, p) == -1
    assert ang(s, None, 2.0, p) == -1
    assert ang(s, p, 2.0, None) == -1
    assert ang(s, ctypes.c_void_p(4104), 2.0, p) == -5
    assert ang(shape(lib, d=65), p, 2.0, p) == -1
    assert ang(None, p, 2.0, p) == -1
