"""Python binding of librace_attn.so, the GB300 (sm_103a) RACE attention library.

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
The function names are those of the C ABI in include/race_attn.h, which states the contract of
each call.  PyTorch supplies device memory and the current stream; tensors are passed by
pointer.  There is no fallback: if the compiled library is missing, importing it raises.
"""
import ctypes
import os

import torch

__all__ = [
    "RaceAttnError", "race_attn_fwd", "race_attn_bwd", "race_attn_workspace_bytes",
    "race_attn_state_bytes", "race_attn_strerror", "race_attn_launch_count", "race_attn_profile",
    "race_attn_profile_read", "race_attn_profile_reset", "library_path", "load_library",
    "race_attn_fwd_noalloc", "RACE_NOALLOC_SCRATCH_BYTES", "race_attn_status", "race_attn_decode",
    "race_attn_angular", "race_attn_noalloc_init", "race_attn_noalloc_status",
    "race_attn_test_withhold_first_load",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "librace_attn.so")

RACE_F32, RACE_BF16 = 0, 1
RACE_ERR_SCRATCH_LIMIT = -6
RACE_ERR_DEVICE_TIMEOUT = -7
RACE_ERR_NUMERIC = -8
RACE_ERR_NOALLOC_SETUP = -9
RACE_NOALLOC_SCRATCH_BYTES = 32 << 20  # size of the library's built-in scratch buffer
_DTYPES = {torch.float32: RACE_F32, torch.bfloat16: RACE_BF16}

_lib = None


class RaceAttnError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, race_attn_strerror(status), status))


class race_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64),
                ("d", ctypes.c_int64), ("dtype", ctypes.c_int32), ("per_head_w", ctypes.c_int32)]


def load_library():
    """Load librace_attn.so (built in-tree by __graft_entry__.build / build.py); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise ImportError("librace_attn.so is not built (expected at %s); run "
                          "`python -m linear_lsh_sketch_gb300.build`" % library_path)
    L = ctypes.CDLL(library_path)
    vp, sz, i, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    shp = ctypes.POINTER(race_shape)
    L.race_attn_workspace_bytes.argtypes = [shp, i, i, i, i]
    L.race_attn_workspace_bytes.restype = sz
    L.race_attn_state_bytes.argtypes = [shp, i, i, i]
    L.race_attn_state_bytes.restype = sz
    L.race_attn_fwd.argtypes = [shp, vp, vp, vp, vp, f, i, i, i, vp, vp, vp, sz, vp]
    L.race_attn_fwd.restype = i
    L.race_attn_bwd.argtypes = [shp, vp, vp, vp, vp, f, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.race_attn_bwd.restype = i
    L.race_attn_fwd_noalloc.argtypes = [shp, vp, vp, vp, vp, f, i, i, i, vp, vp]
    L.race_attn_fwd_noalloc.restype = i
    L.race_attn_decode.argtypes = [shp, vp, vp, vp, vp, f, i, i, vp, vp, vp]
    L.race_attn_decode.restype = i
    L.race_attn_angular.argtypes = [shp, vp, vp, vp, f, i, vp, vp]
    L.race_attn_angular.restype = i
    L.race_attn_status.argtypes = [vp, vp]
    L.race_attn_status.restype = i
    L.race_attn_noalloc_init.argtypes = []
    L.race_attn_noalloc_init.restype = i
    L.race_attn_noalloc_status.argtypes = [vp]
    L.race_attn_noalloc_status.restype = i
    L.race_attn_test_withhold_first_load.argtypes = [i]
    L.race_attn_test_withhold_first_load.restype = i
    L.race_attn_strerror.argtypes = [i]
    L.race_attn_strerror.restype = ctypes.c_char_p
    L.race_attn_launch_count.argtypes = []
    L.race_attn_launch_count.restype = ctypes.c_uint64
    L.race_attn_profile.argtypes = [i]
    L.race_attn_profile.restype = i
    L.race_attn_profile_read.argtypes = [i, ctypes.POINTER(ctypes.c_char_p),
                                         ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_double)]
    L.race_attn_profile_read.restype = i
    L.race_attn_profile_reset.argtypes = []
    L.race_attn_profile_reset.restype = None
    _lib = L
    return L


def make_shape(B, H, N, d, dtype, per_head_w=False):
    code = _DTYPES.get(dtype, dtype) if not isinstance(dtype, int) else dtype
    return race_shape(int(B), int(H), int(N), int(d), int(code), int(bool(per_head_w)))


def _shape_of(Q, W=None, L=None, P=None):
    """race_shape of the token tensor Q; with W also checks the hyperplanes: float32, contiguous,
    [L, P, d] (shared by every head) or [H, L, P, d] (one set per head)."""
    if Q.dim() != 4:
        raise ValueError("token tensors must be [B, H, N, d]")
    if Q.dtype not in _DTYPES:
        raise TypeError("token tensors must be float32 or bfloat16")
    B, H, N, d = Q.shape
    per_head = False
    if W is not None:
        shared, heads = (L, P, d), (H, L, P, d)
        if W.dtype != torch.float32 or not W.is_contiguous() or tuple(W.shape) not in (shared, heads):
            raise ValueError("W must be a contiguous float32 tensor of shape [L, P, d] or [H, L, P, d]")
        per_head = tuple(W.shape) == heads and W.dim() == 4
        if W.device != Q.device:
            raise ValueError("W must be on the token tensors' device")
    return make_shape(B, H, N, d, Q.dtype, per_head)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_like(name, t, ref):
    if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
        raise ValueError("%s must match Q in shape, dtype and device" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def race_attn_workspace_bytes(shape, L, P, causal, is_bwd):
    return load_library().race_attn_workspace_bytes(ctypes.byref(shape), int(L), int(P), int(causal),
                                                    int(is_bwd))


def race_attn_state_bytes(shape, L, P, causal):
    return load_library().race_attn_state_bytes(ctypes.byref(shape), int(L), int(P), int(causal))


def race_attn_strerror(status):
    return load_library().race_attn_strerror(int(status)).decode()


def race_attn_status(workspace, stream=None):
    """Synchronise and read the device status word of `workspace`: 0 = ok, -7 = a bounded wait
    ran out, -8 = an output row had a zero or non-finite denominator (see race_attn_status in
    include/race_attn.h)."""
    with torch.cuda.device(workspace.device):
        return load_library().race_attn_status(_ptr(workspace), _stream(stream))


def race_attn_noalloc_init(device=None):
    """Set up the built-in scratch buffer of race_attn_fwd_noalloc on `device` (default: the
    current one); do it before an allocator takes the device's memory and before any capture."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        rc = load_library().race_attn_noalloc_init()
    if rc != 0:
        raise RaceAttnError(rc, "race_attn_noalloc_init")


def race_attn_noalloc_status(device=None, stream=None):
    """Synchronise and read the device status word of the last race_attn_fwd_noalloc call on
    `device` (codes as race_attn_status)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return load_library().race_attn_noalloc_status(_stream(stream))


def race_attn_test_withhold_first_load(enable):
    """Test hook of the failure path (see include/race_attn.h): while enabled, the causal bf16
    tcgen05 forward never requests its first tiles, its waits run out and the status word reports
    a timeout."""
    return load_library().race_attn_test_withhold_first_load(int(bool(enable)))


def race_attn_launch_count():
    return int(load_library().race_attn_launch_count())


def race_attn_profile(enable):
    return load_library().race_attn_profile(int(bool(enable)))


def race_attn_profile_reset():
    load_library().race_attn_profile_reset()


def race_attn_profile_read():
    """{kernel name: (launches, total device ms)} for the launches recorded since the last reset."""
    L = load_library()
    out = {}
    name = ctypes.c_char_p()
    n_l = ctypes.c_int64()
    ms = ctypes.c_double()
    n = L.race_attn_profile_read(0, ctypes.byref(name), ctypes.byref(n_l), ctypes.byref(ms))
    for i in range(max(n, 0)):
        L.race_attn_profile_read(i, ctypes.byref(name), ctypes.byref(n_l), ctypes.byref(ms))
        out[name.value.decode()] = (int(n_l.value), float(ms.value))
    return out


def _bytes_buffer(nbytes, device, given):
    if given is not None:
        return given
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def race_attn_fwd(Q, K, V, W, beta, L, P, causal, O=None, state=None, workspace=None, stream=None):
    """O = RACE attention of Q, K, V ([B, H, N, d], float32 or bfloat16, CUDA); W float32 [L, P, d]
    (shared by every head) or [H, L, P, d] (one set per head).

    O, state and workspace are allocated with torch when not given.  Returns O.
    """
    with torch.cuda.device(Q.device):
        shape = _shape_of(Q, W, L, P)
        _check_like("K", K, Q)
        _check_like("V", V, Q)
        _check_like("Q", Q, Q)
        if O is None:
            O = torch.empty_like(Q)
        _check_like("O", O, Q)
        ws_bytes = race_attn_workspace_bytes(shape, L, P, causal, 0)
        if ws_bytes == 0:
            raise RaceAttnError(-1, "race_attn_fwd")
        workspace = _bytes_buffer(ws_bytes, Q.device, workspace)
        rc = load_library().race_attn_fwd(
            ctypes.byref(shape), _ptr(Q), _ptr(K), _ptr(V), _ptr(W), float(beta), int(L), int(P),
            int(causal), _ptr(O), _ptr(state), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream))
        if rc != 0:
            raise RaceAttnError(rc, "race_attn_fwd")
        return O


def race_attn_bwd(Q, K, V, W, beta, L, P, causal, dO, O=None, dQ=None, dK=None, dV=None, state=None,
                  workspace=None, stream=None, want_dbeta=False, dbeta=None, want_dW=False, dW=None):
    """(dQ, dK, dV) of RACE attention for the output cotangent dO; allocates what is not given.
    With want_dbeta (or a float32 [B, H] `dbeta` given) also d(loss)/d(beta) per (b, h), returned
    next; the shared beta's gradient is its sum.  With want_dW (or a float32 [B, H, L, P, d] `dW`
    given) also d(loss)/d(W) per (b, h), returned last; a shared W's gradient is its sum over b
    and h, a per-head W's its sum over b."""
    with torch.cuda.device(Q.device):
        shape = _shape_of(Q, W, L, P)
        for n, t in (("K", K), ("V", V), ("dO", dO), ("Q", Q)):
            _check_like(n, t, Q)
        dQ = torch.empty_like(Q) if dQ is None else dQ
        dK = torch.empty_like(Q) if dK is None else dK
        dV = torch.empty_like(Q) if dV is None else dV
        for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV)):
            _check_like(n, t, Q)
        if dbeta is None and want_dbeta:
            dbeta = torch.empty((Q.shape[0], Q.shape[1]), dtype=torch.float32, device=Q.device)
        if dbeta is not None and (dbeta.dtype != torch.float32 or tuple(dbeta.shape) != tuple(Q.shape[:2])
                                  or not dbeta.is_contiguous() or dbeta.device != Q.device):
            raise ValueError("dbeta must be a contiguous float32 tensor of shape [B, H] on Q's device")
        dw_shape = (Q.shape[0], Q.shape[1], L, P, Q.shape[3])
        if dW is None and want_dW:
            dW = torch.empty(dw_shape, dtype=torch.float32, device=Q.device)
        if dW is not None and (dW.dtype != torch.float32 or tuple(dW.shape) != dw_shape or not dW.is_contiguous()
                               or dW.device != Q.device):
            raise ValueError("dW must be a contiguous float32 tensor of shape [B, H, L, P, d] on Q's device")
        ws_bytes = race_attn_workspace_bytes(shape, L, P, causal, 2 if dW is not None else 1)
        if ws_bytes == 0:
            raise RaceAttnError(-1, "race_attn_bwd")
        workspace = _bytes_buffer(ws_bytes, Q.device, workspace)
        rc = load_library().race_attn_bwd(
            ctypes.byref(shape), _ptr(Q), _ptr(K), _ptr(V), _ptr(W), float(beta), int(L), int(P),
            int(causal), _ptr(O), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dbeta), _ptr(dW), _ptr(state),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
        if rc != 0:
            raise RaceAttnError(rc, "race_attn_bwd")
        return (dQ, dK, dV) + ((dbeta,) if dbeta is not None else ()) + ((dW,) if dW is not None else ())


def race_attn_decode(q, k, v, W, beta, L, P, state, o=None, stream=None):
    """One causal decode step: q, k, v [B, H, 1, d] (float32 or bfloat16, CUDA); state float32
    [B, H, L * 2^P, d + 1] (updated in place).  Returns o [B, H, 1, d]."""
    with torch.cuda.device(q.device):
        shape = _shape_of(q, W, L, P)
        for n, t in (("k", k), ("v", v), ("q", q)):
            _check_like(n, t, q)
        want = (q.shape[0], q.shape[1], L << P, q.shape[3] + 1)
        if state.dtype != torch.float32 or tuple(state.shape) != want or not state.is_contiguous():
            raise ValueError("state must be a contiguous float32 tensor of shape %s" % (want,))
        o = torch.empty_like(q) if o is None else o
        _check_like("o", o, q)
        rc = load_library().race_attn_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(W), float(beta),
                                             int(L), int(P), _ptr(state), _ptr(o), _stream(stream))
        if rc != 0:
            raise RaceAttnError(rc, "race_attn_decode")
        return o


def race_attn_angular(Q, K, V, gamma, causal, O=None, stream=None):
    """Exact angular attention O_i = sum_j S_ij V_j / sum_j S_ij, S_ij = (1 - angle_ij / pi)^gamma
    (j <= i when causal), O(N^2): the reference RACE attention approximates.  Returns O."""
    with torch.cuda.device(Q.device):
        shape = _shape_of(Q)
        for n, t in (("K", K), ("V", V), ("Q", Q)):
            _check_like(n, t, Q)
        O = torch.empty_like(Q) if O is None else O
        _check_like("O", O, Q)
        rc = load_library().race_attn_angular(ctypes.byref(shape), _ptr(Q), _ptr(K), _ptr(V), float(gamma),
                                              int(bool(causal)), _ptr(O), _stream(stream))
        if rc != 0:
            raise RaceAttnError(rc, "race_attn_angular")
        return O


def race_attn_fwd_noalloc(Q, K, V, W, beta, L, P, causal, O=None, stream=None):
    """Forward pass through the entry point that allocates nothing and takes no workspace.

    For callers that cannot allocate device memory: the library uses its own built-in scratch
    buffer (RACE_NOALLOC_SCRATCH_BYTES per GPU) instead.  Calls that overlap on the GPU share
    that buffer and must be serialised by the caller.  Only O is allocated here, and only when
    it is not given.  Returns O.
    """
    with torch.cuda.device(Q.device):
        shape = _shape_of(Q, W, L, P)
        _check_like("K", K, Q)
        _check_like("V", V, Q)
        _check_like("Q", Q, Q)
        if O is None:
            O = torch.empty_like(Q)
        _check_like("O", O, Q)
        rc = load_library().race_attn_fwd_noalloc(
            ctypes.byref(shape), _ptr(Q), _ptr(K), _ptr(V), _ptr(W), float(beta), int(L), int(P), int(causal),
            _ptr(O), _stream(stream))
        if rc != 0:
            raise RaceAttnError(rc, "race_attn_fwd_noalloc")
        return O
