"""Thin ctypes binding of libcoli_moe.so with the same names as the C ABI (include/coli_moe.h).

Argument marshalling only: torch tensors are checked for device, dtype and contiguity and passed
as raw pointers; every step of the computation runs in the library's CUDA kernels. Importing this
module loads the in-tree library and fails loudly if it has not been built (there is no CPU
fallback): build it with ``python -m int4_grouped_expert_router_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcoli_moe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "coli_moe.h")

_lib = None


def _constants():
    consts = {}
    with open(HEADER) as f:
        for m in re.finditer(r"^#define (COLI_\w+)\s+(-?\d+)", f.read(), re.M):
            consts[m.group(1)] = int(m.group(2))
    return consts


_C = _constants()
COLI_OK = _C["COLI_OK"]
COLI_E_INVAL = _C["COLI_E_INVAL"]
COLI_E_OOM = _C["COLI_E_OOM"]
COLI_E_CUDA = _C["COLI_E_CUDA"]
COLI_E_INJECTED = _C["COLI_E_INJECTED"]
COLI_E_FORMAT = _C["COLI_E_FORMAT"]
COLI_E_NONFINITE = _C["COLI_E_NONFINITE"]
COLI_E_ROUTE = _C["COLI_E_ROUTE"]
COLI_E_TIMEOUT = _C["COLI_E_TIMEOUT"]
COLI_DTYPE_F32 = _C["COLI_DTYPE_F32"]
COLI_DTYPE_BF16 = _C["COLI_DTYPE_BF16"]
COLI_MAX_EXPERTS = _C["COLI_MAX_EXPERTS"]
COLI_MAX_K = _C["COLI_MAX_K"]
COLI_MAX_ISSUES = _C["COLI_MAX_ISSUES"]

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_U64 = ctypes.c_uint64

SIGNATURES = {
    "coli_init": (_I, [ctypes.POINTER(_P), _I, _P]),
    "coli_destroy": (None, [_P]),
    "coli_set_stream": (_I, [_P, _P]),
    "coli_last_error": (ctypes.c_char_p, [_P]),
    "coli_last_code": (_I, [_P]),
    "coli_check_error": (_I, [_P]),
    "coli_reserve": (_I, [_P, _I, _I, _I, _I, _I]),
    "coli_router_select": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _I, _F, _P, _P, _P]),
    "coli_router_select_noalloc": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _I, _F, _P, _P, _P]),
    "coli_router_select_shared": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _I, _F, _I, _P, _P, _P]),
    "coli_routes_shard": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "coli_partials_reduce": (_I, [_P, _P, _I, _I, _I, _P, _I, _P]),
    "coli_ans_encode_host": (_I, [_P, _U64, _P, _U64, ctypes.POINTER(ctypes.c_uint64)]),
    "coli_ans_upload": (_U64, [_P, _P, _U64]),
    "coli_ans_info": (_I, [_P, _U64, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "coli_ans_decode": (_I, [_P, _U64, _P]),
    "coli_ans_free": (_I, [_P, _U64]),
    "coli_ans_w4_linear": (_I, [_P, _U64, _P, _I, _I, _I, _P, _I, _P, _P]),
    "coli_expert_upload": (_U64, [_P, _P, _P, _I, _I, _I]),
    "coli_expert_free": (_I, [_P, _U64]),
    "coli_tensor_shape": (_I, [_P, _U64, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                              ctypes.POINTER(ctypes.c_int)]),
    "coli_w4_linear": (_I, [_P, _U64, _P, _I, _I, _P, _P]),
    "coli_expert_table_set": (_I, [_P, _I, _U64, _U64, _U64]),
    "coli_expert_group": (_I, [_P, _P, _I, _I, _P, _P, _P, _I, _P, _P]),
    "coli_expert_group_issue": (_I, [_P, _P, _I, _I, _P, _P, _P, _I]),
    "coli_expert_group_take": (_I, [_P, _P, _P]),
    "coli_profile_enable": (_I, [_P, _I]),
    "coli_profile_read": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]),
}

COLI_KERNEL_ROUTER = _C["COLI_KERNEL_ROUTER"]
COLI_KERNEL_GATEUP = _C["COLI_KERNEL_GATEUP"]
COLI_KERNEL_DOWN = _C["COLI_KERNEL_DOWN"]
COLI_KERNEL_COMBINE = _C["COLI_KERNEL_COMBINE"]
COLI_KERNEL_LINEAR = _C["COLI_KERNEL_LINEAR"]


class ColiError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


def library():
    """Load libcoli_moe.so (once). Raises if the library has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m int4_grouped_expert_router_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def act_dtype(t):
    if t.dtype == torch.float32:
        return COLI_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return COLI_DTYPE_BF16
    raise ValueError("activations must be float32 or bfloat16")


def _check(ctx, rc, what):
    if rc != COLI_OK:
        raise ColiError(rc, f"{what}: {coli_last_error(ctx)}")
    return rc


def coli_init(device=0, stream=None):
    """Create a context; ``stream`` is a torch.cuda.Stream (default: the current stream)."""
    lib = library()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    out = ctypes.c_void_p()
    rc = lib.coli_init(ctypes.byref(out), device, ctypes.c_void_p(stream.cuda_stream))
    if rc != COLI_OK:
        raise ColiError(rc, "coli_init failed")
    return out


def coli_destroy(ctx):
    library().coli_destroy(ctx)


def coli_set_stream(ctx, stream):
    return _check(ctx, library().coli_set_stream(ctx, ctypes.c_void_p(stream.cuda_stream)), "coli_set_stream")


def coli_last_error(ctx):
    s = library().coli_last_error(ctx)
    return s.decode() if s else ""


def coli_last_code(ctx):
    return library().coli_last_code(ctx)


def coli_check_error(ctx):
    """Synchronise and return (and clear) the device error word: 0 when clean."""
    return library().coli_check_error(ctx)


def coli_reserve(ctx, max_S, max_E, max_K, max_D, max_I):
    return _check(ctx, library().coli_reserve(ctx, max_S, max_E, max_K, max_D, max_I), "coli_reserve")


def _router_args(x, Wr, bias, K, idx, w, n_sel, slots=None):
    S, D = x.shape
    slots = K if slots is None else slots
    E = Wr.shape[0]
    _dev(x, name="x")
    _dev(Wr, torch.float32, "Wr")
    _dev(bias, torch.float32, "bias")
    _dev(idx, torch.int32, "idx")
    _dev(w, torch.float32, "w")
    _dev(n_sel, torch.int32, "n_sel")
    if Wr.shape[1] != D or idx.numel() != S * slots or w.numel() != S * slots or \
            (n_sel is not None and n_sel.numel() != S):
        raise ValueError("router_select: inconsistent shapes")
    if bias is not None and bias.numel() != E:
        raise ValueError("router_select: bias must have E entries")
    return S, D, E


def coli_router_select(ctx, x, Wr, bias, K, topp, norm_topk, routed_scale, idx, w, n_sel=None):
    S, D, E = _router_args(x, Wr, bias, K, idx, w, n_sel)
    rc = library().coli_router_select(ctx, _ptr(x), act_dtype(x), S, D, _ptr(Wr), _ptr(bias), E, K, float(topp),
                                      int(bool(norm_topk)), float(routed_scale), _ptr(idx), _ptr(w), _ptr(n_sel))
    return _check(ctx, rc, "coli_router_select")


def coli_router_select_shared(ctx, x, Wr, bias, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel=None):
    """coli_router_select plus the shared expert ``shared`` after each token's kept slots (weight 1):
    idx and w are [S x (K+1)]."""
    S, D, E = _router_args(x, Wr, bias, K, idx, w, n_sel, slots=K + 1)
    rc = library().coli_router_select_shared(ctx, _ptr(x), act_dtype(x), S, D, _ptr(Wr), _ptr(bias), E, K, float(topp),
                                             int(bool(norm_topk)), float(routed_scale), int(shared), _ptr(idx), _ptr(w),
                                             _ptr(n_sel))
    return _check(ctx, rc, "coli_router_select_shared")


def coli_router_select_noalloc(ctx, x, Wr, bias, K, topp, norm_topk, routed_scale, idx, w, n_sel=None):
    """coli_router_select with the library's fixed device scratch (S * E <= 65536): allocates nothing."""
    S, D, E = _router_args(x, Wr, bias, K, idx, w, n_sel)
    rc = library().coli_router_select_noalloc(ctx, _ptr(x), act_dtype(x), S, D, _ptr(Wr), _ptr(bias), E, K,
                                              float(topp), int(bool(norm_topk)), float(routed_scale), _ptr(idx),
                                              _ptr(w), _ptr(n_sel))
    return _check(ctx, rc, "coli_router_select_noalloc")


def coli_expert_upload(ctx, packed, scales, O, I, gs):
    """Upload one int4 tensor from host or device tensors; returns the handle (raises on failure)."""
    if packed.dtype != torch.uint8 or scales.dtype != torch.float32:
        raise ValueError("packed must be uint8 and scales float32")
    if not (packed.is_contiguous() and scales.is_contiguous()):
        raise ValueError("packed and scales must be contiguous")
    if packed.numel() != O * ((I + 1) // 2):
        raise ValueError("packed must hold O * ceil(I/2) bytes")
    nsc = O if gs == 0 else O * ((I + gs - 1) // gs) if gs > 0 else -1
    if scales.numel() != nsc:
        raise ValueError("scale count must be O (gs=0) or O*ceil(I/gs)")
    h = library().coli_expert_upload(ctx, _ptr(packed), _ptr(scales), O, I, gs)
    if h == 0:
        raise ColiError(library().coli_last_code(ctx), f"coli_expert_upload: {coli_last_error(ctx)}")
    return h


def coli_expert_free(ctx, handle):
    return _check(ctx, library().coli_expert_free(ctx, handle), "coli_expert_free")


def coli_tensor_shape(ctx, handle):
    """(O, I, gs) of an uploaded tensor."""
    O, I, gs = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(ctx, library().coli_tensor_shape(ctx, handle, ctypes.byref(O), ctypes.byref(I), ctypes.byref(gs)),
           "coli_tensor_shape")
    return O.value, I.value, gs.value


def coli_w4_linear(ctx, W, x, resid, y):
    """y = resid + W x for every row of x ([S x I] -> [S x O]); resid may be None."""
    O, I, _ = coli_tensor_shape(ctx, W)
    _dev(x, name="x")
    _dev(resid, x.dtype, "resid")
    _dev(y, x.dtype, "y")
    S = x.shape[0]
    if x.dim() != 2 or x.shape[1] != I or tuple(y.shape) != (S, O) or (resid is not None and resid.shape != y.shape):
        raise ValueError("w4_linear: x must be [S x I] and y, resid [S x O] for the tensor's O and I")
    rc = library().coli_w4_linear(ctx, W, _ptr(x), act_dtype(x), S, _ptr(resid), _ptr(y))
    return _check(ctx, rc, "coli_w4_linear")


def coli_expert_table_set(ctx, e, gate, up, down):
    return _check(ctx, library().coli_expert_table_set(ctx, e, gate, up, down), "coli_expert_table_set")


def coli_expert_group(ctx, x_rows, idx, w, n_sel, K, resid, y):
    S = x_rows.shape[0]
    _dev(x_rows, name="x_rows")
    _dev(idx, torch.int32, "idx")
    _dev(w, torch.float32, "w")
    _dev(n_sel, torch.int32, "n_sel")
    _dev(resid, x_rows.dtype, "resid")
    _dev(y, x_rows.dtype, "y")
    if idx.numel() != S * K or w.numel() != S * K or y.shape != x_rows.shape or \
            (resid is not None and resid.shape != x_rows.shape) or (n_sel is not None and n_sel.numel() != S):
        raise ValueError("expert_group: inconsistent shapes")
    rc = library().coli_expert_group(ctx, _ptr(x_rows), act_dtype(x_rows), S, _ptr(idx), _ptr(w), _ptr(n_sel), K,
                                     _ptr(resid), _ptr(y))
    return _check(ctx, rc, "coli_expert_group")


def coli_expert_group_issue(ctx, x_rows, idx, w, n_sel, K):
    """Issue one group of routes; returns its issue index in the current round."""
    S = x_rows.shape[0]
    _dev(x_rows, name="x_rows")
    _dev(idx, torch.int32, "idx")
    _dev(w, torch.float32, "w")
    _dev(n_sel, torch.int32, "n_sel")
    if idx.numel() != S * K or w.numel() != S * K or (n_sel is not None and n_sel.numel() != S):
        raise ValueError("expert_group_issue: inconsistent shapes")
    rc = library().coli_expert_group_issue(ctx, _ptr(x_rows), act_dtype(x_rows), S, _ptr(idx), _ptr(w), _ptr(n_sel), K)
    if rc < 0:
        raise ColiError(rc, f"coli_expert_group_issue: {coli_last_error(ctx)}")
    return rc


def coli_expert_group_take(ctx, resid, y):
    """Join the round's issued partial sums, in issue order, to the residual: y = resid + sum."""
    _dev(resid, y.dtype, "resid")
    _dev(y, name="y")
    if resid is not None and resid.shape != y.shape:
        raise ValueError("expert_group_take: inconsistent shapes")
    return _check(ctx, library().coli_expert_group_take(ctx, _ptr(resid), _ptr(y)), "coli_expert_group_take")


def coli_routes_shard(ctx, idx, w, n_sel, rank, world, idx_out, w_out, n_out):
    """This rank's kept routes (expert e mod world == rank) moved to the front of each row."""
    S, K = idx.shape
    for t, name, dt in ((idx, "idx", torch.int32), (w, "w", torch.float32), (idx_out, "idx_out", torch.int32),
                        (w_out, "w_out", torch.float32)):
        _dev(t, dt, name)
        if tuple(t.shape) != (S, K):
            raise ValueError(f"routes_shard: {name} must be [S x K]")
    _dev(n_sel, torch.int32, "n_sel")
    _dev(n_out, torch.int32, "n_out")
    if n_out.numel() != S or (n_sel is not None and n_sel.numel() != S):
        raise ValueError("routes_shard: n_sel and n_out must have S entries")
    rc = library().coli_routes_shard(ctx, _ptr(idx), _ptr(w), _ptr(n_sel), S, K, rank, world, _ptr(idx_out),
                                     _ptr(w_out), _ptr(n_out))
    return _check(ctx, rc, "coli_routes_shard")


def coli_partials_reduce(ctx, parts, resid, y):
    """y = resid + (((p_0 + p_1) + ...) in order) for parts [n x S x D] f32; resid may be None."""
    _dev(parts, torch.float32, "parts")
    _dev(y, name="y")
    _dev(resid, y.dtype, "resid")
    n, S, D = parts.shape
    if tuple(y.shape) != (S, D) or (resid is not None and resid.shape != y.shape):
        raise ValueError("partials_reduce: y and resid must be [S x D]")
    rc = library().coli_partials_reduce(ctx, _ptr(parts), n, S, D, _ptr(resid), act_dtype(y), _ptr(y))
    return _check(ctx, rc, "coli_partials_reduce")


def coli_ans_encode_host(data: bytes) -> bytes:
    """The library's encoded stream of ``data`` (host only; no GPU needed)."""
    lib = library()
    n = len(data)
    src = ctypes.create_string_buffer(bytes(data), n)
    need = ctypes.c_uint64()
    lib.coli_ans_encode_host(src, n, None, 0, ctypes.byref(need))
    out = ctypes.create_string_buffer(need.value)
    rc = lib.coli_ans_encode_host(src, n, out, need.value, ctypes.byref(need))
    if rc != COLI_OK:
        raise ColiError(rc, "coli_ans_encode_host failed")
    return out.raw[:need.value]


def coli_ans_upload(ctx, data: bytes):
    src = ctypes.create_string_buffer(bytes(data), len(data))
    h = library().coli_ans_upload(ctx, src, len(data))
    if h == 0:
        raise ColiError(library().coli_last_code(ctx), f"coli_ans_upload: {coli_last_error(ctx)}")
    return h


def coli_ans_info(ctx, handle):
    """(raw bytes, stored bytes) of an uploaded stream."""
    raw, stored = ctypes.c_uint64(), ctypes.c_uint64()
    _check(ctx, library().coli_ans_info(ctx, handle, ctypes.byref(raw), ctypes.byref(stored)), "coli_ans_info")
    return raw.value, stored.value


def coli_ans_w4_linear(ctx, handle, scales, O, I, gs, x, resid, y):
    """y = resid + W x for an int4 tensor W [O x I] kept as a compressed stream (fused decode + GEMV);
    scales is the f32 scale tensor of W on the device, x [I] (or [1 x I]), y and resid [O]."""
    _dev(scales, torch.float32, "scales")
    _dev(x, name="x")
    _dev(resid, x.dtype, "resid")
    _dev(y, x.dtype, "y")
    if x.numel() != I or y.numel() != O or (resid is not None and resid.numel() != O):
        raise ValueError("ans_w4_linear: x must hold I values and y, resid O")
    rc = library().coli_ans_w4_linear(ctx, handle, _ptr(scales), O, I, gs, _ptr(x), act_dtype(x), _ptr(resid),
                                      _ptr(y))
    return _check(ctx, rc, "coli_ans_w4_linear")


def coli_ans_decode(ctx, handle, out):
    """Decode an uploaded stream into ``out`` (a CUDA uint8 tensor of the raw size)."""
    _dev(out, torch.uint8, "out")
    raw, _ = coli_ans_info(ctx, handle)
    if out.numel() != raw:
        raise ValueError("ans_decode: out must hold the raw size")
    return _check(ctx, library().coli_ans_decode(ctx, handle, _ptr(out)), "coli_ans_decode")


def coli_ans_free(ctx, handle):
    return _check(ctx, library().coli_ans_free(ctx, handle), "coli_ans_free")


def coli_profile_enable(ctx, on):
    return _check(ctx, library().coli_profile_enable(ctx, int(bool(on))), "coli_profile_enable")


def coli_profile_read(ctx, kind):
    """(total_ms, launches) of one kernel kind since its previous read (synchronises)."""
    ms = ctypes.c_double()
    n = ctypes.c_longlong()
    _check(ctx, library().coli_profile_read(ctx, kind, ctypes.byref(ms), ctypes.byref(n)), "coli_profile_read")
    return ms.value, n.value
