"""Python handle on the plain-C oracle (``coli_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library never
imports this package, and this package never imports the product.

Every function here is argument marshalling around the C code; the arithmetic
lives in ``coli_oracle.c`` (see its header for the pages each step follows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "coli_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcoli_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no contraction of a*b+c into fma: every fma
    the oracle performs is an explicit fmaf)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i = ctypes.c_int
            f = ctypes.c_float
            L.orc_pack_int4_rows.argtypes = [P, i, i, P, P]
            L.orc_unpack_int4_rows.argtypes = [P, i, i, P]
            L.orc_pack_int8_rows.argtypes = [P, i, i, P, P]
            L.orc_block_dots_w8.argtypes = [P, i, i, P, P]
            L.orc_expert_ffn_w.argtypes = [P, i, P, i, i, P, P, P, P, P, P, P, P]
            L.orc_expert_ffn_w.restype = i
            L.orc_moe_forward_w.argtypes = [P, i, i, i, i, i, f, P, P, i, P, P, P, P, P,
                                            P, P, P, P, P, P]
            L.orc_moe_forward_w.restype = i
            L.orc_q8_0.argtypes = [P, i, P, P]
            L.orc_lrintf.argtypes = [f]
            L.orc_lrintf.restype = ctypes.c_long
            L.orc_exp.argtypes = [f]
            L.orc_exp.restype = f
            L.orc_sigmoid.argtypes = [f]
            L.orc_sigmoid.restype = f
            L.orc_router_logit.argtypes = [P, P, i]
            L.orc_router_logit.restype = f
            L.orc_route.argtypes = [P, i, i, P, P, i, i, f, P, P, P, P]
            L.orc_dispatch.argtypes = [P, i, i, i, P, P, P, P]
            L.orc_rmsnorm.argtypes = [P, i, i, f, P]
            L.orc_block_dots.argtypes = [P, i, i, P, P]
            L.orc_rows_dot.argtypes = [P, P, i, i, P, P, P]
            L.orc_expert_ffn.argtypes = [P, P, i, i, P, P, P, P, P, P, P, P]
            L.orc_moe_forward.argtypes = [P, i, i, i, i, i, f, P, P, P, P, P, P, P,
                                          P, P, P, P, P, P]
            L.orc_moe_forward.restype = i
            L.orc_num_threads.restype = i
            L.orc_set_threads.argtypes = [i]
            L.orc_set_threads.restype = None
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    return lib().orc_num_threads()


def set_threads(n: int) -> None:
    """Threads of the oracle's OpenMP loops (n <= 0: the default)."""
    lib().orc_set_threads(int(n))


def pack_int4_rows(w):
    """O1: F32 rows [R][K] -> (packed uint8 [R][K/2], scale float32 [R])."""
    w = _c(w, np.float32)
    R, K = w.shape
    packed = np.empty((R, K // 2), np.uint8)
    scale = np.empty(R, np.float32)
    lib().orc_pack_int4_rows(_p(w), R, K, _p(packed), _p(scale))
    return packed, scale


def unpack_int4_rows(packed):
    packed = _c(packed, np.uint8)
    R, K2 = packed.shape
    q = np.empty((R, 2 * K2), np.int8)
    lib().orc_unpack_int4_rows(_p(packed), R, 2 * K2, _p(q))
    return q


def pack_int8_rows(w):
    """The int8 container: F32 rows [R][K] -> (int8 codes [R][K], scale float32 [R])."""
    w = _c(w, np.float32)
    R, K = w.shape
    q = np.empty((R, K), np.int8)
    scale = np.empty(R, np.float32)
    lib().orc_pack_int8_rows(_p(w), R, K, _p(q), _p(scale))
    return q, scale


def q8_0(x):
    """O2: F32 [..., n] (n % 32 == 0) -> (int8 [..., n], F32 scales [..., n/32])."""
    x = _c(x, np.float32)
    n = x.shape[-1]
    flat = x.reshape(-1)
    q = np.empty(flat.shape, np.int8)
    d = np.empty(flat.size // 32, np.float32)
    lib().orc_q8_0(_p(flat), flat.size, _p(q), _p(d))
    return q.reshape(x.shape), d.reshape(x.shape[:-1] + (n // 32,))


def lrintf(v: float) -> int:
    return lib().orc_lrintf(float(np.float32(v)))


def exp(z: float) -> float:
    return lib().orc_exp(float(np.float32(z)))


def sigmoid(z: float) -> float:
    return lib().orc_sigmoid(float(np.float32(z)))


def router_logit(x, w) -> float:
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    return lib().orc_router_logit(_p(x), _p(w), x.size)


def route(x, W, bias, k, routed_scale, want_logits=False):
    """O3: returns (idx int32 [T][k], w F32 [T][k]) (+ logits, sigma [T][E])."""
    x = _c(x, np.float32)
    W = _c(W, np.float32)
    bias = _c(bias, np.float32)
    T, H = x.shape
    E = W.shape[0]
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    logits = np.empty((T, E), np.float32) if want_logits else None
    sigma = np.empty((T, E), np.float32) if want_logits else None
    lib().orc_route(_p(x), T, H, _p(W), _p(bias), E, k, float(routed_scale), _p(idx), _p(w),
                    _p(logits), _p(sigma))
    if want_logits:
        return idx, w, logits, sigma
    return idx, w


RMSNORM_EPS = 1e-6


def rmsnorm(x, eps=RMSNORM_EPS):
    """Pre-norm of a stacked layer: x_k / sqrt(mean(x^2) + eps) per token, the
    sum of squares in the router's canonical order (see orc_rmsnorm)."""
    x = _c(x, np.float32)
    T, H = x.shape
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), T, H, float(eps), _p(out))
    return out


def dispatch(idx, E):
    """O4: idx int32 [T][k] -> (counts [E], offsets [E+1], perm [T*k], inv [T*k])."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    lib().orc_dispatch(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    return counts, offsets, perm, inv


def block_dots(w4, q):
    """Per-block int32 dot products I [rows][K/32] of packed rows with int8 q [K]."""
    w4 = _c(w4, np.uint8)
    q = _c(q, np.int8)
    R, K2 = w4.shape
    I = np.empty((R, K2 * 2 // 32), np.int32)
    lib().orc_block_dots(_p(w4), R, 2 * K2, _p(q), _p(I))
    return I


def block_dots_w8(w8, q):
    """Per-block int32 dot products I [rows][K/32] of int8 rows with int8 q [K]."""
    w8 = _c(w8, np.int8)
    q = _c(q, np.int8)
    R, K = w8.shape
    I = np.empty((R, K // 32), np.int32)
    lib().orc_block_dots_w8(_p(w8), R, K, _p(q), _p(I))
    return I


def rows_dot(w4, s, q, d):
    w4 = _c(w4, np.uint8)
    s = _c(s, np.float32)
    q = _c(q, np.int8)
    d = _c(d, np.float32)
    R, K2 = w4.shape
    out = np.empty(R, np.float32)
    lib().orc_rows_dot(_p(w4), _p(s), R, 2 * K2, _p(q), _p(d), _p(out))
    return out


_E_WBITS = -1000000   # orc_moe_forward_w: weight container other than 4 or 8 bits


def _weight_bytes(w, H, F, wbits):
    """One expert's weights as flat bytes, checked against the container's
    size (3*F*H*wbits/8 bytes: gate, up and down)."""
    if wbits not in (4, 8):
        raise ValueError(f"oracle: unsupported weight container wbits={wbits} (4 or 8)")
    a = np.ascontiguousarray(w).view(np.uint8).reshape(-1)
    want = 3 * F * H * wbits // 8
    if a.size != want:
        raise ValueError(f"expert weights: {a.size} bytes, expected 3*F*H*{wbits}/8 = {want}")
    return a


def expert_ffn(ew4, ers, H, F, qx, dx, wbits=4):
    """O5 for one expert and one token: returns dict(qh, dh, y, g, u, h).
    ``wbits`` is the weight container: 4 (packed int4 bytes, 3*F*H/2) or 8
    (int8 codes as bytes, 3*F*H)."""
    ew4 = _weight_bytes(ew4, H, F, wbits)
    ers = _c(ers, np.float32).reshape(-1)
    if ers.size != 2 * F + H:
        raise ValueError(f"row scales: {ers.size} values, expected 2F+H = {2 * F + H}")
    qx = _c(qx, np.int8)
    dx = _c(dx, np.float32)
    qh = np.empty(F, np.int8)
    dh = np.empty(F // 32, np.float32)
    y = np.empty(H, np.float32)
    g = np.empty(F, np.float32)
    u = np.empty(F, np.float32)
    h = np.empty(F, np.float32)
    if lib().orc_expert_ffn_w(_p(ew4), int(wbits), _p(ers), H, F, _p(qx), _p(dx), _p(qh), _p(dh), _p(y),
                              _p(g), _p(u), _p(h)) != 0:
        raise ValueError(f"oracle: unsupported weight container wbits={wbits}")
    return dict(qh=qh, dh=dh, y=y, g=g, u=u, h=h)


def moe_forward(x, router_w, router_b, experts_w4, experts_rs, shared_w4, shared_rs, H, F, k,
                routed_scale, intermediates=False, wbits=4):
    """O6: the whole layer on T tokens.

    ``experts_w4``/``experts_rs`` are sequences of length E holding, per expert,
    its weight bytes and row scales (F32, 2F+H), or None for an expert no token
    selects.  ``wbits`` is the weight container: 4 (packed int4, 3*F*H/2
    bytes per expert) or 8 (int8 codes, 3*F*H bytes).
    """
    x = _c(x, np.float32)
    T = x.shape[0]
    E = len(experts_w4)
    keep = []
    W4 = (ctypes.c_void_p * E)()
    RS = (ctypes.c_void_p * E)()
    for e in range(E):
        if experts_w4[e] is None:
            W4[e] = None
            RS[e] = None
        else:
            a = _weight_bytes(experts_w4[e], H, F, wbits)
            b = _c(experts_rs[e], np.float32)
            if b.size != 2 * F + H:
                raise ValueError(f"expert {e}: {b.size} row scales, expected 2F+H = {2 * F + H}")
            keep += [a, b]
            W4[e] = a.ctypes.data
            RS[e] = b.ctypes.data
    rw = _c(router_w, np.float32)
    rb = _c(router_b, np.float32)
    sw = _weight_bytes(shared_w4, H, F, wbits)
    srs = _c(shared_rs, np.float32)
    if srs.size != 2 * F + H:
        raise ValueError(f"shared expert: {srs.size} row scales, expected 2F+H = {2 * F + H}")
    out = np.empty((T, H), np.float32)
    qx = np.empty((T, H), np.int8) if intermediates else None
    dx = np.empty((T, H // 32), np.float32) if intermediates else None
    idx = np.empty((T, k), np.int32) if intermediates else None
    w = np.empty((T, k), np.float32) if intermediates else None
    yr = np.empty((T, k, H), np.float32) if intermediates else None
    ys = np.empty((T, H), np.float32) if intermediates else None
    st = lib().orc_moe_forward_w(_p(x), T, H, F, E, k, float(routed_scale), _p(rw), _p(rb), int(wbits),
                                 ctypes.cast(W4, ctypes.c_void_p), ctypes.cast(RS, ctypes.c_void_p),
                                 _p(sw), _p(srs), _p(out), _p(qx), _p(dx), _p(idx), _p(w),
                                 _p(yr), _p(ys))
    if st == _E_WBITS:
        raise ValueError(f"oracle: unsupported weight container wbits={wbits}")
    if st != 0:
        raise ValueError(f"oracle: routed expert {-st - 1} was selected but not supplied")
    if intermediates:
        return out, dict(qx=qx, dx=dx, idx=idx, w=w, y_routed=yr, y_shared=ys)
    return out
