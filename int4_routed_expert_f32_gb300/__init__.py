"""Python binding of the GB300 quantized MoE layer (``libcoli_moe.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The functions carry the C ABI's names without the ``coli_moe_``
prefix (``include/coli_moe.h`` documents each one).  Tensors are
``torch.Tensor`` objects on the current CUDA device; PyTorch provides the
device memory and the stream, nothing else.

Importing this package raises if the shared library is missing: there is no
CPU or PyTorch fallback for any step.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcoli_moe.so")

OK, E_INVAL, E_NOSHAPE, E_NOMEM, E_CUDA, E_TIMEOUT, E_UNIMPL, E_DEVICE = 0, -1, -2, -3, -4, -5, -6, -7
PATH_AUTO, PATH_GEMV, PATH_GEMM = 0, 1, 2
GEMM_MIN_PAIRS_PER_EXPERT = 7   # AUTO runs the grouped GEMM when n_tok * top_k >= 7 * n_experts


def auto_uses_gemm(n_tok: int, top_k: int, n_experts: int, gemm_min_tokens: int = 0) -> bool:
    """The AUTO path's choice (mirrors the library's rule)."""
    if gemm_min_tokens > 0:
        return n_tok >= gemm_min_tokens
    return n_tok * top_k >= GEMM_MIN_PAIRS_PER_EXPERT * n_experts

EXPORTS = (
    "coli_moe_configure", "coli_moe_layer_forward", "coli_moe_layer_forward_residual",
    "coli_moe_layer_forward_hostio",
    "coli_moe_set_path", "coli_moe_get_device_status", "coli_moe_strerror", "coli_moe_release",
    "coli_moe_pack_int4", "coli_moe_timing_enable", "coli_moe_timing_read",
    "coli_moe_launch_count", "coli_moe_trace_enable", "coli_moe_trace_read",
    "coli_moe_dbg_quantize", "coli_moe_dbg_route",
    "coli_moe_dbg_dispatch", "coli_moe_dbg_rmsnorm", "coli_moe_dbg_block_dots",
    "coli_moe_dbg_forward_intermediates",
    "coli_moe_dbg_expert_hidden", "coli_moe_route_noalloc", "coli_moe_dbg_inject",
    "coli_moe_layer_forward_residual_prefetch", "coli_moe_pack_int8", "coli_moe_set_weight_bits",
    "coli_moe_dbg_block_dots_w8", "coli_moe_tier_configure", "coli_moe_tier_forward", "coli_moe_tier_stats",
    "coli_moe_tier_release", "coli_moe_dbg_stream_read", "coli_moe_dbg_check_guards",
)
INJECT_NONE, INJECT_ALLOC_FAIL, INJECT_LAUNCH_FAIL, INJECT_WAIT_TIMEOUT, INJECT_GUARD = 0, 1, 2, 3, 4


class ColiError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_lib.coli_moe_strerror(code).decode()} ({code})")


class _Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("ffn", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("routed_scale", ctypes.c_float),
                ("max_tok", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no fallback path)")
    L = ctypes.CDLL(LIB_PATH)
    P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "coli_moe_configure": ([ctypes.POINTER(_Shape)], i),
        "coli_moe_layer_forward": ([P, i, P, P, P, P, P, P, P, P], i),
        "coli_moe_layer_forward_residual": ([P, i, P, P, P, P, P, P, P, P], i),
        "coli_moe_layer_forward_hostio": ([P, i, P, P, P, P, P, P, P, P], i),
        "coli_moe_set_path": ([i, i], i),
        "coli_moe_get_device_status": ([P], i),
        "coli_moe_strerror": ([i], ctypes.c_char_p),
        "coli_moe_release": ([], None),
        "coli_moe_pack_int4": ([P, i, i, P, P, P], i),
        "coli_moe_timing_enable": ([i], i),
        "coli_moe_timing_read": ([ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)], i),
        "coli_moe_launch_count": ([], ctypes.c_longlong),
        "coli_moe_trace_enable": ([i], i),
        "coli_moe_trace_read": ([P, ctypes.c_longlong, ctypes.POINTER(ctypes.c_int),
                                 ctypes.POINTER(ctypes.c_int)], i),
        "coli_moe_dbg_quantize": ([P, i, P, P, P], i),
        "coli_moe_dbg_route": ([P, i, P, P, P, P, P, P], i),
        "coli_moe_dbg_dispatch": ([P, i, P, P, P, P, P], i),
        "coli_moe_dbg_rmsnorm": ([P, i, i, P, P], i),
        "coli_moe_dbg_block_dots": ([P, i, i, P, P, P], i),
        "coli_moe_dbg_forward_intermediates": ([P, i, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P], i),
        "coli_moe_dbg_expert_hidden": ([P, P, P, P, i, P, P, P, P], i),
        "coli_moe_route_noalloc": ([ctypes.POINTER(_Shape), P, i, P, P, P, P, P], i),
        "coli_moe_dbg_inject": ([i, ctypes.c_longlong], i),
        "coli_moe_layer_forward_residual_prefetch": ([P, i, P, P, P, P, P, P, P, P, P, P], i),
        "coli_moe_pack_int8": ([P, i, i, P, P, P], i),
        "coli_moe_set_weight_bits": ([i], i),
        "coli_moe_dbg_block_dots_w8": ([P, i, i, P, P, P], i),
        "coli_moe_tier_configure": ([i], i),
        "coli_moe_tier_forward": ([P, i, P, P, P, P, P, P, P, P], i),
        "coli_moe_tier_stats": ([ctypes.POINTER(ctypes.c_longlong)] * 3 + [ctypes.POINTER(ctypes.c_int)], i),
        "coli_moe_tier_release": ([], None),
        "coli_moe_dbg_stream_read": ([P, ctypes.c_size_t, i, i, i, P, P], i),
        "coli_moe_dbg_check_guards": ([ctypes.POINTER(ctypes.c_int)], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


_lib = _load()


def lib():
    return _lib


# Pointers travel as plain integers (the argtypes convert them); the current
# stream is read as a raw handle where this PyTorch exposes it, which keeps
# the per-call marshalling to a few microseconds.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _host_ptr(t):
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous host tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return _raw_stream(_cur_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(code: int, what: str):
    if code != OK:
        raise ColiError(code, what)


# --------------------------------------------------------------------------- #
def configure(hidden: int, ffn: int, n_experts: int, top_k: int, routed_scale: float, max_tok: int):
    s = _Shape(hidden, ffn, n_experts, top_k, routed_scale, max_tok)
    _check(_lib.coli_moe_configure(ctypes.byref(s)), "configure")


def release():
    _lib.coli_moe_release()


def set_path(path: int, gemm_min_tokens: int = 0):
    _check(_lib.coli_moe_set_path(path, gemm_min_tokens), "set_path")


def layer_forward(x, router_w, router_bias, expert_w4, expert_rowscale, shared_w4, shared_rowscale,
                  out=None, stream=None):
    if out is None:
        out = torch.empty_like(x)
    n_tok = x.shape[0] if x.dim() == 2 else 0
    _check(_lib.coli_moe_layer_forward(_ptr(x), n_tok, _ptr(router_w), _ptr(router_bias),
                                       _ptr(expert_w4), _ptr(expert_rowscale), _ptr(shared_w4),
                                       _ptr(shared_rowscale), _ptr(out), _stream(stream)),
           "layer_forward")
    return out


def layer_forward_residual(x, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                           shared_rowscale, out=None, stream=None):
    """out = x + MoE(x) (one layer of a stacked decoder, residual fused)."""
    if out is None:
        out = torch.empty_like(x)
    n_tok = x.shape[0] if x.dim() == 2 else 0
    _check(_lib.coli_moe_layer_forward_residual(_ptr(x), n_tok, _ptr(router_w), _ptr(router_bias),
                                                _ptr(expert_w4), _ptr(expert_rowscale),
                                                _ptr(shared_w4), _ptr(shared_rowscale), _ptr(out),
                                                _stream(stream)),
           "layer_forward_residual")
    return out


def layer_forward_residual_prefetch(x, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                                    shared_rowscale, next_router_w=None, next_shared_w4=None, out=None,
                                    stream=None):
    """layer_forward_residual, plus an L2 prefetch of the next layer's router
    weights and shared expert during this layer's expert-kernel tail."""
    if out is None:
        out = torch.empty_like(x)
    n_tok = x.shape[0] if x.dim() == 2 else 0
    _check(_lib.coli_moe_layer_forward_residual_prefetch(
        _ptr(x), n_tok, _ptr(router_w), _ptr(router_bias), _ptr(expert_w4), _ptr(expert_rowscale),
        _ptr(shared_w4), _ptr(shared_rowscale), _ptr(next_router_w), _ptr(next_shared_w4), _ptr(out),
        _stream(stream)), "layer_forward_residual_prefetch")
    return out


def tier_configure(n_slots: int):
    """Host-memory expert tier: an LRU cache of n_slots experts in HBM."""
    _check(_lib.coli_moe_tier_configure(int(n_slots)), "tier_configure")


def tier_forward(x, router_w, router_bias, host_expert_w, host_expert_rowscale, shared_w4, shared_rowscale,
                 out=None, stream=None):
    """The layer forward with the routed experts in host memory (host tensors,
    pinned for asynchronous copies); x, the router and the shared expert on
    the device."""
    if out is None:
        out = torch.empty_like(x)
    n_tok = x.shape[0] if x.dim() == 2 else 0
    _check(_lib.coli_moe_tier_forward(_ptr(x), n_tok, _ptr(router_w), _ptr(router_bias),
                                      _host_ptr(host_expert_w), _host_ptr(host_expert_rowscale),
                                      _ptr(shared_w4), _ptr(shared_rowscale), _ptr(out), _stream(stream)),
           "tier_forward")
    return out


def tier_stats():
    """(hits, misses, bytes copied to HBM, resident experts)."""
    h, m, b = ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_longlong(0)
    r = ctypes.c_int(0)
    _check(_lib.coli_moe_tier_stats(ctypes.byref(h), ctypes.byref(m), ctypes.byref(b), ctypes.byref(r)),
           "tier_stats")
    return h.value, m.value, b.value, r.value


def tier_release():
    _lib.coli_moe_tier_release()


def layer_forward_hostio(x_host, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                         shared_rowscale, out_host, stream=None):
    _check(_lib.coli_moe_layer_forward_hostio(_host_ptr(x_host), x_host.shape[0], _ptr(router_w),
                                              _ptr(router_bias), _ptr(expert_w4),
                                              _ptr(expert_rowscale), _ptr(shared_w4),
                                              _ptr(shared_rowscale), _host_ptr(out_host),
                                              _stream(stream)),
           "layer_forward_hostio")
    return out_host


class PreparedLayer:
    """One layer's device weights, checked and converted to C arguments once,
    for repeated forwards: the per-call marshalling is then the activation and
    output pointers only.  The tensors are kept alive by the object; they must
    not be resized or moved while it is used."""

    def __init__(self, router_w, router_bias, expert_w4, expert_rowscale, shared_w4, shared_rowscale):
        self._tensors = (router_w, router_bias, expert_w4, expert_rowscale, shared_w4, shared_rowscale)
        self._w = tuple(ctypes.c_void_p(_ptr(t)) for t in self._tensors)

    def forward(self, x, out=None, stream=None):
        if out is None:
            out = torch.empty_like(x)
        n_tok = x.shape[0] if x.dim() == 2 else 0
        _check(_lib.coli_moe_layer_forward(_ptr(x), n_tok, *self._w, _ptr(out), _stream(stream)), "layer_forward")
        return out

    def forward_hostio(self, x_host, out_host, stream=None):
        _check(_lib.coli_moe_layer_forward_hostio(_host_ptr(x_host), x_host.shape[0], *self._w,
                                                  _host_ptr(out_host), _stream(stream)),
               "layer_forward_hostio")
        return out_host


def get_device_status(stream=None) -> int:
    return _lib.coli_moe_get_device_status(_stream(stream))


def pack_int4(w, packed=None, scale=None, stream=None):
    rows, K = w.shape
    if packed is None:
        packed = torch.empty((rows, K // 2), dtype=torch.uint8, device=w.device)
    if scale is None:
        scale = torch.empty((rows,), dtype=torch.float32, device=w.device)
    _check(_lib.coli_moe_pack_int4(_ptr(w), rows, K, _ptr(packed), _ptr(scale), _stream(stream)),
           "pack_int4")
    return packed, scale


def pack_int8(w, q=None, scale=None, stream=None):
    """The int8 weight container: F32 rows [rows][K] -> (int8 codes, scales)."""
    rows, K = w.shape
    if q is None:
        q = torch.empty((rows, K), dtype=torch.int8, device=w.device)
    if scale is None:
        scale = torch.empty((rows,), dtype=torch.float32, device=w.device)
    _check(_lib.coli_moe_pack_int8(_ptr(w), rows, K, _ptr(q), _ptr(scale), _stream(stream)), "pack_int8")
    return q, scale


def set_weight_bits(bits: int):
    """Weight container of later forwards: 4 (packed int4) or 8 (int8 codes)."""
    _check(_lib.coli_moe_set_weight_bits(int(bits)), "set_weight_bits")


def timing_enable(on: bool = True):
    _check(_lib.coli_moe_timing_enable(1 if on else 0), "timing_enable")


def timing_read():
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int(0)
    _check(_lib.coli_moe_timing_read(ctypes.byref(ms), ctypes.byref(n)), "timing_read")
    return ms.value, n.value


def trace_enable(events_per_block: int):
    _check(_lib.coli_moe_trace_enable(events_per_block), "trace_enable")


def trace_read():
    """Returns (events: uint64 [blocks][n][2], blocks, n); see the header."""
    import numpy as np
    nb, ne = ctypes.c_int(0), ctypes.c_int(0)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    cap = sms * 32 * 4096 * 2
    buf = np.zeros(cap, np.uint64)
    _check(_lib.coli_moe_trace_read(buf.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(nb),
                                    ctypes.byref(ne)), "trace_read")
    n = nb.value * ne.value * 2
    return buf[:n].reshape(nb.value, ne.value, 2), nb.value, ne.value


def launch_count() -> int:
    return int(_lib.coli_moe_launch_count())


STATIC_MAX_TOK = 64


def route_noalloc(x, router_w, router_bias, hidden, n_experts, top_k, routed_scale, idx=None, w=None,
                  stream=None):
    """Router for callers that cannot allocate device memory (see the header):
    no configure() needed; scratch is a static device array of the library.
    ``idx``/``w`` may be given pre-allocated by the caller."""
    if x.dim() != 2 or x.shape[1] != hidden:
        raise ValueError(f"x must be [n_tok][{hidden}]")
    T = x.shape[0]
    if tuple(router_w.shape) != (n_experts, hidden):
        raise ValueError(f"router_w must be [{n_experts}][{hidden}]")
    if router_bias.numel() != n_experts:
        raise ValueError(f"router_bias must hold {n_experts} values")
    for name, t in (("x", x), ("router_w", router_w), ("router_bias", router_bias)):
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    if idx is None:
        idx = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    if idx.dtype != torch.int32 or idx.numel() < T * top_k:
        raise ValueError(f"idx must be int32 with at least n_tok*top_k = {T * top_k} elements")
    if w.dtype != torch.float32 or w.numel() < T * top_k:
        raise ValueError(f"w must be float32 with at least n_tok*top_k = {T * top_k} elements")
    for name, t in (("x", x), ("router_w", router_w), ("router_bias", router_bias), ("idx", idx), ("w", w)):
        if not t.is_cuda or t.device != x.device:
            raise ValueError(f"{name} must be on x's CUDA device")
    s = _Shape(hidden, 0, n_experts, top_k, routed_scale, 0)
    _check(_lib.coli_moe_route_noalloc(ctypes.byref(s), _ptr(x), T, _ptr(router_w), _ptr(router_bias),
                                       _ptr(idx), _ptr(w), _stream(stream)), "route_noalloc")
    return idx, w


def dbg_inject(what: int, arg: int = 0):
    """Failure injection for tests (see the header): INJECT_ALLOC_FAIL,
    INJECT_LAUNCH_FAIL, INJECT_WAIT_TIMEOUT (arg in microseconds),
    INJECT_GUARD (arg: a workspace guard region) or INJECT_NONE to clear."""
    _check(_lib.coli_moe_dbg_inject(int(what), int(arg)), "dbg_inject")


def dbg_check_guards():
    """(changed, total): how many workspace guard regions had changed since
    configure or the last check (they are restored), and how many there are.
    Synchronises the device; raises ColiError before configure."""
    n = ctypes.c_int(0)
    r = _lib.coli_moe_dbg_check_guards(ctypes.byref(n))
    if r < 0:
        raise ColiError(r, "dbg_check_guards")
    return r, n.value


# ---- stage entry points ---------------------------------------------------- #
def dbg_quantize(x, stream=None):
    n = x.numel()
    q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    d = torch.empty(x.shape[:-1] + (x.shape[-1] // 32,), dtype=torch.float32, device=x.device)
    _check(_lib.coli_moe_dbg_quantize(_ptr(x), n, _ptr(q), _ptr(d), _stream(stream)), "dbg_quantize")
    return q, d


def dbg_route(x, router_w, router_bias, top_k, want_logits=False, stream=None):
    T = x.shape[0]
    idx = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    logits = (torch.empty((T, router_w.shape[0]), dtype=torch.float32, device=x.device)
              if want_logits else None)
    _check(_lib.coli_moe_dbg_route(_ptr(x), T, _ptr(router_w), _ptr(router_bias), _ptr(idx),
                                   _ptr(w), _ptr(logits), _stream(stream)), "dbg_route")
    return (idx, w, logits) if want_logits else (idx, w)


def dbg_dispatch(idx, n_experts, stream=None):
    T, k = idx.shape
    dev = idx.device
    counts = torch.empty(n_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    _check(_lib.coli_moe_dbg_dispatch(_ptr(idx), T, _ptr(counts), _ptr(offsets), _ptr(perm),
                                      _ptr(inv), _stream(stream)), "dbg_dispatch")
    return counts, offsets, perm, inv


def dbg_block_dots(w4, q, stream=None):
    rows, K2 = w4.shape
    I = torch.empty((rows, 2 * K2 // 32), dtype=torch.int32, device=w4.device)
    _check(_lib.coli_moe_dbg_block_dots(_ptr(w4), rows, 2 * K2, _ptr(q), _ptr(I), _stream(stream)),
           "dbg_block_dots")
    return I


def dbg_block_dots_w8(w8, q, stream=None):
    rows, K = w8.shape
    I = torch.empty((rows, K // 32), dtype=torch.int32, device=w8.device)
    _check(_lib.coli_moe_dbg_block_dots_w8(_ptr(w8), rows, K, _ptr(q), _ptr(I), _stream(stream)),
           "dbg_block_dots_w8")
    return I


def dbg_stream_read(buf, n_bytes=None, sum_out=None, chunk=0, stages=0, blocks_per_sm=0, stream=None):
    """One bare read of the first n_bytes of the device tensor buf (default:
    all of it) in one launch (chunk / stages / blocks_per_sm 0: the expert
    kernel's arrangement); returns the device u64 checksum tensor (the sum of
    the four 32-bit words at every 1024-byte offset)."""
    nb = buf.numel() * buf.element_size() if n_bytes is None else int(n_bytes)
    if sum_out is None:
        sum_out = torch.empty(1, dtype=torch.int64, device=buf.device)
    _check(_lib.coli_moe_dbg_stream_read(_ptr(buf), nb, chunk, stages, blocks_per_sm, _ptr(sum_out),
                                         _stream(stream)), "dbg_stream_read")
    return sum_out


def dbg_forward_intermediates(x, router_w, router_bias, expert_w4, expert_rowscale, shared_w4,
                              shared_rowscale, hidden, ffn, top_k, stream=None):
    T = x.shape[0]
    dev = x.device
    R = T * top_k + T
    r = dict(
        out=torch.empty_like(x),
        qx=torch.empty((T, hidden), dtype=torch.int8, device=dev),
        dx=torch.empty((T, hidden // 32), dtype=torch.float32, device=dev),
        idx=torch.empty((T, top_k), dtype=torch.int32, device=dev),
        w=torch.empty((T, top_k), dtype=torch.float32, device=dev),
        qh=torch.empty((R, ffn), dtype=torch.int8, device=dev),
        dh=torch.empty((R, ffn // 32), dtype=torch.float32, device=dev),
        y=torch.empty((R, hidden), dtype=torch.float32, device=dev),
    )
    _check(_lib.coli_moe_dbg_forward_intermediates(
        _ptr(x), T, _ptr(router_w), _ptr(router_bias), _ptr(expert_w4), _ptr(expert_rowscale),
        _ptr(shared_w4), _ptr(shared_rowscale), _ptr(r["out"]), _ptr(r["qx"]), _ptr(r["dx"]),
        _ptr(r["idx"]), _ptr(r["w"]), _ptr(r["qh"]), _ptr(r["dh"]), _ptr(r["y"]),
        _stream(stream)), "dbg_forward_intermediates")
    return r


def dbg_rmsnorm(x, stream=None):
    """The stacked layer's pre-norm alone: x / sqrt(mean(x^2) + 1e-6) per token."""
    xn = torch.empty_like(x)
    _check(_lib.coli_moe_dbg_rmsnorm(_ptr(x), x.shape[0], x.shape[1], _ptr(xn), _stream(stream)),
           "dbg_rmsnorm")
    return xn


def dbg_expert_hidden(ew4, ers, qx, dx, ffn, stream=None):
    n = qx.shape[0]
    dev = qx.device
    h = torch.empty((n, ffn), dtype=torch.float32, device=dev)
    qh = torch.empty((n, ffn), dtype=torch.int8, device=dev)
    dh = torch.empty((n, ffn // 32), dtype=torch.float32, device=dev)
    _check(_lib.coli_moe_dbg_expert_hidden(_ptr(ew4), _ptr(ers), _ptr(qx), _ptr(dx), n, _ptr(h),
                                           _ptr(qh), _ptr(dh), _stream(stream)),
           "dbg_expert_hidden")
    return h, qh, dh
