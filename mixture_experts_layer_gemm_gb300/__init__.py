"""Python binding of ``libmoe_layer.so`` (the C ABI in ``include/moe_layer.h``).

Argument marshalling only: every step of the MoE layer runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  Importing this
module loads the in-tree library and fails loudly if it has not been built
(``python -c "import __graft_entry__ as g; g.build()"``); there is no
fallback of any kind.

The functions carry the C names (``moe_layer_create``, ``moe_route``,
``moe_route_from_logits``, ``moe_route_from_topk``, ``moe_forward``,
``moe_destroy``, ...).  ``MoELayer`` bundles a layer handle with caller-owned
routing buffers allocated as torch tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_layer.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "moe_layer.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_OOM, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT, MOE_ERR_INTERNAL = range(7)
MOE_F32, MOE_BF16, MOE_I8 = 0, 1, 2
MOE_EXPERT_RELU2, MOE_EXPERT_SWIGLU = 0, 1
MOE_OPT_REGIME, MOE_OPT_TIMING, MOE_OPT_PAIR_TILES, MOE_OPT_HOST_TIMEOUT_MS = 1, 2, 3, 4
REGIME_AUTO, REGIME_DECODE, REGIME_BATCH = 0, 1, 2

DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16, "i8": MOE_I8}
EXPERTS = {"relu2": MOE_EXPERT_RELU2, "swiglu": MOE_EXPERT_SWIGLU}


class moe_config_t(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int), ("p", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("act_dtype", ctypes.c_int),
                ("weight_dtype", ctypes.c_int), ("expert", ctypes.c_int),
                ("has_router_bias", ctypes.c_int), ("paged", ctypes.c_int)]


class moe_routing_t(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("gather_index", ctypes.c_void_p), ("scatter_index", ctypes.c_void_p),
                ("logits", ctypes.c_void_p), ("T", ctypes.c_int)]


class moe_layer_info_t(ctypes.Structure):
    _fields_ = [("expert_bytes", ctypes.c_size_t), ("weight_bytes", ctypes.c_size_t),
                ("workspace_bytes", ctypes.c_size_t), ("decode_splits_up", ctypes.c_int),
                ("decode_splits_down", ctypes.c_int), ("num_sms", ctypes.c_int)]


MOE_NUM_PHASES = 8
PHASES = ("router", "permute", "gather", "up", "up_finish", "down", "combine", "copy")


class moe_timings_t(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * MOE_NUM_PHASES),
                ("launches", ctypes.c_uint64 * MOE_NUM_PHASES)]


class moe_stats_t(ctypes.Structure):
    _fields_ = [("kernel_launches", ctypes.c_uint64), ("forwards", ctypes.c_uint64), ("slot_hits", ctypes.c_uint64),
                ("slot_misses", ctypes.c_uint64), ("h2d_bytes", ctypes.c_uint64),
                ("h2d_ms", ctypes.c_double), ("forward_ms", ctypes.c_double),
                ("prefetch_copies", ctypes.c_uint64), ("prefetch_hits", ctypes.c_uint64),
                ("gemv_runs", ctypes.c_uint64), ("tc_runs", ctypes.c_uint64)]


MOE_PATH_NONE, MOE_PATH_SIMT, MOE_PATH_GEMV, MOE_PATH_TENSOR = 0, 1, 2, 3
PATHS = {MOE_PATH_NONE: "none", MOE_PATH_SIMT: "simt", MOE_PATH_GEMV: "gemv", MOE_PATH_TENSOR: "tensor-core"}


class moe_plan_t(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("mean_tokens", ctypes.c_int), ("tile_up", ctypes.c_int),
                ("tile_down", ctypes.c_int), ("splits_up", ctypes.c_int), ("splits_down", ctypes.c_int),
                ("pair_up", ctypes.c_int)]


class MoeError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                 3: "MOE_ERR_OOM", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_INTERNAL"}

_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "moe_layer_create": [ctypes.POINTER(moe_config_t), _vp, _vp, _vp, _vp, _vp, _vp, _i,
                         ctypes.POINTER(_vp)],
    "moe_destroy": [_vp],
    "moe_route": [_vp, _vp, _i, ctypes.POINTER(moe_routing_t), _vp],
    "moe_route_from_logits": [_vp, _vp, _i, ctypes.POINTER(moe_routing_t), _vp],
    "moe_route_from_topk": [_vp, _vp, _vp, _i, ctypes.POINTER(moe_routing_t), _vp],
    "moe_forward": [_vp, _vp, ctypes.POINTER(moe_routing_t), _vp, _vp],
    "moe_forward_static_scratch": [_vp, _vp, ctypes.POINTER(moe_routing_t), _vp, _vp],
    "moe_layer_set_option": [_vp, _i, _i],
    "moe_plan_forward": [ctypes.POINTER(moe_config_t), _i, _i, _i, _i, ctypes.POINTER(moe_plan_t)],
    "moe_layer_info": [_vp, ctypes.POINTER(moe_layer_info_t)],
    "moe_layer_stats": [_vp, ctypes.POINTER(moe_stats_t)],
    "moe_layer_timings": [_vp, ctypes.POINTER(moe_timings_t), _i],
    "moe_layer_sync_check": [_vp, _i, ctypes.POINTER(ctypes.c_uint32)],
    "moe_layer_read_expert": [_vp, _i, _i, _vp, _vp],
    "moe_pool_geometry": [_sz, _sz, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)],
    "moe_pool_create": [_sz, _sz, _i, _sz, ctypes.POINTER(_vp)],
    "moe_pool_destroy": [_vp],
    "moe_pool_query_log": [_vp, _vp, _vp, _vp, _vp, _i, ctypes.POINTER(_i)],
    "moe_pool_set_prefetch": [_vp, _i],
    "moe_selftest_bounded_wait": [ctypes.c_uint32, _vp, _vp],
    "moe_status_string": [_i],
    "moe_last_error": [],
    "moe_version": [],
}

_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def exported_names() -> Sequence[str]:
    return tuple(_SIGNATURES)


def _check(status):
    if status != MOE_OK:
        raise MoeError(status, lib().moe_last_error().decode(errors="replace"))
    return status


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


# ---- the C entry points, same names ------------------------------------------------
def moe_layer_create(cfg: moe_config_t, w_router, b_router, w1, w2, w3, pool=None,
                     layer_id: int = 0):
    """Host numpy arrays in; returns an opaque handle (int)."""
    E = cfg.E
    keep = [np.ascontiguousarray(a) for a in w1] + [np.ascontiguousarray(a) for a in w2]
    a1 = (ctypes.c_void_p * E)(*[keep[e].ctypes.data for e in range(E)])
    a2 = (ctypes.c_void_p * E)(*[keep[E + e].ctypes.data for e in range(E)])
    a3 = None
    if w3 is not None:
        k3 = [np.ascontiguousarray(a) for a in w3]
        keep += k3
        a3 = (ctypes.c_void_p * E)(*[a.ctypes.data for a in k3])
    wr = np.ascontiguousarray(w_router)
    br = None if b_router is None else np.ascontiguousarray(b_router, dtype=np.float32)
    out = ctypes.c_void_p()
    _check(lib().moe_layer_create(ctypes.byref(cfg), wr.ctypes.data,
                                  None if br is None else br.ctypes.data,
                                  ctypes.cast(a1, ctypes.c_void_p), ctypes.cast(a2, ctypes.c_void_p),
                                  None if a3 is None else ctypes.cast(a3, ctypes.c_void_p),
                                  pool, layer_id, ctypes.byref(out)))
    del keep
    return out.value


def moe_destroy(handle):
    _check(lib().moe_destroy(handle))


def moe_route(handle, x, T, routing: moe_routing_t, stream=None):
    _check(lib().moe_route(handle, _ptr(x), T, ctypes.byref(routing), _stream_ptr(stream)))


def moe_route_from_logits(handle, logits, T, routing: moe_routing_t, stream=None):
    _check(lib().moe_route_from_logits(handle, _ptr(logits), T, ctypes.byref(routing),
                                       _stream_ptr(stream)))


def moe_route_from_topk(handle, ids, w, T, routing: moe_routing_t, stream=None):
    _check(lib().moe_route_from_topk(handle, _ptr(ids), _ptr(w), T, ctypes.byref(routing),
                                     _stream_ptr(stream)))


def moe_forward(handle, x, routing: moe_routing_t, y, stream=None):
    _check(lib().moe_forward(handle, _ptr(x), ctypes.byref(routing), _ptr(y), _stream_ptr(stream)))


def moe_forward_static_scratch(handle, x, routing: moe_routing_t, y, stream=None):
    """moe_forward's decode path with its scratch in the library's static
    device array: for callers that cannot allocate device memory."""
    _check(lib().moe_forward_static_scratch(handle, _ptr(x), ctypes.byref(routing), _ptr(y),
                                            _stream_ptr(stream)))


def moe_layer_set_option(handle, opt, value):
    _check(lib().moe_layer_set_option(handle, opt, value))


def moe_plan_forward(cfg: moe_config_t, T, num_sms=152, regime=REGIME_AUTO, pair_tiles=1) -> moe_plan_t:
    """The launch plan moe_forward follows for T tokens (host arithmetic only)."""
    out = moe_plan_t()
    _check(lib().moe_plan_forward(ctypes.byref(cfg), T, num_sms, regime, pair_tiles, ctypes.byref(out)))
    return out


def moe_layer_info(handle) -> moe_layer_info_t:
    out = moe_layer_info_t()
    _check(lib().moe_layer_info(handle, ctypes.byref(out)))
    return out


def moe_layer_stats(handle) -> moe_stats_t:
    out = moe_stats_t()
    _check(lib().moe_layer_stats(handle, ctypes.byref(out)))
    return out


def moe_layer_timings(handle, reset=True):
    """{phase: (total ms, launches)} from the layer's launch events."""
    out = moe_timings_t()
    _check(lib().moe_layer_timings(handle, ctypes.byref(out), int(reset)))
    return {name: (out.ms[i], int(out.launches[i])) for i, name in enumerate(PHASES)}


def moe_layer_sync_check(handle, timeout_ms=10000):
    """Returns (status, flags) without raising on MOE_ERR_INVALID_ARG."""
    flags = ctypes.c_uint32(0)
    st = lib().moe_layer_sync_check(handle, timeout_ms, ctypes.byref(flags))
    if st not in (MOE_OK, MOE_ERR_INVALID_ARG):
        _check(st)
    return st, flags.value


def moe_layer_read_expert(handle, expert, which, shape, dtype):
    vals = np.empty(shape, dtype)
    scales = np.empty(shape[1], np.float32) if dtype == np.int8 else None
    _check(lib().moe_layer_read_expert(handle, expert, which, vals.ctypes.data,
                                       None if scales is None else scales.ctypes.data))
    return vals, scales


def moe_pool_geometry(budget_bytes, expert_bytes, ways):
    n, s = ctypes.c_int(), ctypes.c_int()
    _check(lib().moe_pool_geometry(budget_bytes, expert_bytes, ways, ctypes.byref(n), ctypes.byref(s)))
    return n.value, s.value


def moe_pool_create(budget_bytes, expert_bytes, ways, page_bytes=0):
    out = ctypes.c_void_p()
    _check(lib().moe_pool_create(budget_bytes, expert_bytes, ways, page_bytes, ctypes.byref(out)))
    return out.value


def moe_pool_destroy(pool):
    _check(lib().moe_pool_destroy(pool))


def moe_pool_set_prefetch(pool, max_experts):
    _check(lib().moe_pool_set_prefetch(pool, max_experts))


LOG_MISS, LOG_HIT, LOG_PREFETCH, LOG_PREFETCH_HIT = 0, 1, 2, 3


def moe_pool_query_log(pool, max_entries=1 << 20):
    """(layer, expert, kind, slot) arrays of the pool's lookups and prefetch
    inserts so far; kind is LOG_MISS, LOG_HIT, LOG_PREFETCH or LOG_PREFETCH_HIT."""
    arrs = [np.empty(max_entries, np.int32) for _ in range(4)]
    n = ctypes.c_int()
    _check(lib().moe_pool_query_log(pool, *[a.ctypes.data for a in arrs], max_entries,
                                    ctypes.byref(n)))
    return tuple(a[:n.value].copy() for a in arrs)


MOE_FLAG_EXPERT_ID, MOE_FLAG_DUPLICATE_ID, MOE_FLAG_GATHER_INDEX = 1, 2, 4
MOE_FLAG_OFFSETS, MOE_FLAG_WAIT_TIMEOUT, MOE_FLAG_TMEM_ALLOC = 8, 16, 32


def moe_selftest_bounded_wait(polls, stream=None):
    """(status, flags) of one kernel whose bounded wait cannot succeed; the
    expected status is MOE_ERR_TIMEOUT (not raised)."""
    flags = ctypes.c_uint32(0)
    st = lib().moe_selftest_bounded_wait(polls, ctypes.byref(flags),
                                         _stream_ptr(stream) if stream is not None else None)
    if st not in (MOE_ERR_TIMEOUT, MOE_ERR_INTERNAL, MOE_ERR_INVALID_ARG):
        _check(st)
    return st, flags.value


def moe_status_string(s) -> str:
    return lib().moe_status_string(s).decode()


def moe_last_error() -> str:
    return lib().moe_last_error().decode(errors="replace")


def moe_version() -> int:
    return lib().moe_version()


# ---- convenience: a layer plus its routing buffers (torch tensors) ------------------
class MoELayer:
    """One MoE FFN layer on the current CUDA device.

    ``layer`` is a ``workloads.Layer``-like object with host numpy arrays
    (w_router, b_router, w1, w2, w3) and a ``shape`` with m, p, E, k, expert,
    act, weight.  Routing buffers are torch tensors sized for max_tokens.
    """

    def __init__(self, layer, max_tokens: int, pool=None, layer_id: int = 0,
                 with_logits: bool = False, device=None):
        import torch
        s = layer.shape
        self.shape = s
        self.max_tokens = max_tokens
        self.cfg = moe_config_t(s.m, s.p, s.E, s.k, max_tokens, DTYPES[s.act], DTYPES[s.weight],
                                EXPERTS[s.expert], int(layer.b_router is not None),
                                int(pool is not None))
        self.handle = moe_layer_create(self.cfg, layer.w_router, layer.b_router, layer.w1,
                                       layer.w2, layer.w3, pool, layer_id)
        dev = device or torch.device("cuda", torch.cuda.current_device())
        n = max_tokens * s.k
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_ids = torch.empty(n, **i32)
        self.topk_w = torch.empty(n, dtype=torch.float32, device=dev)
        self.counts = torch.empty(s.E, **i32)
        self.offsets = torch.empty(s.E + 1, **i32)
        self.gather_index = torch.empty(n, **i32)
        self.scatter_index = torch.empty(n, **i32)
        self.logits = (torch.empty(max_tokens * s.E, dtype=torch.float32, device=dev)
                       if with_logits else None)
        self.routing = moe_routing_t(self.topk_ids.data_ptr(), self.topk_w.data_ptr(),
                                     self.counts.data_ptr(), self.offsets.data_ptr(),
                                     self.gather_index.data_ptr(), self.scatter_index.data_ptr(),
                                     None if self.logits is None else self.logits.data_ptr(), 0)

    def route(self, x, T: Optional[int] = None, stream=None):
        moe_route(self.handle, x, x.shape[0] if T is None else T, self.routing, stream)

    def route_from_logits(self, logits, T=None, stream=None):
        moe_route_from_logits(self.handle, logits, logits.shape[0] if T is None else T,
                              self.routing, stream)

    def route_from_topk(self, ids, w, T=None, stream=None):
        moe_route_from_topk(self.handle, ids, w, ids.shape[0] if T is None else T, self.routing,
                            stream)

    def forward(self, x, y, stream=None):
        moe_forward(self.handle, x, self.routing, y, stream)

    def set_regime(self, regime: int):
        moe_layer_set_option(self.handle, MOE_OPT_REGIME, regime)
        self._regime = regime

    def plan(self, T: int) -> moe_plan_t:
        """The launch plan this layer's forward takes for T tokens."""
        return moe_plan_forward(self.cfg, T, moe_layer_info(self.handle).num_sms,
                                getattr(self, "_regime", REGIME_AUTO), getattr(self, "_pair_tiles", 1))

    def set_timing(self, on: bool):
        moe_layer_set_option(self.handle, MOE_OPT_TIMING, int(on))

    def set_pair_tiles(self, on: bool):
        moe_layer_set_option(self.handle, MOE_OPT_PAIR_TILES, int(on))
        self._pair_tiles = int(on)

    def set_host_timeout_ms(self, ms: int):
        """Longest host wait of this layer's calls (-1: no limit)."""
        moe_layer_set_option(self.handle, MOE_OPT_HOST_TIMEOUT_MS, int(ms))

    def timings(self, reset=True):
        return moe_layer_timings(self.handle, reset)

    def info(self):
        return moe_layer_info(self.handle)

    def stats(self):
        return moe_layer_stats(self.handle)

    def sync_check(self, timeout_ms=10000):
        return moe_layer_sync_check(self.handle, timeout_ms)

    def close(self):
        if self.handle:
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
