"""fp64 CPU oracle for one MoE FFN layer's forward pass (ctypes over moe_oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  It shares no code with
the CUDA library (``mixture_experts_layer_gemm_gb300``) and never calls it;
the two see the same seeded inputs from ``workloads.py`` and nothing else.

Functions follow the pages' statement of the problem:
  router_logits  -- router GEMM (HARMOEny write-up, part 1 "What is MoE"; the
                    GPU gating network of the expert-cache article, section 3.1)
  topk           -- top-k on the logits, ties to the lower id, softmax
                    renormalised over the k chosen (reading of the pages)
  permute        -- histogram / exclusive scan / stable scatter: the one-device
                    form of the dispatch (HARMOEny write-up, part 2, part 3.3)
  quantize_cols  -- per-column symmetric int8 (DeepSpeed-Inference article,
                    part 4, INT8 support; the scheme is this build's reading)
  expert         -- one expert x.W1.W2 (ReLU) or SiLU(x.W1)*(x.W3).W2
                    (HARMOEny write-up, part 3.2)
  layer          -- weighted combine over the k experts, ascending slot order
  cache_replay   -- N-index x M-way set-associative LRU expert cache
                    (expert-cache article, section 2.2)

Parity status of each function is listed in the module ``PINS`` table;
every function here is pinned by a ``-m "not gpu"`` test.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, I8, F64 = 0, 1, 2, 3
RELU2, SWIGLU = 0, 1

PINS = {
    "router_logits": "numpy fp64 matmul on the same inputs; one-hot closed forms",
    "topk": "brute force over all k-subsets; sigmoid closed form for k=2; full softmax",
    "permute": "library stable sort; bijection / monotone-offset invariants",
    "quantize_cols": "hand-built columns with known codes (tests/golden)",
    "expert": "|O| closed form (op counter); dense-MLP numpy reduction; one-hot entries",
    "layer": "identical experts make y routing-independent; E=1,k=1 dense MLP",
    "cache_replay": "slot-count formulas of the expert-cache article; hand traces",
    "cache_replay_calls": "equals cache_replay with prefetch off; hand traces with prefetch; "
                          "closed-form hit counts for repeated expert sets",
}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, dp = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        L.moe_oracle_router_logits.argtypes = [vp, i32, vp, i32, dp, i32, i32, i32, dp, dp]
        L.moe_oracle_topk.argtypes = [dp, i32, i32, i32, vp, dp]
        L.moe_oracle_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.moe_oracle_quantize_cols.argtypes = [vp, i32, i32, i32, vp, vp]
        L.moe_oracle_expert.argtypes = [vp, i32, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32,
                                        dp, dp, vp]
        L.moe_oracle_layer.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, i32,
                                       vp, vp, vp, i32, vp, dp, vp, i32, dp, vp, i32]
        L.moe_oracle_cache_replay.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        L.moe_oracle_cache_replay_calls.argtypes = [i32, i32, i32, vp, i32, vp, i32, i32, vp, vp,
                                                    vp, vp, i32, vp]
        for f in (L.moe_oracle_router_logits, L.moe_oracle_topk, L.moe_oracle_permute,
                  L.moe_oracle_quantize_cols, L.moe_oracle_expert, L.moe_oracle_layer,
                  L.moe_oracle_cache_replay, L.moe_oracle_cache_replay_calls):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a):
    """Element type code of a numpy array.  bf16 data is carried as uint16."""
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.int8:
        return I8
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported element type {a.dtype}")


def _c(a):
    return np.ascontiguousarray(a)


def router_logits(x, w_router, bias=None, with_abssum=False):
    """logits[t, e] = sum_c x[t, c] w_router[c, e] (+ bias[e]) in fp64."""
    x, w = _c(x), _c(w_router)
    T, m = x.shape
    m2, E = w.shape
    assert m == m2
    b = None if bias is None else _c(np.asarray(bias, dtype=np.float64))
    logits = np.empty((T, E), np.float64)
    mag = np.empty((T, E), np.float64) if with_abssum else None
    _check(lib().moe_oracle_router_logits(_ptr(x), _dtype_code(x), _ptr(w), _dtype_code(w),
                                          _ptr(b), T, m, E, _ptr(logits), _ptr(mag)),
           "router_logits")
    return (logits, mag) if with_abssum else logits


def topk(logits, k):
    """(ids [T,k] int32, weights [T,k] fp64) from fp64 logits [T,E]."""
    l = _c(np.asarray(logits, dtype=np.float64))
    T, E = l.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(lib().moe_oracle_topk(_ptr(l), T, E, k, _ptr(ids), _ptr(w)), "topk")
    return ids, w


def permute(ids, E):
    """(counts[E], offsets[E+1], gather[T*k], scatter[T*k]) for ids [T,k]."""
    ids = _c(np.asarray(ids, dtype=np.int32))
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    gather = np.empty(T * k, np.int32)
    scatter = np.empty(T * k, np.int32)
    _check(lib().moe_oracle_permute(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets),
                                    _ptr(gather), _ptr(scatter)), "permute")
    return counts, offsets, gather, scatter


def quantize_cols(w):
    """Per-column symmetric int8 codes and fp32 scales of a rows x cols matrix."""
    w = _c(w)
    rows, cols = w.shape
    q = np.empty((rows, cols), np.int8)
    s = np.empty(cols, np.float32)
    _check(lib().moe_oracle_quantize_cols(_ptr(w), _dtype_code(w), rows, cols, _ptr(q), _ptr(s)),
           "quantize_cols")
    return q, s


def expert(x_row, w1, w2, w3=None, kind=RELU2, scales=(None, None, None), count_ops=False):
    """One expert on one token.  Returns (h [p], out [m]) or (h, out, ops[4])."""
    x_row, w1, w2 = _c(x_row), _c(w1), _c(w2)
    w3 = None if w3 is None else _c(w3)
    m, p = w1.shape
    s1, s2, s3 = (None if s is None else _c(np.asarray(s, np.float32)) for s in scales)
    h = np.empty(p, np.float64)
    out = np.empty(m, np.float64)
    ops = np.zeros(4, np.int64) if count_ops else None
    _check(lib().moe_oracle_expert(_ptr(x_row), _dtype_code(x_row), _ptr(w1), _ptr(w2),
                                   _ptr(w3), _dtype_code(w1), _ptr(s1), _ptr(s2), _ptr(s3),
                                   m, p, kind, _ptr(h), _ptr(out), _ptr(ops)), "expert")
    return (h, out, ops) if count_ops else (h, out)


def _ptr_array(mats):
    arr = (ctypes.c_void_p * len(mats))(*[m.ctypes.data for m in mats])
    return arr


def layer(x, w1, w2, w3, ids, weights, kind, scales=None, tokens=None,
          count_ops=False, nthreads=0):
    """y[s] = sum_j weights[t, j] * expert_{ids[t, j]}(x[t]) for t = tokens[s].

    w1, w2, w3: lists of E row-major matrices (w3 None for the ReLU form).
    scales: None, or (s1, s2, s3) lists of per-column fp32 scales (int8).
    Returns y [n, m] fp64, or (y, ops [E, 4]) with count_ops.
    """
    x = _c(x)
    T, m = x.shape
    E = len(w1)
    ids = _c(np.asarray(ids, np.int32))
    weights = _c(np.asarray(weights, np.float64))
    k = ids.shape[1]
    w1 = [_c(a) for a in w1]
    w2 = [_c(a) for a in w2]
    p = w1[0].shape[1]
    w3l = None if w3 is None else [_c(a) for a in w3]
    keep = [w1, w2, w3l]
    a1, a2 = _ptr_array(w1), _ptr_array(w2)
    a3 = None if w3l is None else _ptr_array(w3l)
    sp = [None, None, None]
    if scales is not None:
        sc = [[_c(np.asarray(s, np.float32)) for s in lst] if lst is not None else None
              for lst in scales]
        keep.append(sc)
        sp = [None if lst is None else _ptr_array(lst) for lst in sc]
    tok = None if tokens is None else _c(np.asarray(tokens, np.int32))
    n = T if tok is None else len(tok)
    y = np.empty((n, m), np.float64)
    ops = np.zeros((E, 4), np.int64) if count_ops else None
    _check(lib().moe_oracle_layer(_ptr(x), _dtype_code(x), T, m, p, E, k,
                                  ctypes.cast(a1, ctypes.c_void_p), ctypes.cast(a2, ctypes.c_void_p),
                                  None if a3 is None else ctypes.cast(a3, ctypes.c_void_p),
                                  _dtype_code(w1[0]),
                                  *(None if s is None else ctypes.cast(s, ctypes.c_void_p) for s in sp),
                                  kind, _ptr(ids), _ptr(weights), _ptr(tok), n, _ptr(y), _ptr(ops),
                                  nthreads), "layer")
    del keep
    return (y, ops) if count_ops else y


def cache_replay(n_index, n_way, layers, experts):
    """Replay (layer, expert) queries through an N-index x M-way LRU cache.

    Returns (hit [n] int32 0/1, slot [n] int32)."""
    layers = _c(np.asarray(layers, np.int32))
    experts = _c(np.asarray(experts, np.int32))
    n = len(layers)
    hit = np.empty(n, np.int32)
    slot = np.empty(n, np.int32)
    _check(lib().moe_oracle_cache_replay(n_index, n_way, n, _ptr(layers), _ptr(experts),
                                         _ptr(hit), _ptr(slot)), "cache_replay")
    return hit, slot


MISS, HIT, PREFETCH, PREFETCH_HIT = 0, 1, 2, 3


def cache_replay_calls(n_index, n_way, call_layers, counts, n_layers, n_prefetch):
    """Replay whole layer calls (layer id, per-expert token counts [E]) through
    the N-index x M-way LRU cache, prefetching up to n_prefetch of each call's
    experts for the next layer.

    Returns (layer, expert, kind, slot) int32 arrays, one entry per lookup or
    prefetch insert; kind is MISS, HIT, PREFETCH or PREFETCH_HIT."""
    call_layers = _c(np.asarray(call_layers, np.int32))
    counts = _c(np.asarray(counts, np.int32))
    n_calls = len(call_layers)
    E = counts.shape[1] if counts.ndim == 2 and n_calls else 1
    cap = max(1, int((counts > 0).sum()) + n_calls * max(n_prefetch, 0))
    out = [np.empty(cap, np.int32) for _ in range(4)]
    n = ctypes.c_int(0)
    _check(lib().moe_oracle_cache_replay_calls(n_index, n_way, n_calls, _ptr(call_layers), E,
                                               _ptr(counts), n_layers, n_prefetch,
                                               *[_ptr(o) for o in out], cap, ctypes.byref(n)),
           "cache_replay_calls")
    return tuple(o[:n.value] for o in out)


def forward(x, w_router, w1, w2, w3, k, kind, bias=None, scales=None, tokens=None):
    """Route all T tokens and evaluate the chosen ones: the whole layer."""
    logits = router_logits(x, w_router, bias)
    ids, w = topk(logits, k)
    y = layer(x, w1, w2, w3, ids, w, kind, scales=scales, tokens=tokens)
    return y, ids, w, logits
