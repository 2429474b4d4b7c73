"""Helpers for the GPU parity tests: run the library through its C ABI on
seeded inputs and compare with the fp64 oracle on the same inputs."""
import numpy as np
import torch

import mixture_experts_layer_gemm_gb300 as moe
import oracle
import workloads as wl

TOL = {"f32": 1e-5, "bf16": 1e-2, "i8": 3e-2}


def to_device(a: np.ndarray, device="cuda"):
    """numpy fp32 / bf16 bit patterns -> torch tensor on the device."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_device(t) -> np.ndarray:
    """torch tensor -> numpy (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f64(a):
    if a.dtype == np.uint16:
        return wl.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def max_token_rel_l2(y, ref):
    """max over tokens of ||y_t - ref_t|| / ||ref_t||, and the global rel-L2."""
    y, ref = f64(y), np.asarray(ref, np.float64)
    num = np.linalg.norm(y - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max()), float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def logit_error_bound(abssum, m):
    """Bound on |fp32 logit - exact logit| for the fused router kernel.

    Every product is rounded once and then passes through at most n
    additions, each with relative error <= u = 2^-24, so |error| <=
    n u sum_c |x_c W_r[c,e]| to first order.  The kernel spreads the m
    products over 256 threads (a few in sequence per thread), adds the lane
    sums with a 5-level shuffle tree, the 8 warp sums in sequence and the
    bias: n <= m/256 + 16.  The bound uses the larger n = m/32 + 20, which
    covers any split of m over at least 32 sequential partial sums, and keeps
    a factor 2 as margin."""
    n = m / 32 + 20
    return 2.0 * n * 2.0 ** -24 * abssum


def near_tie_tokens(logits64, abssum, m, k):
    """Tokens whose top-(k+1) oracle logits contain an adjacent gap smaller
    than twice the logit error bound: their fp32 selection or slot order may
    legitimately differ from the exact one."""
    srt = -np.sort(-logits64, axis=1)[:, :k + 1]
    gaps = np.abs(np.diff(srt, axis=1)).min(axis=1) if srt.shape[1] > 1 else np.full(len(srt), np.inf)
    delta = 2.0 * logit_error_bound(abssum, m).max(axis=1)
    return np.nonzero(gaps < delta)[0]


def oracle_quantized(layer):
    """The oracle's own int8 codes and scales of every expert matrix."""
    q = {"w1": [], "w2": [], "w3": [] if layer.w3 is not None else None,
         "s1": [], "s2": [], "s3": [] if layer.w3 is not None else None}
    for e in range(layer.shape.E):
        c, s = oracle.quantize_cols(layer.w1[e]); q["w1"].append(c); q["s1"].append(s)
        c, s = oracle.quantize_cols(layer.w2[e]); q["w2"].append(c); q["s2"].append(s)
        if layer.w3 is not None:
            c, s = oracle.quantize_cols(layer.w3[e]); q["w3"].append(c); q["s3"].append(s)
    return q


class Run:
    """Route + forward one batch through the library; keep every table."""

    def __init__(self, ml: "moe.MoELayer", x_np, routing="route", ids=None, w=None, logits=None,
                 forward=True):
        s = ml.shape
        self.T = x_np.shape[0]
        self.x = to_device(x_np)
        if routing == "route":
            ml.route(self.x)
        elif routing == "logits":
            ml.route_from_logits(to_device(logits.astype(np.float32)), T=self.T)
        else:
            ml.route_from_topk(to_device(ids.astype(np.int32).reshape(-1)),
                               to_device(w.astype(np.float32).reshape(-1)), T=self.T)
        ydt = torch.float32 if s.act == "f32" else torch.bfloat16
        self.y = torch.empty((self.T, s.m), dtype=ydt, device="cuda")
        if forward:
            ml.forward(self.x, self.y)
        torch.cuda.synchronize()
        n = self.T * s.k
        self.ids = from_device(ml.topk_ids[:n]).reshape(self.T, s.k)
        self.w = from_device(ml.topk_w[:n]).reshape(self.T, s.k)
        self.counts = from_device(ml.counts)
        self.offsets = from_device(ml.offsets)
        self.gather = from_device(ml.gather_index[:n])
        self.scatter = from_device(ml.scatter_index[:n])
        self.logits = (from_device(ml.logits[:self.T * s.E]).reshape(self.T, s.E)
                       if ml.logits is not None else None)
        self.y_np = from_device(self.y) if forward else None
