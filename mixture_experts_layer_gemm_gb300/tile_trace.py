"""Per-expert tile timeline of the batch regime's tensor-core kernels.

Builds the tile-trace library (``build(trace=True)``: the same sources with
per-tile globaltimer stamps compiled in), runs one route + forward call of a
Mixtral-shaped layer (m = 4096, p = 14336, E = 8, top-2, SwiGLU, bf16) with the
Zipf(1.2) router bias on seeded synthetic tokens -- the inputs of the bench's
batch step -- and prints, for the up projection and the down projection of each
batch size:

- the launch plan and the tokens routed to each expert;
- per expert: its tiles (count and token widths), the median time from a
  tile's first stage landing to its last stage issued, and the window from its
  first tile's start to its last tile's end, relative to the kernel's first CTA
  entry;
- per kernel: the span to the last tile's last stage, the spread of the CTAs'
  (CTA pairs') last stages, the median gap between a CTA's consecutive tiles,
  and how busy the CTAs were (time inside tiles over the span).

Usage: python -m mixture_experts_layer_gemm_gb300.tile_trace [--tokens 512,2048,8192]
The trace build is a separate library (``libmoe_layer_trace.so``); the
product's library and kernels are not changed by it.
"""
import argparse
import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

N_CTAS, N_TILES = 160, 128  # the trace buffers' shape (csrc/tile_trace.cuh)


def _read(L, name):
    t = np.zeros((2, N_CTAS, N_TILES, 2), np.uint64)
    t0 = np.zeros((2, N_CTAS), np.uint64)
    info = np.zeros((2, N_CTAS, N_TILES, 4), np.int32)
    f = getattr(L, name)
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    f.restype = ctypes.c_int
    st = f(t.ctypes.data, t0.ctypes.data, info.ctypes.data, 0)
    if st != 0:
        raise RuntimeError(f"{name}: CUDA error {st}")
    return t.astype(np.int64), t0.astype(np.int64), info


def _arm(L, name):
    f = getattr(L, name)
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    f.restype = ctypes.c_int
    st = f(None, None, None, 1)
    if st != 0:
        raise RuntimeError(f"{name}: CUDA error {st}")


def summarize(title, t, t0, info, ctas, counts):
    """One kernel's records: t [CTA][tile][2], t0 [CTA], info [CTA][tile][4]."""
    t, t0, info = t[ctas], t0[ctas], info[ctas]
    rec = t[:, :, 0] > 0
    if not rec.any():
        print(f"  {title}: no tiles recorded")
        return
    base = t0[t0 > 0].min()
    us = lambda v: v / 1e3
    print(f"  {title}: {int(rec.sum())} tiles on {int(rec.any(axis=1).sum())} CTAs"
          f"{' (pairs)' if 'pair' in title else ''}")
    for e in range(len(counts)):
        m = rec & (info[:, :, 0] == e)
        if not m.any():
            continue
        dur = (t[:, :, 1] - t[:, :, 0])[m]
        widths = sorted(set(int(w) for w in info[:, :, 2][m]))
        ntt = len(set(int(v) for v in info[:, :, 1][m]))
        print(f"    expert {e}: {counts[e]:5d} tokens, {int(m.sum()):4d} tiles ({ntt} token tile(s), widths "
              f"{widths}), tile {us(np.median(dur)):6.2f} us median, window "
              f"{us(t[:, :, 0][m].min() - base):7.1f} .. {us(t[:, :, 1][m].max() - base):7.1f} us")
    last = np.array([t[c, rec[c], 1].max() for c in range(len(t)) if rec[c].any()]) - base
    gaps, busy = [], []
    for c in range(len(t)):
        idx = np.nonzero(rec[c])[0]
        if not len(idx):
            continue
        d = t[c, idx, 1] - t[c, idx, 0]
        busy.append(d.sum() / max(t[c, idx, 1].max() - base, 1))
        gaps.extend((t[c, idx[1:], 0] - t[c, idx[:-1], 1]).tolist())
    print(f"    span to the last stage {us(last.max()):.1f} us; CTAs' last stages "
          f"{us(last.min()):.1f} .. {us(np.median(last)):.1f} (median) .. {us(last.max()):.1f} us; "
          f"gap between tiles {us(np.median(gaps)) if gaps else float('nan'):.2f} us median; "
          f"busy {np.median(busy):.2f} of the span (median CTA)")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--tokens", default="512,2048,8192")
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)

    from mixture_experts_layer_gemm_gb300 import build as lib_build
    lib_path = lib_build.build(trace=True)
    import mixture_experts_layer_gemm_gb300 as moe
    if moe._lib is not None and moe.LIB_PATH != lib_path:
        raise RuntimeError("the product library is already loaded in this process")
    moe.LIB_PATH = lib_path
    L = moe.lib()

    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch
    import workloads as wl

    dev = "cuda"
    shape = wl.MIXTRAL.with_zipf(1.2)
    base = wl.make_layer(wl.MIXTRAL, seed=args.seed, device=dev)
    layer = wl.Layer(shape, base.w_router, wl.zipf_bias(shape.E, 1.2), base.w1, base.w2, base.w3)
    for T in [int(v) for v in args.tokens.split(",")]:
        x = wl.make_tokens(shape, T, seed=args.seed + 1, device=dev)
        ml = moe.MoELayer(layer, T)
        y = torch.empty((T, shape.m), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            ml.route(x)
            ml.forward(x, y)
        torch.cuda.synchronize()
        for name in ("moe_tile_trace_tc2", "moe_tile_trace_tc"):
            _arm(L, name)
        ml.route(x)
        ml.forward(x, y)
        torch.cuda.synchronize()
        t2, t20, i2 = _read(L, "moe_tile_trace_tc2")
        t1, t10, i1 = _read(L, "moe_tile_trace_tc")
        counts = ml.counts.cpu().numpy()
        pl = ml.plan(T)
        print(f"== T = {T}: plan tile_up {pl.tile_up} (pairs {pl.pair_up}), tile_down {pl.tile_down}, "
              f"splits {pl.splits_up}/{pl.splits_down}; tokens per expert {counts.tolist()}")
        if pl.pair_up:
            summarize("up projection, CTA pairs", t2[0], t20[0], i2[0], np.arange(0, N_CTAS, 2), counts)
        else:
            summarize("up projection", t1[0], t10[0], i1[0], np.arange(N_CTAS), counts)
        summarize("down projection", t1[1], t10[1], i1[1], np.arange(N_CTAS), counts)
        ml.close()


if __name__ == "__main__":
    main()
