"""The tile-trace tool's summary, on synthetic records (no GPU).

The tool reads per-tile stamps from the trace build of the library and
prints, per expert, the tiles' count, widths, median duration and window.
These tests feed it hand-made records whose answers are known."""
import io
import os
import shutil
from contextlib import redirect_stdout

import numpy as np
import pytest

from mixture_experts_layer_gemm_gb300 import build as lib_build
from mixture_experts_layer_gemm_gb300 import tile_trace as tt


def records():
    """Two CTAs; CTA 0 runs expert 0's two tiles, CTA 1 one tile of each
    expert.  Times in ns from an entry at 1000."""
    n_ctas, n_tiles = 2, 4
    t = np.zeros((n_ctas, n_tiles, 2), np.int64)
    t0 = np.array([1000, 1500], np.int64)
    info = np.zeros((n_ctas, n_tiles, 4), np.int32)
    # (cta, tile): first landed, last issued, expert, token tile, width
    rows = [(0, 0, 2000, 12000, 0, 0, 256), (0, 1, 13000, 23000, 0, 1, 160),
            (1, 0, 3000, 9000, 0, 2, 64), (1, 1, 10000, 30000, 1, 0, 32)]
    for c, i, a, b, e, tok, n in rows:
        t[c, i] = (a, b)
        info[c, i, :3] = (e, tok, n)
    return t, t0, info


def test_per_expert_lines():
    t, t0, info = records()
    out = io.StringIO()
    with redirect_stdout(out):
        tt.summarize("down projection", t, t0, info, np.arange(2), np.array([500, 20]))
    text = out.getvalue()
    assert "4 tiles on 2 CTAs" in text
    # expert 0: three tiles (durations 10, 10, 6 us: median 10), widths 64/160/256,
    # three token tiles, window from 2000 - 1000 to 23000 - 1000 ns
    assert "expert 0:   500 tokens,    3 tiles (3 token tile(s), widths [64, 160, 256])" in text
    assert "tile  10.00 us median, window     1.0 ..    22.0 us" in text
    assert "expert 1:    20 tokens,    1 tiles (1 token tile(s), widths [32]), tile  20.00 us" in text
    # the span ends at the last stage (30000 - 1000); CTA 0 ends at 22 us
    assert "span to the last stage 29.0 us" in text
    assert "CTAs' last stages 22.0 .. 25.5 (median) .. 29.0 us" in text
    # gaps 13000 - 12000 and 10000 - 9000: 1 us
    assert "gap between tiles 1.00 us median" in text


def test_no_records():
    t, t0, info = records()
    out = io.StringIO()
    with redirect_stdout(out):
        tt.summarize("up projection", np.zeros_like(t), t0, info, np.arange(2), np.array([1, 1]))
    assert "no tiles recorded" in out.getvalue()


def test_trace_build_compiles_the_instrumented_kernels():
    """The two instrumented kernel files compile with MOE_TILE_TRACE (nvcc
    cross-compiles here; objects go to the trace build's own folder)."""
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not available")
    os.makedirs(lib_build.BUILD_TRACE, exist_ok=True)
    for name in ("expert_tc.cu", "expert_tc2.cu"):
        obj, _ = lib_build._compile(os.path.join(lib_build.CSRC, name), ["-DMOE_TILE_TRACE"], False,
                                    lib_build.BUILD_TRACE)
        assert os.path.getsize(obj) > 0
