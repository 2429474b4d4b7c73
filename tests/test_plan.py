"""The forward pass's launch plan (moe_plan_forward), checked on the host.

moe_forward takes its plan from the same function, so these tests pin the
host logic that picks the regime and cuts the work -- without a GPU.  They
check properties the plan must have, not a retyping of its formulas: the
regime switches where the mean number of tokens per expert crosses the
measured crossovers, token passes and tiles grow with the batch and cover
the average expert, the split reductions fit the workspace and the shared
memory, and the kernels fill the SMs in near-whole waves whenever some split
count allows it.  A GPU test checks that the kernels a forward call launches
are the ones its plan names."""
import math

import pytest

import mixture_experts_layer_gemm_gb300 as moe

SMS = 152
BF16, I8 = moe.MOE_BF16, moe.MOE_I8
SWIGLU, RELU = moe.MOE_EXPERT_SWIGLU, moe.MOE_EXPERT_RELU2


def cfg(m=4096, p=14336, E=8, k=2, max_tokens=8192, act=BF16, weight=BF16, expert=SWIGLU, paged=0):
    return moe.moe_config_t(m, p, E, k, max_tokens, act, weight, expert, 0, paged)


MIXTRAL = cfg()
MIXTRAL_I8 = cfg(weight=I8)
PHI = cfg(p=6400, E=16)


def plan(c, T, **kw):
    return moe.moe_plan_forward(c, T, kw.pop("num_sms", SMS), **kw)


def expected_distinct_experts(T, k, E):
    """Mean number of distinct experts that T tokens, each choosing k of E
    uniformly, touch: E (1 - (1 - k/E)^T)."""
    return E * (1.0 - (1.0 - k / E) ** T)


@pytest.mark.parametrize("c, last_gemv", [(MIXTRAL, 16), (MIXTRAL_I8, 48), (PHI, 32)])
def test_regime_switches_at_the_mean_tokens_per_expert(c, last_gemv):
    """Weight-streaming GEMV up to 4 tokens per expert on average (12 with
    int8 weights), tensor cores from the next batch size on, for every T."""
    threshold = 12 if c.weight_dtype == I8 else 4
    for T in range(1, 400):
        p = plan(c, T)
        assert p.mean_tokens == math.ceil(T * c.k / c.E)
        want = moe.MOE_PATH_GEMV if p.mean_tokens <= threshold else moe.MOE_PATH_TENSOR
        assert p.path == want, T
    assert plan(c, last_gemv).path == moe.MOE_PATH_GEMV
    assert plan(c, last_gemv + 1).path == moe.MOE_PATH_TENSOR


def test_gemv_passes_grow_with_the_batch_and_cover_the_average_expert():
    for c in (MIXTRAL, MIXTRAL_I8, PHI):
        prev = 0
        for T in range(1, 257):
            p = plan(c, T, regime=moe.REGIME_DECODE)
            assert p.path == moe.MOE_PATH_GEMV
            assert p.tile_up == p.tile_down and p.tile_up in (8, 16, 24, 32)
            assert p.tile_up >= prev, T
            prev = p.tile_up
            mean = T * c.k / c.E
            # one pass holds the average expert while it fits in the largest
            if mean <= 32:
                assert p.tile_up >= mean, T
        assert plan(c, 1, regime=moe.REGIME_DECODE).tile_up == 8


def test_gemv_splits_fit_the_workspace_and_fill_the_sms():
    """A split count is allowed when the partial-sum buffers hold it (4 up,
    16 down), every split has a reduction block, and a pass's staged token
    rows (K / splits bf16 values per token) fit 64 KB of shared memory.  The
    plan takes the smallest allowed count whose 128-row units fill the SMs in
    waves at least 92% full, or, if none does, one with the fullest waves."""
    for c in (MIXTRAL, MIXTRAL_I8, PHI):
        bk = 128 if c.weight_dtype == I8 else 64
        for T in (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 128, 256):
            p = plan(c, T, regime=moe.REGIME_DECODE)
            n_act = max(c.k, min(c.E, int(expected_distinct_experts(T, c.k, c.E) + 0.5)))
            for K, rows, S, cap in ((c.m, 2 * c.p, p.splits_up, 4), (c.p, c.m, p.splits_down, 16)):

                def allowed(s):
                    return 1 <= s <= min(cap, K // bk) and p.tile_up * 2 * K <= 64 * 1024 * s

                def fill(s):
                    units = n_act * s * math.ceil(rows / 128)
                    return units / (math.ceil(units / SMS) * SMS)

                assert allowed(S), (T, K, S)
                full = [s for s in range(1, cap + 1) if allowed(s) and fill(s) >= 0.92]
                if full:
                    assert S == full[0], (T, K, S, full)
                else:
                    assert fill(S) == max(fill(s) for s in range(1, cap + 1) if allowed(s))


def test_tensor_core_tiles_cover_the_average_expert():
    for c in (MIXTRAL, MIXTRAL_I8, PHI):
        prev = 0
        for T in (20, 32, 48, 64, 96, 128, 192, 256, 384, 512, 1024, 2048, 4096, 8192):
            p = plan(c, T, regime=moe.REGIME_BATCH)
            assert p.path == moe.MOE_PATH_TENSOR
            allowed = (16, 32, 64, 128, 192) if c.weight_dtype == I8 else (16, 32, 64, 128, 256)
            assert p.tile_up in allowed and p.tile_up >= prev
            prev = p.tile_up
            if p.mean_tokens <= 128:
                assert p.tile_up >= p.mean_tokens, T
            if c.weight_dtype == I8:
                assert p.tile_down == p.tile_up
            else:
                # down tiles of 128 while experts average at most 192 tokens
                assert p.tile_down == (128 if p.tile_up == 256 and p.mean_tokens <= 192 else p.tile_up)


def test_cta_pairs_only_for_resident_bf16_256_token_tiles():
    p = plan(MIXTRAL, 8192)
    assert p.tile_up == 256 and p.pair_up == 1 and p.splits_up == 1
    assert plan(MIXTRAL, 8192, pair_tiles=0).pair_up == 0
    assert plan(cfg(paged=1), 8192).pair_up == 0
    assert plan(MIXTRAL_I8, 8192).pair_up == 0
    assert plan(MIXTRAL, 64).pair_up == 0  # 32-token tiles
    # ReLU form: p = 14336 stored rows is a multiple of 256 too
    assert plan(cfg(expert=RELU), 8192).pair_up == 1
    assert plan(cfg(p=14336 + 128, expert=RELU), 8192).pair_up == 0


def test_tensor_core_splits_follow_the_workspace():
    """At decode sizes (T k <= 512) the tensor-core kernels split their
    reductions within the partial-sum buffers (4 up, 16 down), like the GEMV.
    Beyond, the up projection never splits and the down projection splits at
    most in two, and only while the fp32 partial rows (max(max_tokens k,
    16 x 512) of them) hold two copies of its output."""
    for T in (20, 64, 128, 256):
        p = plan(MIXTRAL, T)
        assert p.path == moe.MOE_PATH_TENSOR
        assert 1 <= p.splits_up <= 4 and 1 <= p.splits_down <= 16
    for T in (257, 512, 1024, 2048, 4096, 8192):
        p = plan(MIXTRAL, T)
        assert p.splits_up == 1 and p.splits_down in (1, 2)
    # max_tokens = 8192: 16384 partial rows; T = 8192 needs 2 x 16384
    assert plan(MIXTRAL, 8192).splits_down == 1
    roomy = cfg(max_tokens=16384)
    assert plan(roomy, 8192).splits_up == 1


def test_edge_cases_and_forced_regimes():
    assert plan(MIXTRAL, 0).path == moe.MOE_PATH_NONE
    f32 = cfg(m=128, p=256, max_tokens=16, act=moe.MOE_F32, weight=moe.MOE_F32, expert=RELU)
    for T in (1, 16):
        p = plan(f32, T)
        assert p.path == moe.MOE_PATH_SIMT and p.splits_up == p.splits_down == 1
    # the GEMV takes T k <= 512 only
    assert plan(MIXTRAL, 256, regime=moe.REGIME_DECODE).path == moe.MOE_PATH_GEMV
    with pytest.raises(moe.MoeError) as e:
        plan(MIXTRAL, 257, regime=moe.REGIME_DECODE)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    # automatic: beyond T k = 512 the tensor cores, whatever the mean
    wide = cfg(E=64, k=2)
    assert plan(wide, 257).path == moe.MOE_PATH_TENSOR and plan(wide, 257).mean_tokens <= 12
    # the tensor-core path needs 128-row blocks; without them small batches stay on the GEMV
    odd = cfg(m=4096 + 64)
    assert plan(odd, 64).path == moe.MOE_PATH_GEMV
    with pytest.raises(moe.MoeError) as e:
        plan(odd, 64, regime=moe.REGIME_BATCH)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    # one SM: every split count gives whole waves, so the smallest allowed is taken
    p1 = plan(MIXTRAL, 16, num_sms=1)
    assert p1.splits_up == 1


def test_bad_arguments_are_rejected():
    L = moe.lib()
    import ctypes
    out = moe.moe_plan_t()
    assert L.moe_plan_forward(None, 1, SMS, 0, 1, ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_plan_forward(ctypes.byref(MIXTRAL), 1, SMS, 0, 1, None) == moe.MOE_ERR_INVALID_ARG
    for T, sms, regime, pair in ((-1, SMS, 0, 1), (8193, SMS, 0, 1), (1, 0, 0, 1), (1, SMS, 3, 1),
                                 (1, SMS, 0, 2)):
        st = L.moe_plan_forward(ctypes.byref(MIXTRAL), T, sms, regime, pair, ctypes.byref(out))
        assert st == moe.MOE_ERR_INVALID_ARG, (T, sms, regime, pair)
    bad = cfg(E=0)
    assert L.moe_plan_forward(ctypes.byref(bad), 1, SMS, 0, 1, ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG
