"""The C-ABI library loads without a GPU, exports every entry point that
include/moe_layer.h declares, and rejects bad arguments before touching the
device.  Host-only arithmetic (the expert-cache geometry) is checked against
the expert-cache article's own numbers.  No compute call runs here."""
import ctypes
import json
import os
import re

import pytest

import mixture_experts_layer_gemm_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _declared_functions():
    src = open(moe.HEADER_PATH).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    declared = _declared_functions()
    assert len(declared) >= 15, declared
    L = moe.lib()
    missing = [n for n in declared if not hasattr(L, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    assert sorted(moe.exported_names()) == declared


def test_status_strings_and_version():
    assert moe.moe_status_string(moe.MOE_OK) == "ok"
    assert moe.moe_status_string(moe.MOE_ERR_TIMEOUT) == "timeout"
    assert moe.moe_version() >= 100


def test_create_rejects_bad_configs_before_touching_the_device():
    L = moe.lib()
    out = ctypes.c_void_p()
    assert L.moe_layer_create(None, None, None, None, None, None, None, 0,
                              ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG
    bad = [
        dict(E=0), dict(E=65), dict(k=0), dict(k=9), dict(m=0), dict(max_tokens=0),
    ]
    for change in bad:
        c = dict(m=128, p=256, E=8, k=2, max_tokens=16, act_dtype=moe.MOE_F32,
                 weight_dtype=moe.MOE_F32, expert=moe.MOE_EXPERT_RELU2, has_router_bias=0, paged=0)
        c.update(change)
        cfg = moe.moe_config_t(**c)
        st = L.moe_layer_create(ctypes.byref(cfg), None, None, None, None, None, None, 0,
                                ctypes.byref(out))
        assert st == moe.MOE_ERR_INVALID_ARG, change
    # valid shape but unsupported type combinations
    for act, wt in [(moe.MOE_F32, moe.MOE_BF16), (moe.MOE_BF16, moe.MOE_F32),
                    (moe.MOE_F32, moe.MOE_I8)]:
        cfg = moe.moe_config_t(128, 256, 8, 2, 16, act, wt, moe.MOE_EXPERT_RELU2, 0, 0)
        st = L.moe_layer_create(ctypes.byref(cfg), None, None, None, None, None, None, 0,
                                ctypes.byref(out))
        assert st == moe.MOE_ERR_UNSUPPORTED
    cfg = moe.moe_config_t(100, 256, 8, 2, 16, moe.MOE_BF16, moe.MOE_BF16, moe.MOE_EXPERT_RELU2, 0, 0)
    assert L.moe_layer_create(ctypes.byref(cfg), None, None, None, None, None, None, 0,
                              ctypes.byref(out)) == moe.MOE_ERR_UNSUPPORTED
    assert "64" in moe.moe_last_error()


def test_calls_on_null_layer_are_rejected():
    L = moe.lib()
    r = moe.moe_routing_t()
    assert L.moe_route(None, None, 1, ctypes.byref(r), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, None, ctypes.byref(r), None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_layer_set_option(None, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_destroy(None) == moe.MOE_OK


def test_pool_geometry_matches_expert_cache_article():
    """Expert-cache article, sections 2.2 and 5.1 (binary units)."""
    cases = json.load(open(os.path.join(GOLDEN, "expert_cache_geometry.json")))["cases"]
    MiB = 1 << 20
    for c in cases:
        n, slots = moe.moe_pool_geometry(int(c["available_mib"] * MiB), int(c["expert_mib"] * MiB),
                                         c["ways"])
        assert (n, slots) == (c["n_index"], c["usable_slots"]), c["note"]


def test_pool_geometry_for_the_mixtral_slot_budget():
    # a 16 GiB budget of 336 MiB bf16 Mixtral experts (3 x 4096 x 14336 x 2 bytes), 4-way
    expert = 3 * 4096 * 14336 * 2
    assert expert == 336 * (1 << 20)
    assert moe.moe_pool_geometry(16 << 30, expert, 4) == (12, 48)
    with pytest.raises(moe.MoeError):
        moe.moe_pool_geometry(expert * 3, expert, 4)  # not even one set
    assert moe.moe_pool_geometry(expert * 4, expert, 4) == (1, 4)    # exactly one set
    assert moe.moe_pool_geometry(expert * 11, expert, 4) == (2, 8)   # 3 slots that fill no set stay unused
    for expert_b, ways in ((0, 4), (expert, 0)):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_pool_geometry(16 << 30, expert_b, ways)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG


def test_selftest_rejects_bad_poll_counts_before_touching_the_device():
    for polls in (0, (1 << 24) + 1):
        st, flags = moe.moe_selftest_bounded_wait(polls)
        assert st == moe.MOE_ERR_INVALID_ARG and flags == 0


def test_public_error_flags_are_distinct_bits():
    bits = [moe.MOE_FLAG_EXPERT_ID, moe.MOE_FLAG_DUPLICATE_ID, moe.MOE_FLAG_GATHER_INDEX,
            moe.MOE_FLAG_OFFSETS, moe.MOE_FLAG_WAIT_TIMEOUT, moe.MOE_FLAG_TMEM_ALLOC]
    assert all(b & (b - 1) == 0 for b in bits) and len(set(bits)) == len(bits)


def test_phi_expert_size_in_binary_units():
    # the expert-cache article's Phi-3.5-MoE expert: 3 x 4096 x 6400 bf16 values
    expert = 3 * 4096 * 6400 * 2
    assert expert == 150 * (1 << 20) and round(expert / 1e6, 1) == 157.3


def test_transfer_threshold_is_where_loading_stops_dominating():
    """HARMOEny write-up, 3.2: an expert is worth fetching over the link when its
    compute outlasts its transfer, q > phi * dtype / (2 beta).  The crossover of
    the two times -- load 2 m p dtype / beta, compute 4 q m p / phi (two
    multiply-adds per weight and token) -- found by search must equal that
    closed form; with GB300-like numbers decode batches sit far below it."""
    m, p, dtype = 4096, 14336, 2
    phi, beta = 1944e12, 211e9
    load = 2 * m * p * dtype / beta
    q = 1
    while 4 * q * m * p / phi <= load:
        q += 1
    closed = phi * dtype / (2 * beta)
    assert q - 1 <= closed < q
    assert 16 < closed / 100  # decode (q <= 16 per expert) is link-bound by two orders of magnitude


def _header_text():
    return re.sub(r"/\*.*?\*/", " ", open(moe.HEADER_PATH).read(), flags=re.S)


def _int_expr(src):
    """Value of an integer constant of the header: a literal (decimal or hex,
    optional u suffix) or a left shift of two of them."""
    if "<<" in src:
        a, b = src.split("<<")
        return _int_expr(a) << _int_expr(b)
    return int(re.sub(r"[uUlL]+$", "", src.strip()), 0)


def _header_constants(text):
    values = {m.group(1): _int_expr(m.group(2))
              for m in re.finditer(r"\b(MOE_\w+)\s*=\s*([^,}]+)", text)}
    values.update({m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(MOE_\w+)\s+(\d+)", text)})
    return values


_C_SIZES = {"int": 4, "int32_t": 4, "uint32_t": 4, "uint64_t": 8, "size_t": 8, "double": 8, "float": 4,
            "moe_dtype_t": 4, "moe_expert_t": 4}


def _header_structs(text):
    """{name: [(member, element bytes, count)]} of every typedef struct { ... } name;"""
    defines = _header_constants(text)
    out = {}
    for m in re.finditer(r"typedef\s+struct\s*\{(.*?)\}\s*(\w+)\s*;", text, flags=re.S):
        members = []
        for decl in m.group(1).split(";"):
            decl = decl.strip()
            if not decl:
                continue
            ctype, rest = decl.split(None, 1)
            for name in rest.split(","):
                name = name.strip()
                size = 8 if name.startswith("*") else _C_SIZES[ctype]
                name = name.lstrip("*").strip()
                count = 1
                arr = re.match(r"(\w+)\s*\[(\w+)\]", name)
                if arr:
                    name = arr.group(1)
                    count = defines.get(arr.group(2)) or int(arr.group(2))
                members.append((name, size, count))
        out[m.group(2)] = members
    return out


def test_binding_structs_mirror_the_header():
    """Every struct the binding passes through the C ABI has the header's
    members, in order, with the same element sizes."""
    structs = _header_structs(_header_text())
    for name in ("moe_config_t", "moe_routing_t", "moe_layer_info_t", "moe_timings_t", "moe_stats_t",
                 "moe_plan_t"):
        py = getattr(moe, name)
        got = []
        for fname, ftype in py._fields_:
            count = getattr(ftype, "_length_", 1)
            elem = ftype._type_ if count > 1 else ftype
            got.append((fname, ctypes.sizeof(elem), count))
        assert got == structs[name], name


def test_binding_constants_match_the_header():
    values = _header_constants(_header_text())
    shared = [k for k in values if hasattr(moe, k)]
    assert len(shared) >= 20, shared
    for k in shared:
        assert getattr(moe, k) == values[k], k
