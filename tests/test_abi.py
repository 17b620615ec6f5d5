"""C-ABI checks that need no GPU: the library loads, exports every entry point the
header declares, and its host-side logic (config validation, capacity, buffer
and workspace sizing, argument checks that run before any CUDA call) behaves."""
import os
import re

import pytest
import torch

from mixture_experts_sparse_gemm_b300 import binding as B
from mixture_experts_sparse_gemm_b300 import build as build_mod
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    build_mod.build()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"^(?:moe_status|const char \*)\s*(moe_\w+)\(", text, flags=re.M)))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert len(names) >= 12
    assert set(names) == set(B.EXPORTS)
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    for code, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARG"), (2, "MOE_ERR_UNSUPPORTED"),
                       (3, "MOE_ERR_MISALIGNED"), (4, "MOE_ERR_WORKSPACE"), (5, "MOE_ERR_CUDA"),
                       (6, "MOE_ERR_TIMEOUT")]:
        assert B.status_string(code) == name
    assert B.status_string(99) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workload_configs_are_valid(name):
    cfg = B.config_from_workload(WORKLOADS[name])
    assert B.moe_validate_config(cfg) == B.MOE_OK
    assert B.moe_workspace_size(cfg) > 0
    assert B.moe_packed_weights_size(cfg) > 0


def test_fp8up_sizes():
    # the up projection's weights are one byte each, W2 stays bf16; scales for W1 | W3 only
    cfg = B.config(T=64, d=256, E=4, f=128, k=1, dtype="fp8up")
    ref = B.config(T=64, d=256, E=4, f=128, k=1, dtype="bf16")
    kib = lambda n: (n + 1023) // 1024 * 1024   # noqa: E731
    assert B.moe_packed_weights_size(cfg) == kib(4 * 2 * 128 * 256) + kib(4 * 256 * 128 * 2) + kib(4 * 4 * 2 * 128)
    assert B.moe_packed_weights_size(ref) == kib(4 * 2 * 128 * 256 * 2) + kib(4 * 256 * 128 * 2)
    # the FFN stage holds E4M3 codes and scales of its rows and of the tokens
    assert B.moe_workspace_size(cfg, B.MOE_STAGE_GROUPED_FFN) > B.moe_workspace_size(ref, B.MOE_STAGE_GROUPED_FFN)


@pytest.mark.parametrize("kw,want", [
    (dict(k=9, E=16), B.MOE_ERR_UNSUPPORTED),
    (dict(k=3, E=2), B.MOE_ERR_INVALID_ARG),
    (dict(k=0), B.MOE_ERR_INVALID_ARG),
    (dict(E=300, k=2), B.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(d=100), B.MOE_ERR_UNSUPPORTED),
    (dict(f=100), B.MOE_ERR_UNSUPPORTED),
    (dict(capacity_factor=float("nan")), B.MOE_ERR_INVALID_ARG),
    (dict(mode="ec", ec_capacity=0), B.MOE_ERR_INVALID_ARG),
    (dict(mode="ec", ec_capacity=65), B.MOE_ERR_INVALID_ARG),
    (dict(mode="ec", ec_capacity=8, gate="sigmoid"), B.MOE_ERR_UNSUPPORTED),
    (dict(n_shared=1, f_shared=0), B.MOE_ERR_INVALID_ARG),
    (dict(n_shared=1, f_shared=96), B.MOE_ERR_UNSUPPORTED),
    # FP8 expert weights: 256-wide tiles in both GEMMs
    (dict(dtype="fp8w", d=384), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype="fp8w", f=64), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype="fp8w", n_shared=1, f_shared=64), B.MOE_ERR_UNSUPPORTED),
    # FP8 up projection: the same tile widths (one fused launch)
    (dict(dtype="fp8up", d=384), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype="fp8up", f=64), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype="fp8up", n_shared=1, f_shared=64), B.MOE_ERR_UNSUPPORTED),
    (dict(dtype="fp8up", d=256, f=128, n_shared=1, f_shared=128), B.MOE_OK),
    (dict(dtype="f32", d=96), B.MOE_ERR_UNSUPPORTED),
    # accepted: the smallest shapes of each mode, an empty batch, the affinity drop
    (dict(dtype="fp8w", d=256, f=128, n_shared=1, f_shared=128), B.MOE_OK),
    (dict(dtype="f32", d=64, f=64), B.MOE_OK),
    (dict(d=128, f=64), B.MOE_OK),
    (dict(T=0), B.MOE_OK),
    (dict(capacity_factor=1.0, drop_policy="affinity"), B.MOE_OK),
])
def test_config_rejections(kw, want):
    base = dict(T=64, d=256, E=8, f=128, k=2)
    base.update(kw)
    cfg = B.config(**base)
    assert B.moe_validate_config(cfg) == want


def test_capacity_follows_printed_examples():
    with open(os.path.join(GOLDEN, "capacity.txt"), encoding="utf-8") as fh:
        rows = [ln.split('"')[0].split() for ln in fh if ln.strip() and not ln.startswith("#")]
    for C, T, k, E, want in rows:
        cfg = B.config(T=int(T), d=128, E=int(E), f=64, k=int(k), capacity_factor=float(C))
        assert B.moe_expert_capacity(cfg) == int(want)
    assert B.moe_expert_capacity(B.config(T=100, d=128, E=8, f=64, k=2)) == -1
    assert B.moe_expert_capacity(B.config(T=100, d=128, E=8, f=64, mode="ec", ec_capacity=17)) == 17


def test_buffer_rows():
    assert B.moe_buffer_rows(B.config(T=100, d=128, E=8, f=64, k=2)) == (200, 200)
    assert B.moe_buffer_rows(B.config(T=100, d=128, E=8, f=64, k=2, n_shared=1, f_shared=64)) == (200, 300)
    assert B.moe_buffer_rows(B.config(T=100, d=128, E=8, f=64, mode="ec", ec_capacity=25)) == (200, 200)


def test_argument_checks_run_before_any_cuda_call():
    cfg = B.config(T=64, d=256, E=8, f=128, k=2)
    L = B.lib()
    import ctypes
    c = ctypes.byref(cfg)
    A = 0x10000          # aligned fake device addresses: never dereferenced, the checks fail first
    ws_need = B.moe_workspace_size(cfg, B.MOE_STAGE_DISPATCH)
    assert L.moe_route(c, None, A, None, None, A, A, None, A, 1 << 20, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_route(c, A + 8, A, None, None, A, A, None, A, 1 << 20, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_route(c, A, A, None, None, A + 2, A, None, A, 1 << 20, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_dispatch(c, A, None, A, A, A, A, A, A, ws_need - 1, None) == B.MOE_ERR_WORKSPACE
    assert L.moe_dispatch(c, A, None, A, A, A, A, A, A + 64, ws_need, None) == B.MOE_ERR_MISALIGNED
    aff = B.config(T=64, d=256, E=8, f=128, k=2, capacity_factor=1.0, drop_policy="affinity")
    ws_aff = B.moe_workspace_size(aff, B.MOE_STAGE_DISPATCH)
    assert ws_aff > ws_need                                   # dense weights and kept lists
    assert L.moe_dispatch(ctypes.byref(aff), A, None, A, A, A, A, A, A, ws_aff, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(ctypes.byref(aff), A, A + 2, A, A, A, A, A, A, ws_aff, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_dispatch_noalloc(ctypes.byref(aff), A, A, A, A, A, A, None) == B.MOE_ERR_UNSUPPORTED
    bad = B.config(T=64, d=256, E=8, f=128, k=2)
    bad.drop_policy = 7
    assert B.lib().moe_validate_config(ctypes.byref(bad)) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(c, A, A, None, A, None, 0, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward(c, A, A, None, None, A + 128, A, A, 1 << 40, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_forward(None, A, A, None, None, A, A, A, 1 << 40, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_grouped_ffn(c, A, A, A, None, A, A, 0, None) == B.MOE_ERR_WORKSPACE
    ec = B.config(T=64, d=256, E=8, f=128, mode="ec", ec_capacity=8)
    assert L.moe_route(ctypes.byref(ec), A, A, None, A, A, A, None, A, 1 << 30, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_pack_weights(c, A, A, A, None, None, None, A, 10, None) == B.MOE_ERR_WORKSPACE
    assert L.moe_route(c, A, A, None, None, A, A, A + 2, A, 1 << 20, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_load_stats(c, A, A, None, A, A, A, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_load_stats(c, A, A, A, A, A, A + 4, None) == B.MOE_ERR_MISALIGNED
    assert L.moe_load_stats(None, A, A, A, A, A, A, None) == B.MOE_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gpu_reports_cuda_error():
    cfg = B.config(T=64, d=256, E=8, f=128, k=2)
    import ctypes
    A = 0x10000
    st = B.lib().moe_combine(ctypes.byref(cfg), A, A, A, A, None, 0, None)
    assert st == B.MOE_ERR_CUDA


# Kernels each call launches (moe_launch_count; bench.py's gpu_launches is K times the
# forward count), per stage: route, dispatch, grouped FFN, combine, forward.
#   route:    tensor-core router GEMM (W_r read in place) = 1, also with fewer than 74
#             token tiles and a long d (split-K in clusters, reduced and selected in
#             the same launch); Expert Choice adds the column select; E not a
#             multiple of 8 adds the W_r transpose; fp32: 1
#   dispatch: plan (one cluster) + gather = 2 (at most 32768 assignments), else count,
#             scan, rank + gather = 4; Expert Choice: slots + gather = 2
#   FFN:      one fused tensor-core launch; fp32: up + down = 2
#   forward:  the stages, without the combine when it is folded into the down
#             epilogue (one expert per token, no shared experts)
LAUNCHES = {
    "tiny_top2_fp32": [1, 2, 2, 1, 6],
    "switch_top1_cap1.25": [1, 2, 1, 1, 4],
    "mixtral_T16": [1, 2, 1, 1, 5],
    "mixtral_T4096": [1, 2, 1, 1, 5],
    "mixtral_T16384": [1, 2, 1, 1, 5],
    "deepseek_v3": [1, 2, 1, 1, 5],
    "expert_choice_zipf": [2, 2, 1, 1, 6],
}
LAUNCH_EXTRA = {
    # FP8 up projection: the forward quantises x once; the FFN stage quantises its
    # rows (and the shared experts' input) before the fused launch
    "fp8up_switch": (WORKLOADS["switch_top1_cap1.25"].with_(dtype="fp8up", name="fp8up_sw"), [1, 2, 2, 1, 5]),
    "fp8up_deepseek": (WORKLOADS["deepseek_v3"].with_(dtype="fp8up", name="fp8up_ds"), [1, 2, 3, 1, 6]),
    "transposed_router": (WORKLOADS["mixtral_T256"].with_(T=500, d=256, E=12, f=128, name="e12"), [2, 2, 1, 1, 6]),
    "multi_cta_dispatch": (WORKLOADS["mixtral_T256"].with_(T=20000, d=256, E=16, f=128, name="n40000"),
                           [1, 4, 1, 1, 7]),
}


@pytest.mark.parametrize("name", list(LAUNCHES) + list(LAUNCH_EXTRA))
def test_launch_counts(name):
    wl, want = (WORKLOADS[name], LAUNCHES[name]) if name in LAUNCHES else LAUNCH_EXTRA[name]
    cfg = B.config_from_workload(wl)
    got = [B.moe_launch_count(cfg, s) for s in (B.MOE_STAGE_ROUTE, B.MOE_STAGE_DISPATCH, B.MOE_STAGE_GROUPED_FFN,
                                                 B.MOE_STAGE_COMBINE, B.MOE_STAGE_FORWARD)]
    assert got == want
    empty = B.config_from_workload(wl, T=0)
    assert B.moe_launch_count(empty, B.MOE_STAGE_FORWARD) == 0


def test_wait_limit_setting_is_host_only_and_checked():
    build_mod.build()
    L = B.lib()
    default = B.moe_get_wait_limit_ns()
    assert default == 2_000_000_000
    try:
        B.moe_set_wait_limit_ns(1_000_000)
        assert B.moe_get_wait_limit_ns() == 1_000_000
        for bad in (1, 999, 60_000_000_001):
            assert L.moe_set_wait_limit_ns(bad) == B.MOE_ERR_INVALID_ARG
        assert B.moe_get_wait_limit_ns() == 1_000_000   # a rejected value changes nothing
        B.moe_set_wait_limit_ns(0)                      # 0 restores the default
        assert B.moe_get_wait_limit_ns() == default
    finally:
        B.moe_set_wait_limit_ns(0)
    assert L.moe_get_wait_limit_ns(None) == B.MOE_ERR_INVALID_ARG


def test_tile_group_setting_is_host_only_and_checked():
    build_mod.build()
    L = B.lib()
    assert B.moe_get_tile_group_bytes() == (40 << 20, 64 << 20)
    try:
        B.moe_set_tile_group_bytes(3 * 128 * 256 * 2, 1)
        assert B.moe_get_tile_group_bytes() == (3 * 128 * 256 * 2, 1)
        assert L.moe_set_tile_group_bytes((1 << 40) + 1, 0) == B.MOE_ERR_INVALID_ARG
        assert L.moe_set_tile_group_bytes(0, (1 << 40) + 1) == B.MOE_ERR_INVALID_ARG
        assert B.moe_get_tile_group_bytes() == (3 * 128 * 256 * 2, 1)   # a rejected pair changes nothing
        B.moe_set_tile_group_bytes(0, 1 << 40)                           # 0 restores a default
        assert B.moe_get_tile_group_bytes() == (40 << 20, 1 << 40)
    finally:
        B.moe_set_tile_group_bytes(0, 0)
    assert B.moe_get_tile_group_bytes() == (40 << 20, 64 << 20)
    assert L.moe_get_tile_group_bytes(None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_wait_probe(None, 1, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_wait_probe(0x10002, 1, None) == B.MOE_ERR_MISALIGNED
