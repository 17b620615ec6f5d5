"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device
memory (a plugin whose host framework owns all device allocations, or a serving
loop where cudaMalloc could stall the device).  It must give exactly the outputs
of moe_dispatch, call after call, while its scratch lives in one array inside the
library that every call reuses.

This file is collected last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from mixture_experts_sparse_gemm_b300 import binding as B
from mixture_experts_sparse_gemm_b300 import build as build_mod
from workloads import random_assignment, random_rows


def test_noalloc_rejects_oversized_calls_before_any_cuda_call():
    build_mod.build()
    n_max = B.MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS
    cfg = B.config(T=n_max // 2 + 1, d=256, E=64, f=64, k=2)
    A = 0x10000
    st = B.lib().moe_dispatch_noalloc(ctypes.byref(cfg), A, A, A, A, A, A, None)
    assert st == B.MOE_ERR_UNSUPPORTED


def _dispatch_both(cfg, idx, x, dev):
    T, k, E, d = cfg.T, cfg.k, cfg.E, cfg.d
    outs = []
    for noalloc in (False, True):
        off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
        cnt = torch.full((E,), -7, dtype=torch.int32, device=dev)
        slot = torch.full((T, k), -7, dtype=torch.int32, device=dev)
        x_perm = torch.zeros(T * k, d, dtype=x.dtype, device=dev)
        if noalloc:
            B.moe_dispatch_noalloc(cfg, idx, x, off, cnt, slot, x_perm)
        else:
            ws = torch.empty(B.moe_workspace_size(cfg, B.MOE_STAGE_DISPATCH), dtype=torch.uint8, device=dev)
            B.moe_dispatch(cfg, idx, x, off, cnt, slot, x_perm, ws)
        torch.cuda.synchronize()
        B.moe_check_device_error()
        outs.append((off, cnt, slot, x_perm))
    return outs


@pytest.mark.gpu
def test_noalloc_dispatch_matches_moe_dispatch_twice(cuda_device):
    build_mod.build()
    # two calls in a row: the second finds the first call's contents in the shared
    # scratch array and must still match moe_dispatch exactly (integer outputs and
    # copied rows are bit-exact, the tolerance of every dispatch test)
    cases = [
        (B.config(T=8192, d=1024, E=64, f=64, k=1, capacity_factor=1.25), 1.0, 11),
        (B.config(T=4096, d=256, E=256, f=64, k=8), 0.5, 12),
        (B.config(T=4096, d=256, E=256, f=64, k=8), 0.0, 13),   # same shape again, other routing
        (B.config(T=777, d=128, E=8, f=64, k=2, capacity_factor=0.9), 1.5, 14),
        # more than 32768 assignments: the multi-CTA count / scan / rank kernels, which
        # keep per-chunk expert counts in the first part of the array.  8192 x 8 at
        # E = 256 is the documented maximum and fills all of it (256 chunks x 256
        # experts + 65536 row tokens = 131072 ints).
        (B.config(T=8192, d=256, E=256, f=64, k=8), 0.7, 15),
        (B.config(T=8192, d=256, E=256, f=64, k=8, capacity_factor=1.0), 1.2, 16),
        (B.config(T=65536, d=128, E=64, f=64, k=1, capacity_factor=1.25), 1.0, 17),
        (B.config(T=20000, d=128, E=128, f=64, k=2, capacity_factor=1.0), 0.8, 18),
        # back to a one-launch plan after the array was filled by the larger ones
        (B.config(T=777, d=128, E=8, f=64, k=2, capacity_factor=0.9), 1.5, 19),
    ]
    for cfg, skew, seed in cases:
        idx = random_assignment(cfg.T, cfg.E, cfg.k, seed=seed, skew=skew, device=cuda_device)
        x = random_rows(cfg.T, cfg.d, seed=seed, device=cuda_device)
        for call in range(2):   # each case twice in a row
            ref, got = _dispatch_both(cfg, idx, x, cuda_device)
            for r, g in zip(ref, got):
                assert torch.equal(r, g), (cfg.T, cfg.k, cfg.E, call)
            assert int(got[0][-1]) > 0


@pytest.mark.gpu
def test_noalloc_accepts_the_documented_maximum(cuda_device):
    build_mod.build()
    n_max = B.MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS
    cfg = B.config(T=n_max // 8, d=128, E=256, f=64, k=8)
    idx = random_assignment(cfg.T, cfg.E, cfg.k, seed=20, device=cuda_device)
    x = random_rows(cfg.T, cfg.d, seed=20, device=cuda_device)
    off = torch.empty(cfg.E + 1, dtype=torch.int32, device=cuda_device)
    cnt = torch.empty(cfg.E, dtype=torch.int32, device=cuda_device)
    slot = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=cuda_device)
    x_perm = torch.empty(cfg.T * cfg.k, cfg.d, dtype=x.dtype, device=cuda_device)
    B.moe_dispatch_noalloc(cfg, idx, x, off, cnt, slot, x_perm)   # raises unless MOE_OK
    torch.cuda.synchronize()
    B.moe_check_device_error()
    assert int(off[-1]) == n_max
