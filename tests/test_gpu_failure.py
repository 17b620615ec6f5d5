"""Failure detection on the GPU, in the forms that leave the device usable.

* Out-of-range expert ids reaching the dispatch are skipped, treated as dropped
  and flagged: moe_check_device_error reports MOE_ERR_INVALID_ARG once, and every
  other output equals the oracle's dispatch of the valid assignments.
* A bounded device-side wait that is never satisfied gives up after the wait
  limit (moe_set_wait_limit_ns) and is reported as MOE_ERR_TIMEOUT; the probe
  runs the same two wait routines the tensor-core kernels use (an mbarrier
  phase and a counter in global memory), on a flag nothing sets.  Afterwards the
  context still runs the layer bit for bit as before.
No test traps, faults or hangs a GPU: every wait here ends by its limit.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_gemm_b300 import binding as B
from mixture_experts_sparse_gemm_b300 import build as build_mod
from mixture_experts_sparse_gemm_b300.layer import MoELayer
from workloads import WORKLOADS, make_inputs, random_assignment, random_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built(cuda_device):
    build_mod.build()
    B.lib()
    torch.cuda.synchronize()
    B.moe_check_device_error()   # start from a clear error word
    yield
    B.moe_set_wait_limit_ns(0)


@pytest.mark.parametrize("T,E,k,C", [(1000, 16, 2, 1.0), (20000, 16, 2, 1.1), (333, 64, 1, 0.0)])
def test_dispatch_flags_and_drops_out_of_range_ids(T, E, k, C, cuda_device):
    d = 128
    idx = random_assignment(T, E, k, seed=T + 3, skew=1.0)
    g = np.random.default_rng(T)
    bad = g.choice(T * k, size=max(3, T * k // 50), replace=False)
    flat = idx.view(-1)
    flat[bad[0::2]] = E          # one past the last expert
    flat[bad[1::2]] = -1
    cfg = B.config(T=T, d=d, E=E, f=64, k=k, capacity_factor=C)
    x = random_rows(T, d, seed=T + 4, device=cuda_device)
    ws = torch.empty(B.moe_workspace_size(cfg, B.MOE_STAGE_DISPATCH), dtype=torch.uint8, device=cuda_device)
    off = torch.empty(E + 1, dtype=torch.int32, device=cuda_device)
    cnt = torch.empty(E, dtype=torch.int32, device=cuda_device)
    slot = torch.empty(T, k, dtype=torch.int32, device=cuda_device)
    x_perm = torch.empty(T * k, d, dtype=torch.bfloat16, device=cuda_device)
    B.moe_dispatch(cfg, idx.to(cuda_device), x, off, cnt, slot, x_perm, ws)
    torch.cuda.synchronize()
    with pytest.raises(B.MoeError) as ex:
        B.moe_check_device_error()
    assert ex.value.status == B.MOE_ERR_INVALID_ARG
    B.moe_check_device_error()   # read once, then cleared
    # expected: the valid assignments dispatched as usual; an invalid one is dropped.
    # The oracle sees the invalid ids as one extra expert E placed after the real
    # ones, which leaves the real experts' counts, offsets, slots and rows unchanged.
    cap = oracle.capacity(C, T, k, E)
    mod = idx.clone()
    mod[(mod < 0) | (mod >= E)] = E
    o_off, o_cnt, o_slot, o_rows = oracle.dispatch_tc(mod, E + 1, cap)
    invalid = (mod == E).numpy()
    o_slot = np.where(invalid, -1, o_slot)
    np.testing.assert_array_equal(off.cpu().numpy(), o_off[: E + 1])
    np.testing.assert_array_equal(cnt.cpu().numpy(), o_cnt[:E])
    np.testing.assert_array_equal(slot.cpu().numpy(), o_slot)
    A = int(o_off[E])
    assert torch.equal(x_perm[:A], x[torch.from_numpy(o_rows[:A]).long().to(cuda_device)])


def _small_forward(cuda_device):
    wl = WORKLOADS["mixtral_T256"].with_(T=300, d=256, f=256, name="failure_small")
    inp = make_inputs(wl, cuda_device)
    cfg = B.config_from_workload(wl)
    layer = MoELayer(cfg, inp["W1"], inp["W3"], inp["W2"])
    y = layer.forward(inp["x"], inp["W_r"], inp["logit_offset"], None)
    torch.cuda.synchronize()
    B.moe_check_device_error()
    return y


def test_bounded_wait_gives_up_and_the_context_stays_usable(cuda_device):
    y0 = _small_forward(cuda_device)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    B.moe_set_wait_limit_ns(1_000_000)   # 1 ms
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        B.moe_wait_probe(flag, 1)          # nothing ever sets the flag
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        with pytest.raises(B.MoeError) as ex:
            B.moe_check_device_error()
        assert ex.value.status == B.MOE_ERR_TIMEOUT
        assert elapsed < 1.0, elapsed     # two waits of ~1 ms, not the 2 s default
        # a satisfied condition: both waits succeed, nothing is recorded
        flag.fill_(1)
        B.moe_wait_probe(flag, 1)
        torch.cuda.synchronize()
        B.moe_check_device_error()
        # a short limit that the layer's real waits stay under: no false timeout
        B.moe_set_wait_limit_ns(200_000_000)
        y1 = _small_forward(cuda_device)
    finally:
        B.moe_set_wait_limit_ns(0)
    y2 = _small_forward(cuda_device)
    assert torch.equal(y0, y1) and torch.equal(y0, y2)
