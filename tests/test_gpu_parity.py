"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars:
  * integer outputs (routing indices, offsets, slot table, drop mask, row
    gather) bit-exact; tokens whose oracle gap between the k-th and (k+1)-th key
    is below 1e-4 are reported and left out of the index comparison;
  * bf16 outputs: max |err| <= 2e-2 * max |y_ref|; fp32: <= 1e-4 * max |y_ref|;
  * gate weights (fp32 on the GPU, fp64 in the oracle): |err| <= 2e-5.
Stage tests feed both sides the same seeded integer/float inputs; end-to-end
tests compare the routing and the layer output (sampled tokens at full size).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_gemm_b300 import binding as B
from mixture_experts_sparse_gemm_b300 import build as build_mod
from mixture_experts_sparse_gemm_b300.layer import MoELayer
from workloads import WORKLOADS, make_inputs, random_assignment, random_rows, random_weights

pytestmark = pytest.mark.gpu

GAP = 1e-4
TOL = {"bf16": 2e-2, "f32": 1e-4}
NTH = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def built(cuda_device):
    build_mod.build()
    B.lib()


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype != torch.int32 else t.cpu().numpy()


def rel_err(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def _layer(wl, inp):
    cfg = B.config_from_workload(wl)
    return cfg, MoELayer(cfg, inp["W1"], inp["W3"], inp["W2"], inp.get("W1s"), inp.get("W3s"), inp.get("W2s"))


def _check_device_error():
    torch.cuda.synchronize()
    B.moe_check_device_error()


# ------------------------------------------------------------------------------------------ route

SMALL_TC = {
    "ragged_top2": WORKLOADS["mixtral_T256"].with_(T=333, d=256, f=128, name="ragged_top2"),
    "sigmoid_top8_e256": WORKLOADS["deepseek_v3"].with_(T=200, d=384, f=128, f_shared=128, name="sig8"),
    "top1_cap": WORKLOADS["switch_top1_cap1.25"].with_(T=1000, d=256, f=128, E=16, name="top1cap"),
    "t1": WORKLOADS["mixtral_T16"].with_(T=1, d=128, f=64, name="t1"),
    # few token tiles and a long d: the router splits K over CTAs and selects per warp
    "sigmoid_top8_splitk": WORKLOADS["deepseek_v3"].with_(T=200, d=2048, f=128, f_shared=128, name="sig8_split"),
    # 47 token tiles: clusters of 3 K splits, each CTA selecting 43 of its tile's rows
    "sigmoid_top8_split3": WORKLOADS["deepseek_v3"].with_(T=6000, d=1024, f=128, f_shared=128, name="sig8_split3"),
    # W_r read in place by the tensor-core router: two 64-expert chunks (E = 128), and
    # E = 24 (a multiple of 8, not of 64: the chunk past E is zero-filled); E = 12 is
    # not a multiple of 8 and takes the transposed copy of W_r
    "sigmoid_top4_e128": WORKLOADS["deepseek_v3"].with_(T=300, d=256, E=128, k=4, f=128, f_shared=128,
                                                         name="sig4_e128"),
    "top2_e24": WORKLOADS["mixtral_T256"].with_(T=500, d=256, E=24, f=128, name="top2_e24"),
    "top2_e12": WORKLOADS["mixtral_T256"].with_(T=500, d=256, E=12, f=128, name="top2_e12"),
}
ROUTE_CASES = ["tiny_top2_fp32", "switch_top1_cap1.25", "mixtral_T4096", "deepseek_v3"] + list(SMALL_TC)


def _wl(name):
    return WORKLOADS[name] if name in WORKLOADS else SMALL_TC[name]


@pytest.mark.parametrize("name", ROUTE_CASES)
def test_route_token_choice(name, cuda_device):
    wl = _wl(name)
    inp = make_inputs(wl, cuda_device, weights=False)
    cfg = B.config_from_workload(wl)
    ws = torch.empty(max(1, B.moe_workspace_size(cfg, B.MOE_STAGE_ROUTE)), dtype=torch.uint8, device=cuda_device)
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device=cuda_device)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=cuda_device)
    B.moe_route(cfg, inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"], idx, w, ws)
    _check_device_error()
    oi, ow, gap = oracle.route_tc(inp["x"], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                  wl.renorm, nthreads=NTH)
    keep = gap >= GAP
    gi, gw = _np(idx), _np(w)
    print(f"{name}: {int((~keep).sum())} of {wl.T} tokens within {GAP} of a tie, excluded")
    assert (~keep).mean() < 0.02
    np.testing.assert_array_equal(gi[keep], oi[keep])
    assert np.abs(gw[keep] - ow[keep]).max() <= 2e-5


@pytest.mark.parametrize("name", ["ragged_top2", "sigmoid_top8_splitk", "tiny_top2_fp32", "sigmoid_top8_e256"])
def test_route_nan_token_stays_in_range(name, cuda_device):
    """A token whose input row holds a NaN has NaN logits; its slots must still name
    distinct experts in range (the lowest ones), and the other tokens' routing is
    unaffected.  Covers the fused tensor-core epilogue, the split-K select and the
    CUDA-core router."""
    wl = _wl(name)
    inp = make_inputs(wl, cuda_device, weights=False)
    x = inp["x"].clone()
    x[0, 5] = float("nan")
    cfg = B.config_from_workload(wl)
    ws = torch.empty(max(1, B.moe_workspace_size(cfg, B.MOE_STAGE_ROUTE)), dtype=torch.uint8, device=cuda_device)
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device=cuda_device)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=cuda_device)
    B.moe_route(cfg, x, inp["W_r"], inp["logit_offset"], inp["sel_bias"], idx, w, ws)
    _check_device_error()
    gi = _np(idx)
    np.testing.assert_array_equal(gi[0], np.arange(wl.k))
    oi, _, gap = oracle.route_tc(inp["x"][1:], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                 wl.renorm, nthreads=NTH)
    keep = gap >= GAP
    np.testing.assert_array_equal(gi[1:][keep], oi[keep])


EC_CASES = {
    "expert_choice_zipf": WORKLOADS["expert_choice_zipf"],
    "ec_small": WORKLOADS["expert_choice_zipf"].with_(T=1000, d=256, E=16, f=128, ec_capacity=100, name="ec_small"),
    "ec_cap_eq_T": WORKLOADS["expert_choice_zipf"].with_(T=77, d=128, E=4, f=64, ec_capacity=77, name="ec_full"),
    # split-K router feeding the expert-major scores
    "ec_splitk": WORKLOADS["expert_choice_zipf"].with_(T=1000, d=2048, E=16, f=64, ec_capacity=100, name="ec_split"),
    # a column longer than the select kernel keeps in shared memory (49152 tokens)
    "ec_long_column": WORKLOADS["expert_choice_zipf"].with_(T=50000, d=128, E=4, f=64, ec_capacity=1000,
                                                            name="ec_long"),
}


def _check_ec_selection(gt, gw, ot, S, cap, tau=1e-5):
    """Exactly cap ascending tokens per expert; every token clearly above the
    oracle boundary taken, every token clearly below it not taken.

    tau bounds the GPU's error on a score: the logits are an fp32 tensor-core
    accumulation over d (about d/16 rounding steps of 2^-23 relative), which moves
    a softmax score of ~0.3 by up to ~2e-6; tau = 1e-5 leaves a 5x margin.
    Experts whose oracle boundary gap is below 2*tau are checked for validity
    only, and their boundary tokens are reported as ambiguous."""
    E = gt.shape[0]
    ambiguous = set()
    for e in range(E):
        assert (np.diff(gt[e]) > 0).all() and len(gt[e]) == cap
        col = S[:, e]
        srt = np.sort(col)[::-1]
        hi_b = srt[cap - 1]
        lo_b = srt[cap] if cap < len(col) else -np.inf
        taken = np.zeros(len(col), bool)
        taken[gt[e]] = True
        assert taken[col > hi_b + tau].all()
        assert not taken[col < lo_b - tau].any()
        if hi_b - lo_b >= 2 * tau:
            np.testing.assert_array_equal(gt[e], ot[e])
        else:
            ambiguous.update(np.nonzero(np.abs(col - hi_b) <= 2 * tau)[0].tolist())
        np.testing.assert_allclose(gw[e], col[gt[e]], atol=2e-5, rtol=0)
    return ambiguous


@pytest.mark.parametrize("name", list(EC_CASES))
def test_route_expert_choice(name, cuda_device):
    wl = EC_CASES[name]
    inp = make_inputs(wl, cuda_device, weights=False)
    cfg = B.config_from_workload(wl)
    ws = torch.empty(B.moe_workspace_size(cfg, B.MOE_STAGE_ROUTE), dtype=torch.uint8, device=cuda_device)
    tok = torch.empty(wl.E, wl.ec_capacity, dtype=torch.int32, device=cuda_device)
    w = torch.empty(wl.E, wl.ec_capacity, dtype=torch.float32, device=cuda_device)
    B.moe_route(cfg, inp["x"], inp["W_r"], inp["logit_offset"], None, tok, w, ws)
    _check_device_error()
    ot, ow, gap, S = oracle.route_ec(inp["x"], inp["W_r"], wl.ec_capacity, inp["logit_offset"], nthreads=NTH,
                                     want_scores=True)
    amb = _check_ec_selection(_np(tok), _np(w), ot, S, wl.ec_capacity)
    print(f"{name}: {len(amb)} tokens at a near-tie expert boundary")


# ------------------------------------------------------------------------------------------ dispatch

DISPATCH_CASES = [
    # T, E, k, capacity factor, skew, d, dtype
    (8192, 64, 1, 1.25, 1.0, 1024, "bf16"),
    (8192, 64, 1, 1.25, 0.0, 1024, "bf16"),
    (4096, 256, 8, 0.0, 0.5, 256, "bf16"),
    (1000, 8, 2, 1.0, 1.5, 128, "bf16"),
    (257, 16, 3, 0.3, 2.0, 256, "bf16"),
    (1, 4, 2, 0.0, 0.0, 128, "bf16"),
    (7, 8, 2, 0.0, 0.0, 1152, "bf16"),      # few rows: each split into spans, the last one ragged
    (300, 8, 2, 0.01, 0.0, 128, "bf16"),     # capacity 0: every assignment dropped
    (500, 8, 2, 1.25, 1.0, 64, "f32"),
    (6000, 32, 2, 1.25, 1.0, 128, "bf16"),   # 12000 assignments: the plan on a cluster of 8 CTAs
    (16384, 256, 2, 1.0, 0.3, 128, "bf16"),  # exactly 32768: the largest plan (8 CTAs, 4 per lane)
    (2049, 8, 1, 1.25, 1.0, 128, "bf16"),    # 2049: a plan of 2 CTAs, the second one nearly empty
    (4097, 64, 1, 1.25, 1.0, 128, "bf16"),   # 4097: 4 CTAs
    (2731, 16, 3, 0.8, 1.0, 128, "bf16"),    # 8193: 8 CTAs, drops
    (70, 8, 1, 0.5, 2.0, 128, "bf16"),       # fewer assignments than one warp's share, drops
    (16385, 8, 2, 1.0, 1.0, 128, "bf16"),    # 32770: just past it, the multi-kernel count/scan/rank path
    (40000, 16, 2, 1.1, 1.0, 128, "bf16"),   # 80000: multi-CTA
    (32768, 256, 2, 1.0, 0.3, 128, "bf16"),  # 65536: multi-CTA with E = 256
]


@pytest.mark.parametrize("T,E,k,C,skew,d,dt", DISPATCH_CASES)
def test_dispatch_token_choice(T, E, k, C, skew, d, dt, cuda_device):
    cfg = B.config(T=T, d=d, E=E, f=64, k=k, capacity_factor=C, dtype=dt)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    idx = random_assignment(T, E, k, seed=T + E + k, skew=skew, device=cuda_device)
    x = random_rows(T, d, seed=T, dtype=tdt, device=cuda_device)
    ws = torch.empty(B.moe_workspace_size(cfg, B.MOE_STAGE_DISPATCH), dtype=torch.uint8, device=cuda_device)
    off = torch.empty(E + 1, dtype=torch.int32, device=cuda_device)
    cnt = torch.empty(E, dtype=torch.int32, device=cuda_device)
    slot = torch.empty(T, k, dtype=torch.int32, device=cuda_device)
    x_perm = torch.empty(T * k, d, dtype=tdt, device=cuda_device)
    B.moe_dispatch(cfg, idx, x, off, cnt, slot, x_perm, ws)
    _check_device_error()
    cap = oracle.capacity(C, T, k, E)
    assert cap == B.moe_expert_capacity(cfg)
    o_off, o_cnt, o_slot, o_rows = oracle.dispatch_tc(idx, E, cap)
    np.testing.assert_array_equal(_np(off), o_off)
    np.testing.assert_array_equal(_np(cnt), o_cnt)
    np.testing.assert_array_equal(_np(slot), o_slot)
    A = int(o_off[-1])
    assert torch.equal(x_perm[:A], x[torch.from_numpy(o_rows).long().to(cuda_device)])


AFFINITY_CASES = [
    # T, E, k, capacity factor, skew, weight levels (0: continuous), d
    (8192, 64, 1, 1.25, 1.0, 0, 1024),
    (1000, 8, 2, 0.8, 1.5, 7, 128),         # seven weight values: many ties at the boundary
    (4096, 256, 8, 1.0, 0.5, 0, 256),
    (300, 8, 2, 0.01, 0.0, 0, 128),         # capacity 0: every assignment dropped
    (500, 16, 2, 20.0, 1.0, 0, 128),        # no expert reaches the limit: token order
]


@pytest.mark.parametrize("T,E,k,C,skew,levels,d", AFFINITY_CASES)
def test_dispatch_affinity(T, E, k, C, skew, levels, d, cuda_device):
    cfg = B.config(T=T, d=d, E=E, f=64, k=k, capacity_factor=C, drop_policy="affinity")
    idx = random_assignment(T, E, k, seed=T + E + 3 * k, skew=skew, device=cuda_device)
    w = random_weights((T, k), seed=T + 5)
    if levels:
        w = torch.floor(w * levels) / levels + 0.05
    x = random_rows(T, d, seed=T, device=cuda_device)
    ws = torch.empty(B.moe_workspace_size(cfg, B.MOE_STAGE_DISPATCH), dtype=torch.uint8, device=cuda_device)
    off = torch.empty(E + 1, dtype=torch.int32, device=cuda_device)
    cnt = torch.empty(E, dtype=torch.int32, device=cuda_device)
    slot = torch.empty(T, k, dtype=torch.int32, device=cuda_device)
    x_perm = torch.empty(T * k, d, dtype=torch.bfloat16, device=cuda_device)
    B.moe_dispatch(cfg, idx, x, off, cnt, slot, x_perm, ws, topk_w=w.to(cuda_device))
    _check_device_error()
    cap = oracle.capacity(C, T, k, E)
    o_off, o_cnt, o_slot, o_rows = oracle.dispatch_tc_affinity(_np(idx), w.numpy(), E, cap)
    np.testing.assert_array_equal(_np(off), o_off)
    np.testing.assert_array_equal(_np(cnt), o_cnt)
    np.testing.assert_array_equal(_np(slot), o_slot)
    A = int(o_off[-1])
    assert torch.equal(x_perm[:A], x[torch.from_numpy(o_rows).long().to(cuda_device)])
    dropped = int((o_slot < 0).sum())
    print(f"affinity T={T} E={E} k={k} cap={cap}: {dropped} assignments dropped")


def test_forward_affinity_drop(cuda_device):
    wl = WORKLOADS["switch_top1_cap1.25"].with_(T=600, d=256, E=8, f=256, capacity_factor=0.8,
                                                logit_offsets="normal_var0.5", drop_policy="affinity",
                                                name="affinity_drops")
    inp = make_inputs(wl, cuda_device)
    cfg, layer = _layer(wl, inp)
    y = layer.forward(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"], out=_nan_out(layer))
    gi, gw = (_np(t) for t in layer.route(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"]))
    _check_device_error()
    oi, ow, gap = oracle.route_tc(inp["x"], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                  wl.renorm, nthreads=NTH)
    cap = oracle.capacity(wl.capacity_factor, wl.T, wl.k, wl.E)
    # the oracle's drop on its own routing and fp64 weights
    o_off, _, o_slot, _ = oracle.dispatch_tc_affinity(oi, ow, wl.E, cap)
    # the GPU's drop, recomputed from its own routing and weights: compare tokens routed alike
    _, _, g_slot, _ = oracle.dispatch_tc_affinity(gi, gw, wl.E, cap)
    same = (gi == oi).all(axis=1) & ((g_slot >= 0) == (o_slot >= 0)).all(axis=1)
    assert (o_slot < 0).any() and same.mean() > 0.95
    toks = np.nonzero(same)[0]
    ref = oracle.forward_tc_streamed(inp["x"], oi, ow, o_slot, inp["W1"], inp["W3"], inp["W2"], toks,
                                     nthreads=NTH)
    err = rel_err(_np(y)[toks], ref)
    print(f"affinity forward: {len(toks)} tokens, {int((o_slot < 0).sum())} dropped, err {err:.3e}")
    assert err <= TOL["bf16"]


def test_dispatch_expert_choice(cuda_device):
    wl = EC_CASES["ec_small"]
    inp = make_inputs(wl, "cpu", weights=False)
    ot, ow, gap = oracle.route_ec(inp["x"], inp["W_r"], wl.ec_capacity, inp["logit_offset"], nthreads=NTH)
    cfg = B.config_from_workload(wl)
    x = inp["x"].to(cuda_device)
    tok = torch.from_numpy(ot).to(cuda_device)
    off = torch.empty(wl.E + 1, dtype=torch.int32, device=cuda_device)
    cnt = torch.empty(wl.E, dtype=torch.int32, device=cuda_device)
    slot = torch.empty(wl.T, wl.E, dtype=torch.int32, device=cuda_device)
    x_perm = torch.empty(wl.E * wl.ec_capacity, wl.d, dtype=torch.bfloat16, device=cuda_device)
    B.moe_dispatch(cfg, tok, x, off, cnt, slot, x_perm, None)
    _check_device_error()
    cap = wl.ec_capacity
    np.testing.assert_array_equal(_np(off), np.arange(wl.E + 1) * cap)
    np.testing.assert_array_equal(_np(cnt), np.full(wl.E, cap))
    want = -np.ones((wl.T, wl.E), np.int32)
    for e in range(wl.E):
        want[ot[e], e] = e * cap + np.arange(cap)
    np.testing.assert_array_equal(_np(slot), want)
    assert torch.equal(x_perm, x[tok.reshape(-1).long()])


# ------------------------------------------------------------------------------------------ experts

FFN_CASES = [
    # T, d, E, f, k, skew, n_shared, f_shared, dtype
    (700, 256, 8, 320, 2, 1.2, 0, 0, "bf16"),      # f % 128 != 0: 128-wide up tiles; empty experts
    (700, 256, 8, 384, 2, 1.2, 0, 0, "bf16"),      # skewed segments, 256-wide tiles
    (300, 384, 4, 256, 2, 0.0, 2, 128, "bf16"),    # d % 256 != 0: 128-wide down tiles; shared experts
    (1024, 1024, 8, 512, 1, 0.0, 0, 0, "bf16"),    # several full 128-row tiles per expert
    (129, 128, 3, 64, 1, 0.0, 1, 64, "bf16"),
    (200, 128, 8, 256, 2, 1.0, 1, 64, "f32"),      # CUDA-core fp32 path
]


@pytest.mark.parametrize("T,d,E,f,k,skew,ns,fs,dt", FFN_CASES)
def test_grouped_ffn(T, d, E, f, k, skew, ns, fs, dt, cuda_device):
    cfg = B.config(T=T, d=d, E=E, f=f, k=k, n_shared=ns, f_shared=fs, dtype=dt)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    g = torch.Generator(device="cpu").manual_seed(T * 7 + d)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).to(tdt)
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).to(tdt)
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).to(tdt)
    Ws = None
    if ns:
        Ws = [(torch.randn(ns, d, fs, generator=g) / d ** 0.5).to(tdt),
              (torch.randn(ns, d, fs, generator=g) / d ** 0.5).to(tdt),
              (torch.randn(ns, fs, d, generator=g) / fs ** 0.5).to(tdt)]
    x = random_rows(T, d, seed=d + T, dtype=tdt)
    idx = random_assignment(T, E, k, seed=5 + T, skew=skew)
    o_off, _, o_slot, o_rows = oracle.dispatch_tc(idx, E, -1)
    x_perm = torch.zeros(T * k, d, dtype=tdt)
    x_perm[: len(o_rows)] = x[torch.from_numpy(o_rows).long()]
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws) if Ws else (None,) * 3)
    Y = layer.grouped_ffn(x_perm.to(dev), torch.from_numpy(o_off).to(dev), x.to(dev))
    _check_device_error()
    Yn = _np(Y)
    ref = np.zeros((T * k + (T if ns else 0), d))
    for e in range(E):
        a, b = int(o_off[e]), int(o_off[e + 1])
        if b > a:
            ref[a:b] = oracle.expert_rows(x_perm[a:b], W1[e], W3[e], W2[e], nthreads=NTH)
    A = int(o_off[-1])
    assert rel_err(Yn[:A], ref[:A]) <= TOL[dt]
    if ns:
        sref = sum(oracle.expert_rows(x, Ws[0][s], Ws[1][s], Ws[2][s], nthreads=NTH) for s in range(ns))
        assert rel_err(Yn[T * k:], sref) <= TOL[dt]


# Long segments: the expert GEMMs take a segment's M tiles in groups of nearly equal
# size (every N block of a group before the next), at most as many per group as fit
# the tile-group share of L2 (moe_set_tile_group_bytes).  The default shares group
# nothing at these small d and f, so the test also forces groups of 16 and of 3 (up)
# / 5 (down) M tiles.  The sizes give segments of 1, 2, 3, 16, 17 and 33 M tiles
# (last tiles of one row, 2049, of a full tile, 2048 and 4096, and short ones, 2100,
# 4097), short segments next to them (0, 1, 129, 300) and a shared segment of 43 M
# tiles: groups of 3 split 17 into 3+3+3+3+3+2 and 16 into 3+3+3+3+2+2, groups of 5
# split 17 into 5+4+4+4.  Every row is compared with the oracle.
LONG_SEG_CASES = [
    # T, d, f, f_shared, counts of the 8 routed experts
    (5400, 256, 256, 128, [0, 1, 2049, 129, 4097, 2048, 300, 2100]),
    (5400, 512, 384, 256, [4096, 129, 0, 2049, 1, 2100, 300, 1800]),
]
TILE_GROUPS = [None, (16, 16), (3, 5)]   # M tiles per group (up, down); None: the default shares
@pytest.mark.parametrize("groups", TILE_GROUPS)
@pytest.mark.parametrize("T,d,f,fs,counts", LONG_SEG_CASES)
def test_grouped_ffn_long_segments(T, d, f, fs, counts, groups, cuda_device):
    E, k = 8, 2
    A = int(sum(counts))
    assert max(counts) > 16 * 128 and A <= T * k
    cfg = B.config(T=T, d=d, E=E, f=f, k=k, n_shared=1, f_shared=fs)
    g = torch.Generator(device="cpu").manual_seed(9090 + d)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).bfloat16()
    Ws = [(torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, fs, d, generator=g) / fs ** 0.5).bfloat16()]
    off = np.zeros(E + 1, np.int32)
    off[1:] = np.cumsum(counts)
    x_perm = torch.zeros(T * k, d, dtype=torch.bfloat16)
    x_perm[:A] = random_rows(A, d, seed=91 + d, dtype=torch.bfloat16)
    x = random_rows(T, d, seed=92 + d, dtype=torch.bfloat16)
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    try:
        if groups is not None:   # bytes of A rows per group: M tiles x 128 rows x K x 2 bytes
            B.moe_set_tile_group_bytes(groups[0] * 128 * d * 2, groups[1] * 128 * f * 2)
        for _ in range(2):   # twice: the second call reuses the workspace and its counters
            Y = layer.grouped_ffn(x_perm.to(dev), torch.from_numpy(off).to(dev), x.to(dev))
            _check_device_error()
            Yn = _np(Y)
            for e in range(E):
                a, b = int(off[e]), int(off[e + 1])
                if b > a:
                    ref = oracle.expert_rows(x_perm[a:b], W1[e], W3[e], W2[e], nthreads=NTH)
                    assert rel_err(Yn[a:b], ref) <= TOL["bf16"], f"expert {e} ({b - a} rows)"
            sref = oracle.expert_rows(x, Ws[0][0], Ws[1][0], Ws[2][0], nthreads=NTH)
            assert rel_err(Yn[T * k:], sref) <= TOL["bf16"]
    finally:
        B.moe_set_tile_group_bytes(0, 0)


# The same long segments with forced groups of 3 (up) / 5 (down) M tiles in every
# kernel that walks the grouped tile order: the bf16 and FP8-weight (W8) kernels as
# one fused launch and as separate up and down launches, and the fused launch with
# the E4M3 up projection.  Every row compared with the oracle of the mode.
@pytest.mark.parametrize("dt", ["bf16", "fp8w", "fp8up"])
def test_grouped_ffn_long_segments_forced_groups(dt, cuda_device):
    T, d, f, fs, counts = LONG_SEG_CASES[0]
    E, k = 8, 2
    A = int(sum(counts))
    cfg = B.config(T=T, d=d, E=E, f=f, k=k, n_shared=1, f_shared=fs, dtype=dt)
    g = torch.Generator(device="cpu").manual_seed(9191)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).bfloat16()
    Ws = [(torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, fs, d, generator=g) / fs ** 0.5).bfloat16()]
    off = np.zeros(E + 1, np.int32)
    off[1:] = np.cumsum(counts)
    x_perm = torch.zeros(T * k, d, dtype=torch.bfloat16)
    x_perm[:A] = random_rows(A, d, seed=93, dtype=torch.bfloat16)
    x = random_rows(T, d, seed=94, dtype=torch.bfloat16)

    def ref_rows(X, w1, w3, w2):
        Xf = X.float().numpy()
        if dt == "fp8w":
            return oracle.expert_rows_fp8(Xf, *_fp8_quant(w1, w3, w2))
        if dt == "fp8up":
            return oracle.expert_rows_fp8up(Xf, w1.float().numpy(), w3.float().numpy(), w2.float().numpy())
        return oracle.expert_rows(X, w1, w3, w2, nthreads=NTH)

    ref = np.zeros((T * k + T, d))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            ref[a:b] = ref_rows(x_perm[a:b], W1[e], W3[e], W2[e])
    ref[T * k:] = ref_rows(x, Ws[0][0], Ws[1][0], Ws[2][0])
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    off_d, xp_d, x_d = torch.from_numpy(off).to(dev), x_perm.to(dev), x.to(dev)
    try:
        B.moe_set_tile_group_bytes(3 * 128 * d * 2, 5 * 128 * f * 2)
        outs = [_np(layer.grouped_ffn(xp_d, off_d, x_d))]
        if dt != "fp8up":   # the E4M3 up projection has no separate launches
            H = torch.empty(T * k, f, dtype=torch.bfloat16, device=dev)
            Hs = torch.empty(T, fs, dtype=torch.bfloat16, device=dev)
            Y2 = torch.empty(T * k + T, d, dtype=torch.bfloat16, device=dev)
            B.moe_grouped_ffn_up(cfg, xp_d, off_d, layer.packed, x_d, H, Hs)
            B.moe_grouped_ffn_down(cfg, H, Hs, off_d, layer.packed, Y2)
            outs.append(_np(Y2))
        _check_device_error()
    finally:
        B.moe_set_tile_group_bytes(0, 0)
    for got in outs:
        for e in range(E):
            a, b = int(off[e]), int(off[e + 1])
            if b > a:
                assert rel_err(got[a:b], ref[a:b]) <= TOL["bf16"], (dt, e, b - a)
        assert rel_err(got[T * k:], ref[T * k:]) <= TOL["bf16"]


# The fine-grained layout at its widest: 256 routed experts plus one shared expert
# (257 segments) with small d and f, so that every row of every segment can be
# compared with the oracle.  The segment sizes are seeded and skewed and include
# empty experts and sizes on both sides of the 128-row M tile.
MANY_SEG_CASES = [
    # d, f, f_shared: both tiles 256 wide (one fused launch with its per-M-tile
    # counters), then 128-wide up tiles (f % 128 != 0: separate up and down launches)
    (256, 128, 128),
    (384, 192, 64),
]


@pytest.mark.parametrize("d,f,fs", MANY_SEG_CASES)
def test_grouped_ffn_257_segments(d, f, fs, cuda_device):
    E, k = 256, 8
    rng = np.random.default_rng(d + f)
    counts = rng.choice([0, 1, 2, 17, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257], size=E)
    counts[:6] = [0, 129, 1, 128, 0, 256]   # fixed edges first
    A = int(counts.sum())
    T = (A + k - 1) // k + 3                 # rows_routed = T * k >= A; T rows of shared input
    cfg = B.config(T=T, d=d, E=E, f=f, k=k, n_shared=1, f_shared=fs)
    g = torch.Generator(device="cpu").manual_seed(4242 + d)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).bfloat16()
    Ws = [(torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, fs, d, generator=g) / fs ** 0.5).bfloat16()]
    off = np.zeros(E + 1, np.int32)
    off[1:] = np.cumsum(counts)
    x_perm = torch.zeros(T * k, d, dtype=torch.bfloat16)
    x_perm[:A] = random_rows(A, d, seed=77 + d, dtype=torch.bfloat16)
    x = random_rows(T, d, seed=78 + d, dtype=torch.bfloat16)
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    Y = layer.grouped_ffn(x_perm.to(dev), torch.from_numpy(off).to(dev), x.to(dev))
    _check_device_error()
    Yn = _np(Y)
    ref = np.zeros((A, d))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            ref[a:b] = oracle.expert_rows(x_perm[a:b], W1[e], W3[e], W2[e], nthreads=NTH)
    # every routed row, per segment (a failing segment is named), then the shared rows
    scale = np.abs(ref).max()
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            err = np.abs(Yn[a:b] - ref[a:b]).max() / scale
            assert err <= TOL["bf16"], f"expert {e} ({b - a} rows): {err:.3e}"
    sref = oracle.expert_rows(x, Ws[0][0], Ws[1][0], Ws[2][0], nthreads=NTH)
    assert rel_err(Yn[T * k:], sref) <= TOL["bf16"]
    print(f"257 segments, {A} routed rows + {T} shared rows compared, "
          f"max|err|/max|ref| = {rel_err(Yn[:A], ref):.3e}")


# Segment sizes around the 128-row M tile: 1, 15, 16, 17, 111, 112, 113, 127, 128,
# 129, 240 rows and an empty expert; the shared segment (T = 1029 rows) ends in a
# 5-row tile.
# segment sizes on both sides of the 16-row MMA step, of the 64-row limit of the
# M = 64 tiles (also as a second M tile: 192, 193) and of the 128-row M tile
EDGE_COUNTS = [1, 15, 16, 17, 63, 64, 65, 111, 112, 113, 127, 128, 129, 192, 193, 240, 0]


@pytest.mark.parametrize("d,f", [(256, 256), (384, 128)])
def test_grouped_ffn_tile_edges(d, f, cuda_device):
    E, T, ns, fs = len(EDGE_COUNTS), sum(EDGE_COUNTS), 1, 128
    cfg = B.config(T=T, d=d, E=E, f=f, k=1, n_shared=ns, f_shared=fs, dtype="bf16")
    g = torch.Generator(device="cpu").manual_seed(d + f)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).to(torch.bfloat16)
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).to(torch.bfloat16)
    Ws = [(torch.randn(ns, d, fs, generator=g) / d ** 0.5).to(torch.bfloat16),
          (torch.randn(ns, d, fs, generator=g) / d ** 0.5).to(torch.bfloat16),
          (torch.randn(ns, fs, d, generator=g) / fs ** 0.5).to(torch.bfloat16)]
    x = random_rows(T, d, seed=11, dtype=torch.bfloat16)
    order = np.random.default_rng(7).permutation(T)
    idx = np.repeat(np.arange(E, dtype=np.int32), EDGE_COUNTS)[order].reshape(T, 1)
    o_off, _, _, o_rows = oracle.dispatch_tc(idx, E, -1)
    assert np.diff(o_off).tolist() == EDGE_COUNTS
    x_perm = x[torch.from_numpy(o_rows).long()]
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    off_d, xp_d, x_d = torch.from_numpy(o_off).to(dev), x_perm.to(dev), x.to(dev)
    Y = _np(layer.grouped_ffn(xp_d, off_d, x_d))
    # the two GEMMs as separate launches too
    H = torch.empty(T, f, dtype=torch.bfloat16, device=dev)
    Hs = torch.empty(T, fs, dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty(2 * T, d, dtype=torch.bfloat16, device=dev)
    B.moe_grouped_ffn_up(cfg, xp_d, off_d, layer.packed, x_d, H, Hs)
    B.moe_grouped_ffn_down(cfg, H, Hs, off_d, layer.packed, Y2)
    Y2 = _np(Y2)
    _check_device_error()
    ref = np.zeros((2 * T, d))
    for e in range(E):
        a, b = int(o_off[e]), int(o_off[e + 1])
        if b > a:
            ref[a:b] = oracle.expert_rows(x_perm[a:b], W1[e], W3[e], W2[e], nthreads=NTH)
    ref[T:] = oracle.expert_rows(x, Ws[0][0], Ws[1][0], Ws[2][0], nthreads=NTH)
    for got in (Y, Y2):
        # per segment, so that one short tile going wrong cannot hide behind the others
        for e in range(E):
            a, b = int(o_off[e]), int(o_off[e + 1])
            if b > a:
                assert rel_err(got[a:b], ref[a:b]) <= TOL["bf16"], (e, b - a)
        assert rel_err(got[T:], ref[T:]) <= TOL["bf16"]


# ------------------------------------------------------------------------------------- load statistics
# The router's score sums (moe_route's prob_sum) and moe_load_stats against the
# oracle's definitions.  The count-based parts (fractions, LIF, CV) are computed by
# both sides from the GPU's own routing and counts, the GPU in fp32: bar 1e-5
# relative.  The score means come from fp32 scores (bf16 inputs, fp32 tensor-core
# logits, about 1e-6 relative per score) summed in fp32: bar 1e-4 relative.
STATS_CASES = ["tiny_top2_fp32", "switch_top1_cap1.25", "deepseek_v3", "mixtral_T256", "sigmoid_top8_splitk",
               "ec_small", "ec_splitk"]


@pytest.mark.parametrize("name", STATS_CASES)
def test_load_stats(name, cuda_device):
    wl = WORKLOADS[name] if name in WORKLOADS else (SMALL_TC[name] if name in SMALL_TC else EC_CASES[name])
    dev = cuda_device
    inp = make_inputs(wl, dev, weights=False)
    cfg = B.config_from_workload(wl)
    ec = wl.mode == "ec"
    sel = (wl.E, wl.ec_capacity) if ec else (wl.T, wl.k)
    ws = torch.empty(max(1, B.moe_workspace_size(cfg, B.MOE_STAGE_ROUTE)), dtype=torch.uint8, device=dev)
    idx = torch.empty(sel, dtype=torch.int32, device=dev)
    w = torch.empty(sel, dtype=torch.float32, device=dev)
    psum = torch.full((wl.E,), 7.0, dtype=torch.float32, device=dev)   # overwritten, not accumulated into
    B.moe_route(cfg, inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"], idx, w, ws, prob_sum=psum)
    rows_routed, _ = B.moe_buffer_rows(cfg)
    wsd = torch.empty(max(1, B.moe_workspace_size(cfg, B.MOE_STAGE_DISPATCH)), dtype=torch.uint8, device=dev)
    off = torch.empty(wl.E + 1, dtype=torch.int32, device=dev)
    cnt = torch.empty(wl.E, dtype=torch.int32, device=dev)
    slot = torch.empty((wl.T, wl.E) if ec else (wl.T, wl.k), dtype=torch.int32, device=dev)
    xp = torch.empty(max(1, rows_routed), wl.d, dtype=inp["x"].dtype, device=dev)
    B.moe_dispatch(cfg, idx, inp["x"], off, cnt, slot, xp, wsd)
    frac = torch.empty(wl.E, dtype=torch.float32, device=dev)
    pmean = torch.empty(wl.E, dtype=torch.float32, device=dev)
    summary = torch.empty(5, dtype=torch.float64, device=dev)
    B.moe_load_stats(cfg, idx, cnt, psum, frac, pmean, summary)
    _check_device_error()
    if ec:
        scores = oracle.route_ec(inp["x"], inp["W_r"], wl.ec_capacity, inp["logit_offset"], nthreads=NTH,
                                 want_scores=True)[3]
    else:
        scores = oracle.route_tc(inp["x"], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                 wl.renorm, nthreads=NTH, want_scores=True)[3]
    f, P, s = oracle.load_stats(_np(idx), _np(cnt), scores, expert_choice=ec)
    gs = summary.cpu().numpy()
    np.testing.assert_allclose(_np(frac), f, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(_np(pmean), P, rtol=1e-4, atol=1e-7)
    np.testing.assert_allclose(_np(psum) / wl.T, P, rtol=1e-4, atol=1e-7)
    np.testing.assert_allclose(gs[:2], s[:2], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(gs[2:], s[2:], rtol=1e-4, atol=0)
    print(f"{name}: LIF {gs[0]:.3f} CV {gs[1]:.3f} H {gs[2]:.4f} (ln E {np.log(wl.E):.4f}) "
          f"switch {gs[3]:.4f} balance {gs[4]:.4f}")


# ------------------------------------------------------------------------------------------ combine

@pytest.mark.parametrize("T,E,k,C,d,ns,dt", [(1000, 8, 2, 1.0, 256, 0, "bf16"), (4096, 256, 8, 0.0, 7168, 1, "bf16"),
                                             (333, 16, 1, 1.25, 128, 1, "f32"),
                                             # few tokens: rows split into spans, the last one ragged
                                             (16, 8, 2, 0.0, 4096, 0, "bf16"), (5, 8, 3, 0.0, 1152, 1, "bf16"),
                                             (1, 4, 2, 0.0, 576, 1, "f32")])
def test_combine_token_choice(T, E, k, C, d, ns, dt, cuda_device):
    cfg = B.config(T=T, d=d, E=E, f=64, k=k, capacity_factor=C, n_shared=ns, f_shared=64 if ns else 0, dtype=dt)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    idx = random_assignment(T, E, k, seed=3 * T, skew=1.0)
    cap = oracle.capacity(C, T, k, E)
    _, _, o_slot, _ = oracle.dispatch_tc(idx, E, cap)
    rows_total = T * k + (T if ns else 0)
    Y = random_rows(rows_total, d, seed=T + 1, dtype=tdt)
    w = random_weights((T, k), seed=T)
    layer_y = torch.empty(T, d, dtype=tdt, device=cuda_device)
    B.moe_combine(cfg, Y.to(cuda_device), torch.from_numpy(o_slot).to(cuda_device), w.to(cuda_device), layer_y)
    _check_device_error()
    Yf = Y.float().numpy()
    ref = oracle.combine_tc(Yf, o_slot, w.numpy(), Y_shared=Yf[T * k:] if ns else None)
    assert rel_err(_np(layer_y), ref) <= TOL[dt] / 4


def test_combine_expert_choice(cuda_device):
    T, E, cap, d = 1000, 16, 100, 256
    cfg = B.config(T=T, d=d, E=E, f=64, mode="ec", ec_capacity=cap)
    wl = EC_CASES["ec_small"]
    inp = make_inputs(wl, "cpu", weights=False)
    ot, ow, _ = oracle.route_ec(inp["x"], inp["W_r"], cap, inp["logit_offset"], nthreads=NTH)
    slot = -np.ones((T, E), np.int32)
    for e in range(E):
        slot[ot[e], e] = e * cap + np.arange(cap)
    Y = random_rows(E * cap, d, seed=17)
    w = torch.from_numpy(ow.astype(np.float32))
    y = torch.empty(T, d, dtype=torch.bfloat16, device=cuda_device)
    B.moe_combine(cfg, Y.to(cuda_device), torch.from_numpy(slot).to(cuda_device), w.to(cuda_device), y)
    _check_device_error()
    ref = oracle.combine_ec(Y.float().numpy(), slot, w.numpy())
    assert rel_err(_np(y), ref) <= TOL["bf16"] / 4


# ------------------------------------------------------------------------------------------ whole layer

def _sample_tokens(T, n, seed, must=()):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | set(int(t) for t in must)
    return np.array(sorted(pick), np.int64)


def _segment_tails(gi, g_slot, usable, E):
    """For every expert with kept rows, the token of its last kept row in the GPU's
    own routing (the row that ends its segment, in its last M tile).  A tail
    token whose routing differs from the oracle's (a near tie) cannot be compared;
    the expert's last usable token stands in for it.  Returns (tokens, experts
    with rows, experts whose true tail token is compared)."""
    T, k = gi.shape
    kept = g_slot >= 0
    ts = np.repeat(np.arange(T), k)[kept.ravel()]
    es = gi.ravel()[kept.ravel()]
    last = np.full(E, -1)
    np.maximum.at(last, es, ts)
    ok = usable[ts]
    last_ok = np.full(E, -1)
    np.maximum.at(last_ok, es[ok], ts[ok])
    with_rows = np.nonzero(last >= 0)[0]
    exact = int(sum(last_ok[e] == last[e] for e in with_rows))
    toks = np.unique(last_ok[last_ok >= 0]).astype(np.int64)
    return toks, len(with_rows), exact


def _group_starts(mblk, group_m):
    """First M tile of every group of a segment of mblk M tiles in the expert GEMMs'
    tile order: ceil(mblk / group_m) groups of nearly equal size, the larger first."""
    if group_m <= 0 or mblk <= group_m:
        return [0]
    ng = -(-mblk // group_m)
    base, big = divmod(mblk, ng)
    starts, m = [], 0
    for i in range(ng):
        starts.append(m)
        m += base + (1 if i < big else 0)
    return starts


def _segment_group_rows(gi, g_slot, g_off, usable, wl):
    """For every expert, the tokens of the rows that open and close each group of M
    tiles of its segment in the up and in the down projection (the default shares of
    moe_set_tile_group_bytes: 40 MiB of x_perm rows, 64 MiB of H rows), and its first
    and last row, in the GPU's own routing, where the routing agrees with the
    oracle's: the tiles on both sides of every group boundary of the tile order."""
    up_bytes, down_bytes = B.moe_get_tile_group_bytes()
    gms = (max(1, up_bytes // (128 * wl.d * 2)), max(1, down_bytes // (128 * wl.f * 2)))
    toks = []
    for e in range(wl.E):
        n = int(g_off[e + 1] - g_off[e])
        if n == 0:
            continue
        mblk = -(-n // 128)
        ranks = {0, n - 1}
        for gm in gms:
            for m0 in _group_starts(mblk, gm)[1:]:
                ranks.update((128 * m0 - 1, 128 * m0))
        rel = g_slot - g_off[e]
        for t, j in zip(*np.nonzero((gi == e) & (g_slot >= 0))):
            if int(rel[t, j]) in ranks and usable[t]:
                toks.append(int(t))
    return np.unique(np.array(toks, np.int64))


# tokens compared at full size: None = all; an int = a seeded sample of that many;
# "tails" = the last row of every expert segment (+ a seeded sample of 24 and the
# shared segment's last token), so each segment's tail M tile is checked;
# "groups" = the rows at every group boundary of every expert segment (+ 12 sampled)
E2E_CASES = {
    "tiny_top2_fp32": None,
    "switch_top1_cap1.25": 48,
    "mixtral_T16": None,
    "mixtral_T256": 24,
    "mixtral_T4096": 16,
    "mixtral_T16384": "groups",
    "deepseek_v3": "tails",
    "expert_choice_zipf": 16,
}
E2E_SMALL = {
    "small_top2_ragged": WORKLOADS["mixtral_T256"].with_(T=333, d=256, f=384, name="small_top2_ragged"),
    "small_sigmoid_shared": WORKLOADS["deepseek_v3"].with_(T=150, d=256, E=32, f=128, f_shared=192,
                                                            name="small_sigmoid_shared"),
    "small_switch_drops": WORKLOADS["switch_top1_cap1.25"].with_(T=600, d=256, E=8, f=256, capacity_factor=0.8,
                                                                  logit_offsets="normal_var0.5",
                                                                  name="small_switch_drops"),
    "small_ec": EC_CASES["ec_small"],
    "small_fp32_shared": WORKLOADS["tiny_top2_fp32"].with_(T=100, n_shared=2, f_shared=64, name="small_fp32_sh"),
    # degenerate layers: k = E (the full softmax mixture), E = 1 (a dense SwiGLU FFN;
    # the router is a transposed copy since E is not a multiple of 8), one token
    "small_k_eq_E": WORKLOADS["mixtral_T256"].with_(T=200, d=256, E=4, k=4, f=128, name="small_k_eq_E"),
    "small_dense_E1": WORKLOADS["mixtral_T256"].with_(T=130, d=256, E=1, k=1, f=256, name="small_dense_E1"),
    "small_one_token": WORKLOADS["mixtral_T16"].with_(T=1, d=256, f=128, name="small_one_token"),
    # segments longer than 16 M tiles (2048 rows): top-2 softmax, and capacity with
    # the gated down store of k = 1 (at this d and f the default tile-group shares keep
    # each segment in one group; the forced-group tests walk such segments in groups)
    "small_long_top2": WORKLOADS["mixtral_T256"].with_(T=9000, d=256, f=256, name="small_long_top2"),
    "small_long_switch": WORKLOADS["switch_top1_cap1.25"].with_(T=24000, d=256, E=8, f=256,
                                                                 logit_offsets="normal_var0.5",
                                                                 name="small_long_switch"),
}


def _nan_out(layer):
    """Output buffer full of NaN: a row the forward leaves unwritten fails the comparison."""
    return torch.full((layer.cfg.T, layer.cfg.d), float("nan"), dtype=layer.dtype, device=layer.device)


def _run_e2e(wl, n_sample, cuda_device):
    inp = make_inputs(wl, cuda_device)
    cfg, layer = _layer(wl, inp)
    y = layer.forward(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"], out=_nan_out(layer))
    r_idx, r_w = layer.route(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"])
    _check_device_error()
    T = wl.T
    if wl.mode == "ec":
        ot, ow, gap, S = oracle.route_ec(inp["x"], inp["W_r"], wl.ec_capacity, inp["logit_offset"], nthreads=NTH,
                                         want_scores=True)
        amb = _check_ec_selection(_np(r_idx), _np(r_w), ot, S, wl.ec_capacity)
        counts = np.bincount(ot.reshape(-1), minlength=T)
        must = [int(np.argmax(counts))] + np.nonzero(counts == 0)[0][:4].tolist()
        toks = np.arange(T) if n_sample is None else _sample_tokens(T, n_sample, T, must)
        toks = np.array([t for t in toks if t not in amb], np.int64)
        ref = oracle.forward_ec_streamed(inp["x"], ot, ow, inp["W1"], inp["W3"], inp["W2"], toks, inp.get("W1s"),
                                         inp.get("W3s"), inp.get("W2s"), nthreads=NTH)
    else:
        oi, ow, gap = oracle.route_tc(inp["x"], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                      wl.renorm, nthreads=NTH)
        gi = _np(r_idx)
        near = gap < GAP
        np.testing.assert_array_equal(gi[~near], oi[~near])
        cap = oracle.capacity(wl.capacity_factor, T, wl.k, wl.E)
        o_off, o_cnt, o_slot, _ = oracle.dispatch_tc(oi, wl.E, cap)
        g_off, g_cnt, g_slot, _ = oracle.dispatch_tc(gi, wl.E, cap)   # the GPU's own choices, dispatched
        same = (gi == oi).all(axis=1) & ((g_slot >= 0) == (o_slot >= 0)).all(axis=1)
        dropped = np.nonzero((o_slot < 0).any(axis=1))[0]
        if n_sample == "tails":
            tails, n_rows, n_tail = _segment_tails(gi, g_slot, same, wl.E)
            reached = np.unique(gi[tails][g_slot[tails] >= 0])
            print(f"{wl.name}: {n_rows} of {wl.E} experts have rows, {len(reached)} reached by the sample; "
                  f"the segment's last row compared for {n_tail} of them")
            assert len(reached) == n_rows and n_tail >= 0.95 * n_rows
            toks = _sample_tokens(T, 24, T, list(tails) + [T - 1])
        elif n_sample == "groups":
            bounds = _segment_group_rows(gi, g_slot, g_off, same, wl)
            print(f"{wl.name}: {len(bounds)} tokens at group boundaries of the expert segments")
            assert len(bounds) >= wl.E
            toks = _sample_tokens(T, 12, T, list(bounds))
        else:
            toks = np.arange(T) if n_sample is None else _sample_tokens(T, n_sample, T, dropped[:64])
        toks = np.array([t for t in toks if same[t]], np.int64)
        print(f"{wl.name}: {int(near.sum())} near-tie tokens, {len(dropped)} tokens with a dropped slot")
        ref = oracle.forward_tc_streamed(inp["x"], oi, ow, o_slot, inp["W1"], inp["W3"], inp["W2"], toks,
                                         inp.get("W1s"), inp.get("W3s"), inp.get("W2s"), nthreads=NTH)
    got = _np(y)[toks]
    err = rel_err(got, ref)
    print(f"{wl.name}: {len(toks)} tokens compared, max|err|/max|ref| = {err:.3e}")
    assert err <= TOL[wl.dtype]
    return err


@pytest.mark.parametrize("name", list(E2E_CASES))
def test_forward_full_size(name, cuda_device):
    _run_e2e(WORKLOADS[name], E2E_CASES[name], cuda_device)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(E2E_SMALL))
def test_forward_small_all_tokens(name, cuda_device):
    _run_e2e(E2E_SMALL[name], None, cuda_device)


BACK_TO_BACK = dict(E2E_SMALL, split_router_shared=WORKLOADS["deepseek_v3"].with_(
    T=200, d=2048, E=32, f=128, f_shared=128, name="b2b_split"))


@pytest.mark.parametrize("name", list(BACK_TO_BACK))
def test_forward_back_to_back(name, cuda_device):
    """Forwards queued back to back on one stream with no host synchronisation, their
    input rewritten by a torch kernel in between (every kernel after the first of a
    call starts before its predecessor ends and waits on the device): each output
    equals the same forward run on its own, bit for bit."""
    wl = BACK_TO_BACK[name]
    inp = make_inputs(wl, cuda_device)
    cfg, layer = _layer(wl, inp)
    args = (inp["W_r"], inp["logit_offset"], inp["sel_bias"])
    xs = [inp["x"], random_rows(wl.T, wl.d, seed=7, dtype=inp["x"].dtype, device=cuda_device), inp["x"] * 0.5]
    ref = []
    for x in xs:
        y = layer.forward(x, *args, out=_nan_out(layer))
        _check_device_error()
        ref.append(y.clone())
    xbuf = torch.empty_like(inp["x"])
    outs = []
    for _ in range(2):
        for x in xs:
            xbuf.copy_(x)
            outs.append(layer.forward(xbuf, *args, out=_nan_out(layer)))
    _check_device_error()
    for i, y in enumerate(outs):
        assert torch.equal(y, ref[i % len(xs)]), f"forward {i} differs from its isolated run"
    # inputs uploaded from pinned host memory on a side stream, the forward ordered
    # after the upload by an event (the end-to-end loop of bench.py), double-buffered
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    hosts = [x.cpu().pin_memory() for x in xs]
    bufs = [torch.empty_like(inp["x"]) for _ in range(2)]
    done = [None, None]
    outs = []
    for i in range(2 * len(xs)):
        b = i & 1
        with torch.cuda.stream(side):
            if done[b] is not None:
                side.wait_event(done[b])              # the forward two steps back has read bufs[b]
            bufs[b].copy_(hosts[i % len(xs)], non_blocking=True)
            up = torch.cuda.Event()
            up.record(side)
        main.wait_event(up)
        outs.append(layer.forward(bufs[b], *args, out=_nan_out(layer)))
        done[b] = torch.cuda.Event()
        done[b].record(main)
    _check_device_error()
    for i, y in enumerate(outs):
        assert torch.equal(y, ref[i % len(xs)]), f"uploaded forward {i} differs from its isolated run"


def test_forward_empty_batch(cuda_device):
    wl = WORKLOADS["mixtral_T16"].with_(T=0, d=128, f=64)
    cfg = B.config_from_workload(wl)
    dev = cuda_device
    E, d, f = wl.E, wl.d, wl.f
    W = torch.zeros(E, d, f, dtype=torch.bfloat16, device=dev)
    layer = MoELayer(cfg, W, W, torch.zeros(E, f, d, dtype=torch.bfloat16, device=dev))
    x = torch.zeros(1, d, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(1, d, dtype=torch.bfloat16, device=dev)
    B.moe_forward(cfg, x, torch.zeros(d, E, dtype=torch.bfloat16, device=dev), None, None, layer.packed, y,
                  layer.workspace())
    _check_device_error()


# ------------------------------------------------------------------------------------- FP8 expert weights
# MOE_BF16_FP8W: moe_pack_weights stores every expert matrix as E4M3 codes with one
# fp32 scale per output channel; the grouped FFN expands the codes to bf16 in
# shared memory and applies the scales in its epilogue.  Packing is compared bit for
# bit with the oracle's quantiser; layer outputs against the oracle's fp64 expert
# with the same codes and scales, within the bf16 bar.

def _e4m3_decode():
    """Value of every E4M3 code (NaN codes -> nan), from the format's definition."""
    out = np.empty(256)
    for code in range(256):
        sgn = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 7
        if e == 15 and m == 7:
            out[code] = np.nan
        elif e == 0:
            out[code] = sgn * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = sgn * (1 + m / 8.0) * 2.0 ** (e - 7)
    return out


E4M3 = _e4m3_decode()


def _packed_offsets(E, d, f, fs):
    """Byte offsets of the FP8 packed buffer (regions 1024-byte aligned, in order)."""
    sizes = [("w13", E * 2 * f * d), ("w2", E * d * f), ("w13s", 2 * fs * d), ("w2s", d * fs),
             ("sc13", 4 * E * 2 * f), ("sc2", 4 * E * d), ("sc13s", 4 * 2 * fs), ("sc2s", 4 * d)]
    off, o = {}, 0
    for name, n in sizes:
        off[name] = o
        o = (o + n + 1023) // 1024 * 1024
    return off


def _tiled8(p, i, BN, K):
    nb, r, kb = p // BN, p % BN, i // 64
    return ((nb * (K // 64) + kb) * BN + r) * 64 + i % 64


def _unpack_up(buf, base, scbase, W_rows, d, f, BN=256):
    """(codes as values [d][f], scales [f]) of W1 (m = 0) or W3 (m = 1) from the
    packed up image; packed row of hidden column h = (h // 64) * 128 + m * 64 + h % 64."""
    out = []
    for m in (0, 1):
        h = np.arange(f)
        p = (h // 64) * 128 + m * 64 + h % 64
        I, H = np.meshgrid(np.arange(d), h, indexing="ij")
        q = E4M3[buf[base + _tiled8(p[H], I, BN, d)]]
        s = np.frombuffer(buf[scbase:scbase + 4 * 2 * f].tobytes(), np.float32)[p]
        out.append((q, s))
    return out


def _unpack_down(buf, base, scbase, d, f, BN=256):
    n = np.arange(d)
    Hh, N = np.meshgrid(np.arange(f), n, indexing="ij")
    q = E4M3[buf[base + _tiled8(N, Hh, BN, f)]]
    s = np.frombuffer(buf[scbase:scbase + 4 * d].tobytes(), np.float32)
    return q, s


def _fp8_quant(W1, W3, W2):
    (q1, s1), (q3, s3), (q2, s2) = (oracle.quantize_e4m3_columns(w.float().numpy()) for w in (W1, W3, W2))
    return q1, s1, q3, s3, q2, s2


def _merged_shared(W1s, W3s, W2s):
    """The shared experts as one expert of hidden width n_shared * f_shared (as
    packed): W1/W3 concatenated along the hidden columns, W2 along its rows."""
    return (torch.cat(list(W1s), dim=1), torch.cat(list(W3s), dim=1), torch.cat(list(W2s), dim=0))


def test_fp8_packing_is_exact(cuda_device):
    E, d, f, fs = 3, 256, 256, 128
    cfg = B.config(T=16, d=d, E=E, f=f, k=1, n_shared=1, f_shared=fs, dtype="fp8w")
    g = torch.Generator(device="cpu").manual_seed(99)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).bfloat16()
    W1[1, :, 5] = 0                                     # an all-zero channel: scale 0, codes 0
    W2[2, :, 17] = 0
    W1[0, 7, 9] = 3.0e-7                                # tiny weights that land on E4M3 subnormals
    Ws = [(torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, fs, d, generator=g) / fs ** 0.5).bfloat16()]
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    torch.cuda.synchronize()
    buf = layer.packed.cpu().numpy()
    off = _packed_offsets(E, d, f, fs)
    for e in range(E):
        got = _unpack_up(buf, off["w13"] + e * 2 * f * d, off["sc13"] + 4 * e * 2 * f, None, d, f)
        for (gq, gs), W in zip(got, (W1[e], W3[e])):
            q, s = oracle.quantize_e4m3_columns(W.float().numpy())
            assert np.array_equal(gs, s) and np.array_equal(gq, q)
        gq, gs = _unpack_down(buf, off["w2"] + e * d * f, off["sc2"] + 4 * e * d, d, f)
        q, s = oracle.quantize_e4m3_columns(W2[e].float().numpy())
        assert np.array_equal(gs, s) and np.array_equal(gq, q)
    got = _unpack_up(buf, off["w13s"], off["sc13s"], None, d, fs)
    for (gq, gs), W in zip(got, (Ws[0][0], Ws[1][0])):
        q, s = oracle.quantize_e4m3_columns(W.float().numpy())
        assert np.array_equal(gs, s) and np.array_equal(gq, q)
    gq, gs = _unpack_down(buf, off["w2s"], off["sc2s"], d, fs)
    q, s = oracle.quantize_e4m3_columns(Ws[2][0].float().numpy())
    assert np.array_equal(gs, s) and np.array_equal(gq, q)


def test_fp8_grouped_ffn_tile_edges(cuda_device):
    E, d, f, fs = len(EDGE_COUNTS), 256, 256, 128
    T = sum(EDGE_COUNTS)
    cfg = B.config(T=T, d=d, E=E, f=f, k=1, n_shared=1, f_shared=fs, dtype="fp8w")
    g = torch.Generator(device="cpu").manual_seed(5)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).bfloat16()
    Ws = [(torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, fs, d, generator=g) / fs ** 0.5).bfloat16()]
    x = random_rows(T, d, seed=12, dtype=torch.bfloat16)
    idx = np.repeat(np.arange(E, dtype=np.int32), EDGE_COUNTS)[np.random.default_rng(8).permutation(T)]
    o_off, _, _, o_rows = oracle.dispatch_tc(idx.reshape(T, 1), E, -1)
    x_perm = x[torch.from_numpy(o_rows).long()]
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    off_d, xp_d, x_d = torch.from_numpy(o_off).to(dev), x_perm.to(dev), x.to(dev)
    Y = _np(layer.grouped_ffn(xp_d, off_d, x_d))
    H = torch.empty(T, f, dtype=torch.bfloat16, device=dev)
    Hs = torch.empty(T, fs, dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty(2 * T, d, dtype=torch.bfloat16, device=dev)
    B.moe_grouped_ffn_up(cfg, xp_d, off_d, layer.packed, x_d, H, Hs)
    B.moe_grouped_ffn_down(cfg, H, Hs, off_d, layer.packed, Y2)
    Y2 = _np(Y2)
    _check_device_error()
    xf = x_perm.float().numpy()
    ref = np.zeros((2 * T, d))
    for e in range(E):
        a, b = int(o_off[e]), int(o_off[e + 1])
        if b > a:
            ref[a:b] = oracle.expert_rows_fp8(xf[a:b], *_fp8_quant(W1[e], W3[e], W2[e]))
    ref[T:] = oracle.expert_rows_fp8(x.float().numpy(), *_fp8_quant(Ws[0][0], Ws[1][0], Ws[2][0]))
    for got in (Y, Y2):
        for e in range(E):
            a, b = int(o_off[e]), int(o_off[e + 1])
            if b > a:
                assert rel_err(got[a:b], ref[a:b]) <= TOL["bf16"], (e, b - a)
        assert rel_err(got[T:], ref[T:]) <= TOL["bf16"]


def _fp8_forward_ref(wl, inp, toks):
    """Oracle layer output for the tokens `toks` with the FP8-quantised experts:
    oracle routing and capacity dispatch, then per chosen expert the fp64 expert of
    the codes and scales, weighted, plus the merged shared expert.  One expert's
    quantised weights at a time."""
    T, E = wl.T, wl.E
    x = inp["x"].float().cpu().numpy()
    oi, ow, gap = oracle.route_tc(inp["x"], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                  wl.renorm, nthreads=NTH)
    cap = oracle.capacity(wl.capacity_factor, T, wl.k, wl.E)
    _, _, o_slot, _ = oracle.dispatch_tc(oi, E, cap)
    y = np.zeros((len(toks), wl.d))
    pos = {int(t): n for n, t in enumerate(toks)}
    for e in range(E):
        rows = [(pos[int(t)], j) for t in toks for j in range(wl.k) if oi[t, j] == e and o_slot[t, j] >= 0]
        if not rows:
            continue
        qs = _fp8_quant(inp["W1"][e].cpu(), inp["W3"][e].cpu(), inp["W2"][e].cpu())
        n_idx = np.array([r[0] for r in rows])
        out = oracle.expert_rows_fp8(x[toks[n_idx]], *qs)
        for (n, j), o in zip(rows, out):
            y[n] += ow[toks[n], j] * o
    if wl.n_shared:
        m1, m3, m2 = _merged_shared(inp["W1s"].cpu(), inp["W3s"].cpu(), inp["W2s"].cpu())
        y += oracle.expert_rows_fp8(x[toks], *_fp8_quant(m1, m3, m2))
    return y, oi, o_slot, cap


FP8_E2E = {
    "fp8_switch_drops": WORKLOADS["switch_top1_cap1.25"].with_(T=600, d=256, E=8, f=256, capacity_factor=0.8,
                                                                logit_offsets="normal_var0.5", dtype="fp8w",
                                                                name="fp8_switch_drops"),
    "fp8_sigmoid_shared": WORKLOADS["deepseek_v3"].with_(T=150, d=256, E=32, f=128, f_shared=128, dtype="fp8w",
                                                          name="fp8_sigmoid_shared"),
    "fp8_top2": WORKLOADS["mixtral_T256"].with_(T=333, d=512, f=384, dtype="fp8w", name="fp8_top2"),
    "fp8_switch_full": WORKLOADS["switch_top1_cap1.25"].with_(dtype="fp8w", name="fp8_switch_full"),
}


@pytest.mark.parametrize("name", list(FP8_E2E))
def test_fp8_forward(name, cuda_device):
    wl = FP8_E2E[name]
    inp = make_inputs(wl, cuda_device)
    cfg, layer = _layer(wl, inp)
    y = layer.forward(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"], out=_nan_out(layer))
    r_idx, _ = layer.route(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"])
    _check_device_error()
    T = wl.T
    toks = np.arange(T) if T <= 1000 else _sample_tokens(T, 96, T)
    ref, oi, o_slot, cap = _fp8_forward_ref(wl, inp, toks)
    gi = _np(r_idx)
    _, _, g_slot, _ = oracle.dispatch_tc(gi, wl.E, cap)   # the GPU's own choices, dispatched
    # tokens routed alike on both sides, with the same slots dropped
    keep = np.array([(gi[t] == oi[t]).all() and ((g_slot[t] >= 0) == (o_slot[t] >= 0)).all() for t in toks])
    got = _np(y)[toks]
    err = rel_err(got[keep], ref[keep])
    print(f"{name}: {int(keep.sum())} tokens compared, max|err|/max|ref| = {err:.3e}")
    assert keep.mean() > 0.95 and err <= TOL["bf16"]


def test_fp8_subnormal_codes_are_exact(cuda_device):
    # Down projection of one-hot rows: Y[h, n] = q2[h, n] * s2[n] exactly (one product,
    # rounded once to bf16).  Most of W2 is tiny next to its column maximum, so its
    # codes are E4M3 subnormals; a conversion that flushed them would give zeros.
    d, f = 256, 128
    cfg = B.config(T=f, d=d, E=1, f=f, k=1, dtype="fp8w")
    rng = np.random.default_rng(9)
    W2 = (rng.uniform(4.5e-6, 3.4e-5, (f, d)) * rng.choice([-1.0, 1.0], (f, d))).astype(np.float32)
    W2[0, :] = 1.0
    W2t = torch.from_numpy(W2).bfloat16()
    q, s = oracle.quantize_e4m3_columns(W2t.float().numpy())
    sub = (q != 0) & (np.abs(q) < 2.0 ** -6)
    assert sub.sum() > f * d // 2
    dev = cuda_device
    W1 = torch.zeros(1, d, f, dtype=torch.bfloat16, device=dev)
    layer = MoELayer(cfg, W1, W1, W2t.reshape(1, f, d).to(dev))
    H = torch.eye(f, dtype=torch.bfloat16, device=dev)
    off = torch.tensor([0, f], dtype=torch.int32, device=dev)
    Y = torch.empty(f, d, dtype=torch.bfloat16, device=dev)
    B.moe_grouped_ffn_down(cfg, H, None, off, layer.packed, Y)
    _check_device_error()
    ref = q * s.astype(np.float64)
    got = _np(Y)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8), np.abs(got - ref).max()
