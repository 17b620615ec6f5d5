"""The FP8 up projection (MOE_BF16_FP8UP) against the CPU oracle.

The up projection runs on E4M3 operands on the tensor cores: every activation row
quantised per token (s = amax / 448), W1 and W3 per output channel; H, W2 and Y
stay bf16.  The oracle computes the same layer in fp64 from the same codes and
scales (oracle.expert_rows_fp8up), so the bar is the bf16 one, max |err| <=
2e-2 * max |y_ref|; the packed codes and scales must equal the oracle's
quantiser bit for bit.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_gemm_b300 import binding as B
from mixture_experts_sparse_gemm_b300 import build as build_mod
from mixture_experts_sparse_gemm_b300.layer import MoELayer
from workloads import WORKLOADS, make_inputs, random_rows

pytestmark = pytest.mark.gpu

GAP = 1e-4
TOL = 2e-2
NTH = os.cpu_count() or 1
# segment sizes on both sides of the 16-row MMA step, of the 64-row limit of the
# M = 64 tiles (also as a second M tile: 192, 193) and of the 128-row M tile
EDGE_COUNTS = [1, 15, 16, 17, 63, 64, 65, 111, 112, 113, 127, 128, 129, 192, 193, 240, 0]


@pytest.fixture(scope="module", autouse=True)
def built(cuda_device):
    build_mod.build()
    B.lib()


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype != torch.int32 else t.cpu().numpy()


def rel_err(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def _check():
    torch.cuda.synchronize()
    B.moe_check_device_error()


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
    """Byte offsets of the FP8-up packed buffer: E4M3 up images, bf16 down images,
    then the up projection's scales (regions 1024-byte aligned, in order)."""
    sizes = [("w13", E * 2 * f * d), ("w2", E * d * f * 2), ("w13s", 2 * fs * d), ("w2s", d * fs * 2),
             ("sc13", 4 * E * 2 * f), ("sc2", 0), ("sc13s", 4 * 2 * fs), ("sc2s", 0)]
    off, o = {}, 0
    for name, n in sizes:
        off[name] = o
        o = (o + n + 1023) // 1024 * 1024
    return off


def _tiled_f8(p, i, BN, K):
    """Byte of (row p, column i) in the E4M3 tile images: BN x 128 tiles, N-tile then
    K-tile, 16-byte chunks of row r permuted by chunk ^ (r % 8)."""
    nb, r, kb, ch, w = p // BN, p % BN, i // 128, (i % 128) // 16, i % 16
    return ((nb * (K // 128) + kb) * BN + r) * 128 + (ch ^ (r % 8)) * 16 + w


def _tiled_bf16(p, i, BN, K):
    """Element of (row p, column i) in the bf16 tile images: BN x 64 tiles."""
    nb, r, kb, ch, w = p // BN, p % BN, i // 64, (i % 64) // 8, i % 8
    return ((nb * (K // 64) + kb) * BN + r) * 64 + (ch ^ (r % 8)) * 8 + w


def _unpack_up(buf, base, scbase, d, f, BN=256):
    """(codes as values [d][f], scales [f]) of W1 (m = 0) and W3 (m = 1); packed row of
    hidden column h = (h // 64) * 128 + m * 64 + h % 64."""
    out = []
    for m in (0, 1):
        h = np.arange(f)
        p = (h // 64) * 128 + m * 64 + h % 64
        I, H = np.meshgrid(np.arange(d), h, indexing="ij")
        q = E4M3[buf[base + _tiled_f8(p[H], I, BN, d)]]
        s = np.frombuffer(buf[scbase:scbase + 4 * 2 * f].tobytes(), np.float32)[p]
        out.append((q, s))
    return out


def _unpack_down_bf16(buf, base, d, f, BN=256):
    """W2 [f][d] (bf16 values) from its tile images of [d][f]."""
    words = buf[base:base + 2 * d * f].view(np.uint16)
    Hh, N = np.meshgrid(np.arange(f), np.arange(d), indexing="ij")
    bits = words[_tiled_bf16(N, Hh, BN, f)].astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def _weights(E, d, f, fs, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    W1 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W3 = (torch.randn(E, d, f, generator=g) / d ** 0.5).bfloat16()
    W2 = (torch.randn(E, f, d, generator=g) / f ** 0.5).bfloat16()
    Ws = [(torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, d, fs, generator=g) / d ** 0.5).bfloat16(),
          (torch.randn(1, fs, d, generator=g) / fs ** 0.5).bfloat16()]
    return W1, W3, W2, Ws


def test_fp8up_packing_is_exact(cuda_device):
    E, d, f, fs = 3, 256, 256, 128
    cfg = B.config(T=16, d=d, E=E, f=f, k=1, n_shared=1, f_shared=fs, dtype="fp8up")
    W1, W3, W2, Ws = _weights(E, d, f, fs, 99)
    W1[1, :, 5] = 0                                     # an all-zero channel: scale 0, codes 0
    W1[0, 7, 9] = 3.0e-7                                # a tiny weight on an E4M3 subnormal
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    torch.cuda.synchronize()
    buf = layer.packed.cpu().numpy()
    assert buf.size == B.moe_packed_weights_size(cfg)
    off = _packed_offsets(E, d, f, fs)
    for e in range(E):
        got = _unpack_up(buf, off["w13"] + e * 2 * f * d, off["sc13"] + 4 * e * 2 * f, d, f)
        for (gq, gs), W in zip(got, (W1[e], W3[e])):
            q, s = oracle.quantize_e4m3_columns(W.float().numpy())
            assert np.array_equal(gs, s) and np.array_equal(gq, q)
        assert np.array_equal(_unpack_down_bf16(buf, off["w2"] + e * d * f * 2, d, f), W2[e].double().numpy())
    got = _unpack_up(buf, off["w13s"], off["sc13s"], d, fs)
    for (gq, gs), W in zip(got, (Ws[0][0], Ws[1][0])):
        q, s = oracle.quantize_e4m3_columns(W.float().numpy())
        assert np.array_equal(gs, s) and np.array_equal(gq, q)
    assert np.array_equal(_unpack_down_bf16(buf, off["w2s"], d, fs), Ws[2][0].double().numpy())


def test_fp8up_grouped_ffn_tile_edges(cuda_device):
    """Segments of 1..240 rows and an empty one around the 64- and 128-row tile
    limits, plus a shared expert over all rows; every row compared.  An all-zero token row
    (scale 0) is among them."""
    E, d, f, fs = len(EDGE_COUNTS), 256, 256, 128
    T = sum(EDGE_COUNTS)
    cfg = B.config(T=T, d=d, E=E, f=f, k=1, n_shared=1, f_shared=fs, dtype="fp8up")
    W1, W3, W2, Ws = _weights(E, d, f, fs, 5)
    x = random_rows(T, d, seed=12, dtype=torch.bfloat16)
    x[7] = 0
    idx = np.repeat(np.arange(E, dtype=np.int32), EDGE_COUNTS)[np.random.default_rng(8).permutation(T)]
    o_off, _, _, o_rows = oracle.dispatch_tc(idx.reshape(T, 1), E, -1)
    x_perm = x[torch.from_numpy(o_rows).long()]
    dev = cuda_device
    layer = MoELayer(cfg, W1.to(dev), W3.to(dev), W2.to(dev), *(w.to(dev) for w in Ws))
    Y = _np(layer.grouped_ffn(x_perm.to(dev), torch.from_numpy(o_off).to(dev), x.to(dev)))
    _check()
    xf = x_perm.float().numpy()
    for e in range(E):
        a, b = int(o_off[e]), int(o_off[e + 1])
        if b > a:
            ref = oracle.expert_rows_fp8up(xf[a:b], W1[e].float().numpy(), W3[e].float().numpy(),
                                           W2[e].float().numpy())
            assert rel_err(Y[a:b], ref) <= TOL, (e, b - a)
    sref = oracle.expert_rows_fp8up(x.float().numpy(), Ws[0][0].float().numpy(), Ws[1][0].float().numpy(),
                                    Ws[2][0].float().numpy())
    assert rel_err(Y[T:], sref) <= TOL


def test_fp8up_halves_are_unsupported(cuda_device):
    cfg = B.config(T=8, d=256, E=2, f=128, k=1, dtype="fp8up")
    A = 0x10000
    assert B.lib().moe_grouped_ffn_up(B.ctypes.byref(cfg), A, A, A, None, A, None, None) == B.MOE_ERR_UNSUPPORTED
    assert B.lib().moe_grouped_ffn_down(B.ctypes.byref(cfg), A, None, A, A, A, None) == B.MOE_ERR_UNSUPPORTED


def _fp8up_forward_ref(wl, inp, toks, g_idx):
    """Oracle output of the FP8-up layer for the tokens `toks`: oracle routing (and
    capacity dispatch), then per chosen expert the fp64 expert of oracle.expert_rows_fp8up,
    weighted, plus the merged shared expert.  One expert's weights at a time.
    Returns (y, mask of the tokens that may be compared): tokens the GPU routed (and
    dropped) exactly as the oracle, or for Expert Choice tokens clear of every
    expert's selection boundary."""
    T, E = wl.T, wl.E
    x = inp["x"].float().cpu().numpy()
    y = np.zeros((len(toks), wl.d))
    pos = {int(t): n for n, t in enumerate(toks)}
    if wl.mode == "ec":
        ot, ow, gap, S = oracle.route_ec(inp["x"], inp["W_r"], wl.ec_capacity, inp["logit_offset"], nthreads=NTH,
                                         want_scores=True)
        pairs = {e: [(pos[int(t)], float(ow[e, r])) for r, t in enumerate(ot[e]) if int(t) in pos] for e in range(E)}
        bound = np.sort(S, axis=0)[::-1][wl.ec_capacity - 1]          # each expert's cap-th largest score
        near = (np.abs(S - bound[None, :]) < 1e-5).any(axis=1)
        ok = ~near[toks]
    else:
        oi, ow, gap = oracle.route_tc(inp["x"], inp["W_r"], wl.k, wl.gate, inp["logit_offset"], inp["sel_bias"],
                                      wl.renorm, nthreads=NTH)
        cap = oracle.capacity(wl.capacity_factor, T, wl.k, wl.E)
        _, _, o_slot, _ = oracle.dispatch_tc(oi, E, cap)
        _, _, g_slot, _ = oracle.dispatch_tc(g_idx, E, cap)   # the GPU's own choices, dispatched
        same = (g_idx == oi).all(axis=1) & ((g_slot >= 0) == (o_slot >= 0)).all(axis=1)
        pairs = {e: [] for e in range(E)}
        for t in toks:
            for j in range(wl.k):
                if o_slot[t, j] >= 0:
                    pairs[int(oi[t, j])].append((pos[int(t)], float(ow[t, j])))
        ok = same[toks]
    for e in range(E):
        if not pairs[e]:
            continue
        n_idx = np.array([p[0] for p in pairs[e]])
        out = oracle.expert_rows_fp8up(x[toks[n_idx]], inp["W1"][e].float().cpu().numpy(),
                                       inp["W3"][e].float().cpu().numpy(), inp["W2"][e].float().cpu().numpy())
        for (n, w), o in zip(pairs[e], out):
            y[n] += w * o
    if wl.n_shared:
        m1 = torch.cat(list(inp["W1s"].cpu()), dim=1).float().numpy()
        m3 = torch.cat(list(inp["W3s"].cpu()), dim=1).float().numpy()
        m2 = torch.cat(list(inp["W2s"].cpu()), dim=0).float().numpy()
        y += oracle.expert_rows_fp8up(x[toks], m1, m3, m2)
    return y, ok


FP8UP_E2E = {
    # one expert per token: the down tiles write y directly (gated), drops zeroed
    "fp8up_switch_drops": (WORKLOADS["switch_top1_cap1.25"].with_(T=600, d=256, E=8, f=256, capacity_factor=0.8,
                                                                  logit_offsets="normal_var0.5", dtype="fp8up",
                                                                  name="fp8up_switch_drops"), None),
    "fp8up_sigmoid_shared": (WORKLOADS["deepseek_v3"].with_(T=150, d=256, E=32, f=128, f_shared=128, dtype="fp8up",
                                                            name="fp8up_sigmoid_shared"), None),
    "fp8up_top2": (WORKLOADS["mixtral_T256"].with_(T=333, d=512, f=384, dtype="fp8up", name="fp8up_top2"), None),
    "fp8up_ec": (WORKLOADS["expert_choice_zipf"].with_(T=1000, d=256, E=16, f=128, ec_capacity=100, dtype="fp8up",
                                                       name="fp8up_ec"), None),
    "fp8up_switch_full": (WORKLOADS["switch_top1_cap1.25"].with_(dtype="fp8up", name="fp8up_switch_full"), 64),
    "fp8up_deepseek_full": (WORKLOADS["deepseek_v3"].with_(dtype="fp8up", name="fp8up_deepseek_full"), 8),
}


@pytest.mark.parametrize("name", list(FP8UP_E2E))
def test_fp8up_forward(name, cuda_device):
    wl, n_sample = FP8UP_E2E[name]
    inp = make_inputs(wl, cuda_device)
    cfg = B.config_from_workload(wl)
    layer = MoELayer(cfg, inp["W1"], inp["W3"], inp["W2"], inp.get("W1s"), inp.get("W3s"), inp.get("W2s"))
    out = torch.full((wl.T, wl.d), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    y = layer.forward(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"], out=out)
    g_idx = _np(layer.route(inp["x"], inp["W_r"], inp["logit_offset"], inp["sel_bias"])[0])
    _check()
    T = wl.T
    toks = np.arange(T) if n_sample is None else np.sort(np.random.default_rng(T).choice(T, n_sample, replace=False))
    ref, ok = _fp8up_forward_ref(wl, inp, toks, g_idx)
    got = _np(y)[toks]
    err = rel_err(got[ok], ref[ok])
    print(f"{name}: {int(ok.sum())} tokens compared, max|err|/max|ref| = {err:.3e}")
    assert ok.mean() > 0.9 and err <= TOL
    del layer
    torch.cuda.empty_cache()
