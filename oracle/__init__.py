"""CPU oracle for the sparsely-gated MoE SwiGLU FFN forward -- TEST INFRASTRUCTURE.

A thin ctypes binding over ``moe_oracle.c`` (plain C, fp64, one token at a time).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product library never loads it.

Every function takes numpy arrays holding the exact run-dtype values (fp32 arrays;
bf16 values are exact in fp32) and returns float64 results.  ``forward`` chains the
stages the way the layer does: route -> capacity-limited dispatch -> experts ->
gate-weighted combine (plus unweighted shared experts).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_moe.so")
_lock = threading.Lock()
_lib = None

GATE_SOFTMAX = 0
GATE_SIGMOID = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math: IEEE double throughout)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            ppf = ctypes.POINTER(f32p)
            c_int = ctypes.c_int
            lib.oracle_capacity.restype = ctypes.c_int64
            lib.oracle_capacity.argtypes = [ctypes.c_double, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
            lib.oracle_route_tc.argtypes = [c_int, c_int, c_int, c_int, f32p, f32p, f32p, c_int, f32p,
                                            c_int, i32p, f64p, f64p, f64p, c_int]
            lib.oracle_route_ec.argtypes = [c_int, c_int, c_int, c_int, f32p, f32p, f32p, i32p, f64p,
                                            f64p, f64p, c_int]
            lib.oracle_dispatch_tc.argtypes = [c_int, c_int, c_int, ctypes.c_int64, i32p, i32p, i32p,
                                               i32p, i32p]
            lib.oracle_swiglu_expert.restype = None
            lib.oracle_swiglu_expert.argtypes = [c_int, c_int, f32p, f32p, f32p, f32p, ctypes.c_double, f64p]
            lib.oracle_forward_tc.argtypes = [c_int, c_int, c_int, c_int, i32p, f32p, i32p, f64p, i32p,
                                              ppf, ppf, ppf, c_int, c_int, ppf, ppf, ppf, f64p, c_int]
            lib.oracle_forward_ec.argtypes = [c_int, c_int, c_int, c_int, c_int, i32p, f32p, i32p, f64p,
                                              ppf, ppf, ppf, c_int, c_int, ppf, ppf, ppf, f64p, c_int]
            lib.oracle_expert_rows.restype = None
            lib.oracle_expert_rows.argtypes = [c_int, c_int, c_int, f32p, f32p, f32p, f32p, f64p, f64p, c_int]
            lib.oracle_max_threads.restype = c_int
            _lib = lib
    return _lib


def _f32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (any dtype) -> exact fp32 values on the host
        a = a.detach().float().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _ptr_array(mats):
    """ctypes float** over a list of fp32 arrays (None entries allowed)."""
    f32p = ctypes.POINTER(ctypes.c_float)
    arr = (f32p * max(1, len(mats)))()
    for i, m in enumerate(mats):
        arr[i] = _ptr(m, ctypes.c_float) if m is not None else f32p()
    return arr


def max_threads() -> int:
    return _load().oracle_max_threads()


def capacity(C: float, T: int, k: int, E: int) -> int:
    """floor(C*T*k/E); -1 for no limit (C <= 0)."""
    return int(_load().oracle_capacity(float(C), int(T), int(k), int(E)))


def route_tc(x, W_r, k, gate="softmax", logit_offset=None, sel_bias=None, renorm=True,
             nthreads=1, want_scores=False):
    """Token-choice routing -> (topk_idx[T,k] int32, topk_w[T,k] f64, gap[T] f64[, scores[T,E]])."""
    x, W_r = _f32(x), _f32(W_r)
    lo, sb = _f32(logit_offset), _f32(sel_bias)
    T, d = x.shape
    E = W_r.shape[1]
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    gap = np.empty((T,), np.float64)
    sc = np.empty((T, E), np.float64) if want_scores else None
    rc = _load().oracle_route_tc(T, d, E, k, _ptr(x, ctypes.c_float), _ptr(W_r, ctypes.c_float),
                                 _ptr(lo, ctypes.c_float),
                                 GATE_SIGMOID if gate == "sigmoid" else GATE_SOFTMAX,
                                 _ptr(sb, ctypes.c_float), int(bool(renorm)),
                                 _ptr(idx, ctypes.c_int32), _ptr(w, ctypes.c_double),
                                 _ptr(gap, ctypes.c_double), _ptr(sc, ctypes.c_double), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_route_tc failed ({rc})")
    return (idx, w, gap, sc) if want_scores else (idx, w, gap)


def route_ec(x, W_r, cap, logit_offset=None, nthreads=1, want_scores=False):
    """Expert Choice routing -> (ec_tok[E,cap] int32, ec_w[E,cap] f64, gap[E] f64[, S[T,E]])."""
    x, W_r, lo = _f32(x), _f32(W_r), _f32(logit_offset)
    T, d = x.shape
    E = W_r.shape[1]
    tok = np.empty((E, cap), np.int32)
    w = np.empty((E, cap), np.float64)
    gap = np.empty((E,), np.float64)
    S = np.empty((T, E), np.float64) if want_scores else None
    rc = _load().oracle_route_ec(T, d, E, cap, _ptr(x, ctypes.c_float), _ptr(W_r, ctypes.c_float),
                                 _ptr(lo, ctypes.c_float), _ptr(tok, ctypes.c_int32),
                                 _ptr(w, ctypes.c_double), _ptr(gap, ctypes.c_double),
                                 _ptr(S, ctypes.c_double), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_route_ec failed ({rc})")
    return (tok, w, gap, S) if want_scores else (tok, w, gap)


def dispatch_tc(topk_idx, E, cap=-1):
    """Capacity-limited dispatch -> (off[E+1], cnt_raw[E], slot_of[T,k], row_token[A])."""
    idx = _i32(topk_idx)
    T, k = idx.shape
    off = np.empty(E + 1, np.int32)
    cnt = np.empty(E, np.int32)
    slot = np.empty((T, k), np.int32)
    row_token = np.full(T * k, -1, np.int32)
    rc = _load().oracle_dispatch_tc(T, k, E, int(cap), _ptr(idx, ctypes.c_int32), _ptr(off, ctypes.c_int32),
                                    _ptr(cnt, ctypes.c_int32), _ptr(slot, ctypes.c_int32),
                                    _ptr(row_token, ctypes.c_int32))
    if rc != 0:
        raise ValueError(f"oracle_dispatch_tc failed ({rc})")
    return off, cnt, slot, row_token[: off[E]].copy()


def dispatch_tc_affinity(topk_idx, topk_w, E, cap=-1):
    """Capacity-limited dispatch with the DeepSeek-V2 drop ("技术日报 2026-04-14" §5.2:
    over-capacity tokens dropped by descending affinity) -> (off, cnt_raw, slot_of,
    row_token) as dispatch_tc.  Expert e ranks its assignments (t, j) by weight
    topk_w[t, j], largest first, ties to the lower token, and keeps the first cap;
    the kept rows of a segment stay in ascending token order, segments in expert
    order.  Without a limit (cap < 0) this is dispatch_tc."""
    idx = np.asarray(topk_idx)
    w = np.asarray(topk_w, np.float32)
    if cap < 0:
        return dispatch_tc(idx, E, cap)
    T, k = idx.shape
    cnt = np.zeros(E, np.int32)
    for t in range(T):
        for j in range(k):
            cnt[idx[t, j]] += 1
    kept = np.zeros((T, k), bool)
    for e in range(E):
        cand = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        cand.sort(key=lambda tj: (-float(w[tj]), tj[0]))
        for t, j in cand[:cap]:
            kept[t, j] = True
    off = np.zeros(E + 1, np.int32)
    for e in range(E):
        off[e + 1] = off[e] + min(int(cnt[e]), cap)
    slot = np.full((T, k), -1, np.int32)
    row_token = np.full(int(off[E]), -1, np.int32)
    nxt = off[:E].copy()
    for t in range(T):                               # token order inside each segment
        for j in range(k):
            if kept[t, j]:
                e = idx[t, j]
                slot[t, j] = nxt[e]
                row_token[nxt[e]] = t
                nxt[e] += 1
    return off, cnt, slot, row_token


def swiglu_expert(x_row, W1, W3, W2, scale=1.0):
    """(SiLU(x W1) * (x W3)) W2 for one token, fp64."""
    x_row, W1, W3, W2 = _f32(x_row), _f32(W1), _f32(W3), _f32(W2)
    d, f = W1.shape
    out = np.zeros(d, np.float64)
    _load().oracle_swiglu_expert(d, f, _ptr(x_row, ctypes.c_float), _ptr(W1, ctypes.c_float),
                                 _ptr(W3, ctypes.c_float), _ptr(W2, ctypes.c_float), float(scale),
                                 _ptr(out, ctypes.c_double))
    return out


def _expert_mats(W, needed):
    """Per-expert fp32 host matrices for the experts in ``needed`` (others None)."""
    return [(_f32(W[e]) if e in needed else None) for e in range(W.shape[0])]


def expert_rows(X, W1, W3, W2, scale=None, nthreads=1):
    """out[r] = scale[r] * (SiLU(X[r] W1) * (X[r] W3)) W2 for every row of X, fp64."""
    X, W1, W3, W2 = _f32(X), _f32(W1), _f32(W3), _f32(W2)
    n, d = X.shape
    f = W1.shape[1]
    sc = None if scale is None else np.ascontiguousarray(scale, np.float64)
    out = np.empty((n, d), np.float64)
    if n:
        _load().oracle_expert_rows(d, f, n, _ptr(X, ctypes.c_float), _ptr(W1, ctypes.c_float),
                                   _ptr(W3, ctypes.c_float), _ptr(W2, ctypes.c_float),
                                   _ptr(sc, ctypes.c_double), _ptr(out, ctypes.c_double), nthreads)
    return out


# ------------------------------------------------------------------ FP8 (E4M3) expert weights
E4M3_MAX = 448.0   # largest finite E4M3 value: 1.75 * 2^8


def e4m3_round(x):
    """Round to the nearest FP8 E4M3 value, ties to even, saturating at +-448.

    E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities):
    normal values (1 + m/8) * 2^(e-7) for e = 1..15, subnormals (m/8) * 2^-6, so the
    spacing is 2^(E-3) inside the binade [2^E, 2^(E+1)) for E >= -6 and 2^-9 below
    2^-6.  The value is scaled by its spacing (exact in fp64, a power of two),
    rounded half to even, scaled back, then clamped to the largest finite value."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    _, ex = np.frexp(a[nz])                       # a = m * 2^ex, m in [0.5, 1): binade E = ex - 1
    E = np.maximum(ex.astype(np.float64) - 1.0, -6.0)
    spacing = np.ldexp(1.0, (E - 3.0).astype(np.int64))
    out[nz] = np.minimum(np.round(a[nz] / spacing) * spacing, E4M3_MAX)
    return np.copysign(out, x)


def quantize_e4m3_columns(W):
    """Per-output-channel E4M3 quantisation of W[K][N] (channel = column n, over
    its K inputs), as moe_pack_weights defines it in fp32: s_n = amax_n / 448,
    code = E4M3(w / s_n) (fp32 division, then round to nearest even, saturate);
    s_n = 0 and codes 0 for an all-zero column.  Returns (q [K][N] as the E4M3
    values in fp64, s [N] fp32)."""
    W = np.asarray(W, np.float32)
    amax = np.abs(W).max(axis=0)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    q = np.zeros(W.shape, np.float64)
    nzc = s > 0
    v = (W[:, nzc] / s[nzc]).astype(np.float32)   # fp32 division, round to nearest
    q[:, nzc] = e4m3_round(v)
    return q, s


def expert_rows_fp8(x, q1, s1, q3, s3, q2, s2):
    """SwiGLU expert with E4M3 weights q (values) and per-column fp32 scales s, in
    fp64: gate = (x q1) * s1, up = (x q3) * s3 per hidden column, h = SiLU(gate) * up,
    out = (h q2) * s2 per model column -- the expert of "lnwmold.com GPT-4 MoE
    article" §2.2 with W = q * s, the scale taken out of each column's sum."""
    x = np.asarray(x, np.float64)
    g = (x @ np.asarray(q1, np.float64)) * np.asarray(s1, np.float64)
    u = (x @ np.asarray(q3, np.float64)) * np.asarray(s3, np.float64)
    h = g / (1.0 + np.exp(-g)) * u
    return (h @ np.asarray(q2, np.float64)) * np.asarray(s2, np.float64)


def quantize_e4m3_rows(X):
    """Per-row (per-token) E4M3 quantisation of activations X[rows][K], as the
    MOE_BF16_FP8UP layer defines it in fp32: s_r = amax_r / 448, code = E4M3(x / s_r)
    (fp32 division, round to nearest even, saturate); s_r = 0 and codes 0 for an
    all-zero row.  A row of X is a column of X^T, so this is the channel quantiser
    applied to the transpose.  Returns (q [rows][K] as E4M3 values in fp64, s [rows] fp32)."""
    q, s = quantize_e4m3_columns(np.asarray(X, np.float32).T)
    return np.ascontiguousarray(q.T), s


def expert_rows_fp8up(x, W1, W3, W2):
    """SwiGLU expert whose up projection runs on E4M3 operands (MOE_BF16_FP8UP), in
    fp64: every row of x quantised per row (quantize_e4m3_rows: codes qx, scale sx),
    W1 and W3 per output column (quantize_e4m3_columns: q1, s1, q3, s3); then
    gate = (qx q1) * sx * s1, up = (qx q3) * sx * s3, h = SiLU(gate) * up, and the
    down projection h W2 with W2 as given -- the expert of "lnwmold.com GPT-4 MoE
    article" §2.2 with the scales taken out of each sum."""
    qx, sx = quantize_e4m3_rows(x)
    (q1, s1), (q3, s3) = quantize_e4m3_columns(W1), quantize_e4m3_columns(W3)
    sx = np.asarray(sx, np.float64)[:, None]
    g = (qx @ q1) * sx * np.asarray(s1, np.float64)
    u = (qx @ q3) * sx * np.asarray(s3, np.float64)
    h = g / (1.0 + np.exp(-g)) * u
    return h @ np.asarray(W2, np.float64)


def load_stats(topk_idx, cnt_raw, scores, expert_choice=False):
    """Load statistics of one routing, from the definitions of "技术日报 2026-04-14"
    §4.4 (token fraction, LIF, CV, router entropy) and §4.2 (the Switch auxiliary
    term N * sum_i f_i P_i and the DeepSeek V1 expert-level term sum_i f'_i P_i,
    both without their alpha).

    topk_idx: [T, k] (token choice) or ec_tok [E, cap]; cnt_raw: [E] assignments per
    expert before any drop; scores: [T, E] router scores (softmax probability or
    sigmoid score).  Returns (f [E], P [E], summary [5] = LIF, CV, entropy,
    switch_aux, expert_balance), all float64:
      f_i  = cnt_raw[i] / sum(cnt_raw)          (the page's token fraction, ideal 1/E)
      f1_i = share of tokens whose first choice is i (Switch's argmax p; EC: f_i)
      P_i  = mean over tokens of scores[:, i]
      LIF  = E * max_i f_i;  CV = std(f) / mean(f) with the population std
      entropy = -sum_i q_i ln q_i over q = P / sum(P), q_i = 0 terms omitted
      switch_aux = E * sum_i f1_i P_i;  expert_balance = sum_i (E f_i) P_i, which is
      the page's f'_i = N' / (K' T) * count_i with N' = E, K' T = sum(cnt_raw)
    """
    cnt = np.asarray(cnt_raw, np.float64)
    scores = np.asarray(scores, np.float64)
    T, E = scores.shape
    f = cnt / cnt.sum()
    if expert_choice:
        f1 = f.copy()
    else:
        first = np.asarray(topk_idx)[:, 0]
        f1 = np.zeros(E)
        for t in range(T):
            f1[first[t]] += 1.0
        f1 /= T
    P = scores.sum(axis=0) / T
    mean = f.mean()
    cv = np.sqrt(((f - mean) ** 2).mean()) / mean
    q = P / P.sum()
    ent = -sum(qi * np.log(qi) for qi in q if qi > 0.0)
    summary = np.array([E * f.max(), cv, ent, E * float((f1 * P).sum()), E * float((f * P).sum())])
    return f, P, summary


def combine_tc(Y, slot_of, topk_w, tokens=None, Y_shared=None):
    """Gate-weighted combine, token choice: y[t] = sum over kept slots j (in slot
    order) of topk_w[t, j] * Y[slot_of[t, j]], plus Y_shared[t] when given."""
    Y = np.asarray(Y, np.float64)
    slot = _i32(slot_of)
    w = np.asarray(topk_w, np.float64)
    T, k = slot.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    y = np.zeros((len(tokens), Y.shape[1]), np.float64)
    for n, t in enumerate(tokens):
        for j in range(k):
            if slot[t, j] >= 0:
                y[n] += w[t, j] * Y[slot[t, j]]
        if Y_shared is not None:
            y[n] += np.asarray(Y_shared[t], np.float64)
    return y


def combine_ec(Y, slot_of, ec_w, tokens=None, Y_shared=None):
    """Gate-weighted combine, Expert Choice: y[t] = sum over experts e (ascending)
    that took t of ec_w[row] * Y[row], row = slot_of[t, e]; plus Y_shared[t]."""
    Y = np.asarray(Y, np.float64)
    slot = _i32(slot_of)
    w = np.asarray(ec_w, np.float64).reshape(-1)
    T, E = slot.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    y = np.zeros((len(tokens), Y.shape[1]), np.float64)
    for n, t in enumerate(tokens):
        for e in range(E):
            r = slot[t, e]
            if r >= 0:
                y[n] += w[r] * Y[r]
        if Y_shared is not None:
            y[n] += np.asarray(Y_shared[t], np.float64)
    return y


def _shared_sum(x_rows, W1s, W3s, W2s, nthreads):
    out = None
    for s in range(W1s.shape[0]):
        o = expert_rows(x_rows, W1s[s], W3s[s], W2s[s], None, nthreads)
        out = o if out is None else out + o
    return out


def forward_tc_streamed(x, topk_idx, topk_w, slot_of, W1, W3, W2, tokens, W1s=None, W3s=None, W2s=None,
                        nthreads=1):
    """Same result as ``forward_tc``, bit for bit, but visits one expert at a time
    so only one expert's weights are on the host at once (large layers).

    For token t: y[t] = ((0 + c_0) + c_1) + ... over kept slots in slot order,
    c_j = topk_w[t, j] * E_{idx[t, j]}(x_t), then + each shared expert in order.
    """
    idx, slot = _i32(topk_idx), _i32(slot_of)
    w = np.ascontiguousarray(topk_w, np.float64)
    tok = np.asarray(tokens, np.int64)
    k = idx.shape[1]
    d = x.shape[1]
    contrib = {}
    by_expert = {}
    for n, t in enumerate(tok):
        for j in range(k):
            if slot[t, j] >= 0:
                by_expert.setdefault(int(idx[t, j]), []).append((n, j))
    for e, pairs in sorted(by_expert.items()):
        rows = np.stack([_f32(x[int(tok[n])]) for n, _ in pairs])
        sc = np.array([w[tok[n], j] for n, j in pairs], np.float64)
        out = expert_rows(rows, W1[e], W3[e], W2[e], sc, nthreads)
        for (n, j), o in zip(pairs, out):
            contrib[(n, j)] = o
    y = np.zeros((len(tok), d), np.float64)
    for n in range(len(tok)):
        for j in range(k):
            if (n, j) in contrib:
                y[n] = y[n] + contrib[(n, j)]
    if W1s is not None and W1s.shape[0] > 0:
        xs = np.stack([_f32(x[int(t)]) for t in tok])
        for s in range(W1s.shape[0]):
            y = y + expert_rows(xs, W1s[s], W3s[s], W2s[s], None, nthreads)
    return y


def forward_ec_streamed(x, ec_tok, ec_w, W1, W3, W2, tokens, W1s=None, W3s=None, W2s=None, nthreads=1):
    """Same result as ``forward_ec``, bit for bit, one expert at a time."""
    et = _i32(ec_tok)
    ew = np.ascontiguousarray(ec_w, np.float64)
    tok = np.asarray(tokens, np.int64)
    E, cap = et.shape
    d = x.shape[1]
    pos = {int(t): n for n, t in enumerate(tok)}
    contrib = {}
    for e in range(E):
        pairs = [(pos[int(t)], r) for r, t in enumerate(et[e]) if int(t) in pos]
        if not pairs:
            continue
        rows = np.stack([_f32(x[int(tok[n])]) for n, _ in pairs])
        sc = np.array([ew[e, r] for _, r in pairs], np.float64)
        out = expert_rows(rows, W1[e], W3[e], W2[e], sc, nthreads)
        for (n, _), o in zip(pairs, out):
            contrib.setdefault(n, []).append(o)   # experts visited in ascending order
    y = np.zeros((len(tok), d), np.float64)
    for n, parts in contrib.items():
        for o in parts:
            y[n] = y[n] + o
    if W1s is not None and W1s.shape[0] > 0:
        xs = np.stack([_f32(x[int(t)]) for t in tok])
        for s in range(W1s.shape[0]):
            y = y + expert_rows(xs, W1s[s], W3s[s], W2s[s], None, nthreads)
    return y


def forward_tc(x, topk_idx, topk_w, slot_of, W1, W3, W2, tokens, W1s=None, W3s=None, W2s=None,
               nthreads=1):
    """y[len(tokens), d] (f64) for token choice, given routing and dispatch results."""
    x = _f32(x)
    idx, slot = _i32(topk_idx), _i32(slot_of)
    w = np.ascontiguousarray(topk_w, np.float64)
    tok = _i32(np.asarray(tokens))
    T, k = idx.shape
    d = x.shape[1]
    E, _, f = W1.shape
    needed = set(int(e) for t in tok for j, e in enumerate(idx[t]) if slot[t, j] >= 0)
    m1, m3, m2 = _expert_mats(W1, needed), _expert_mats(W3, needed), _expert_mats(W2, needed)
    ns = 0 if W1s is None else W1s.shape[0]
    fs = 0 if W1s is None else W1s.shape[2]
    s1 = [_f32(W1s[s]) for s in range(ns)]
    s3 = [_f32(W3s[s]) for s in range(ns)]
    s2 = [_f32(W2s[s]) for s in range(ns)]
    y = np.zeros((len(tok), d), np.float64)
    _load().oracle_forward_tc(d, f, k, len(tok), _ptr(tok, ctypes.c_int32), _ptr(x, ctypes.c_float),
                              _ptr(idx, ctypes.c_int32), _ptr(w, ctypes.c_double),
                              _ptr(slot, ctypes.c_int32), _ptr_array(m1), _ptr_array(m3),
                              _ptr_array(m2), ns, fs, _ptr_array(s1), _ptr_array(s3), _ptr_array(s2),
                              _ptr(y, ctypes.c_double), nthreads)
    return y


def forward_ec(x, ec_tok, ec_w, W1, W3, W2, tokens, W1s=None, W3s=None, W2s=None, nthreads=1):
    """y[len(tokens), d] (f64) for Expert Choice, given the expert selections."""
    x = _f32(x)
    et = _i32(ec_tok)
    ew = np.ascontiguousarray(ec_w, np.float64)
    tok = _i32(np.asarray(tokens))
    E, cap = et.shape
    d = x.shape[1]
    f = W1.shape[2]
    tokset = set(int(t) for t in tok)
    needed = set(e for e in range(E) if tokset.intersection(et[e].tolist()))
    m1, m3, m2 = _expert_mats(W1, needed), _expert_mats(W3, needed), _expert_mats(W2, needed)
    ns = 0 if W1s is None else W1s.shape[0]
    fs = 0 if W1s is None else W1s.shape[2]
    s1 = [_f32(W1s[s]) for s in range(ns)]
    s3 = [_f32(W3s[s]) for s in range(ns)]
    s2 = [_f32(W2s[s]) for s in range(ns)]
    y = np.zeros((len(tok), d), np.float64)
    _load().oracle_forward_ec(d, f, E, cap, len(tok), _ptr(tok, ctypes.c_int32), _ptr(x, ctypes.c_float),
                              _ptr(et, ctypes.c_int32), _ptr(ew, ctypes.c_double), _ptr_array(m1),
                              _ptr_array(m3), _ptr_array(m2), ns, fs, _ptr_array(s1), _ptr_array(s3),
                              _ptr_array(s2), _ptr(y, ctypes.c_double), nthreads)
    return y


def forward(inp: dict, wl, tokens=None, nthreads=1):
    """The whole layer for ``tokens`` (default: all) of a workload's inputs.

    Routing and dispatch always run over all T tokens (the capacity drop depends on
    the global token order); the experts and the combine run for ``tokens`` only.
    Returns a dict with y[len(tokens), d] and every intermediate the stages produce.
    """
    x = inp["x"]
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    res = {"tokens": tokens}
    if wl.mode == "ec":
        ec_tok, ec_w, gap, S = route_ec(x, inp["W_r"], wl.ec_capacity, inp.get("logit_offset"),
                                        nthreads=nthreads, want_scores=True)
        res.update(ec_tok=ec_tok, ec_w=ec_w, gap=gap, S=S)
        res["y"] = forward_ec_streamed(x, ec_tok, ec_w, inp["W1"], inp["W3"], inp["W2"], tokens,
                              inp.get("W1s"), inp.get("W3s"), inp.get("W2s"), nthreads=nthreads)
        return res
    idx, w, gap, sc = route_tc(x, inp["W_r"], wl.k, wl.gate, inp.get("logit_offset"), inp.get("sel_bias"),
                               wl.renorm, nthreads=nthreads, want_scores=True)
    cap = capacity(wl.capacity_factor, T, wl.k, wl.E)
    off, cnt_raw, slot_of, row_token = dispatch_tc(idx, wl.E, cap)
    res.update(topk_idx=idx, topk_w=w, gap=gap, scores=sc, cap=cap, off=off, cnt_raw=cnt_raw,
               slot_of=slot_of, row_token=row_token)
    res["y"] = forward_tc_streamed(x, idx, w, slot_of, inp["W1"], inp["W3"], inp["W2"], tokens,
                          inp.get("W1s"), inp.get("W3s"), inp.get("W2s"), nthreads=nthreads)
    return res
