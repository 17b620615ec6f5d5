"""Pins for the CPU oracle: checks against facts other than the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong tie-break or drop order) fails:
brute-force enumeration on tiny inputs, closed forms printed on the pages, special
cases that reduce to library routines (scipy softmax / expit, numpy matmul), and
invariants that characterise the result uniquely.
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(1000 + seed)


def _onehot_x(T, d):
    x = np.zeros((T, d), np.float32)
    x[np.arange(T), np.arange(T) % d] = 1.0
    return x


def _silu(z):
    return z * expit(z)


def _dense_swiglu(x, W1, W3, W2):
    """Textbook matrix form, fp64: (SiLU(x W1) * (x W3)) W2."""
    x = x.astype(np.float64)
    return (_silu(x @ W1.astype(np.float64)) * (x @ W3.astype(np.float64))) @ W2.astype(np.float64)


# --------------------------------------------------------------------------- capacity

def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split('"')[0].split())
    return rows


def test_capacity_printed_examples():
    rows = _golden_rows("capacity.txt")
    assert rows
    for C, T, k, E, want in rows:
        assert oracle.capacity(float(C), int(T), int(k), int(E)) == int(want)


def test_capacity_no_limit_and_floor():
    assert oracle.capacity(0.0, 100, 2, 8) == -1
    assert oracle.capacity(-1.0, 100, 2, 8) == -1
    assert oracle.capacity(1.0, 10, 1, 3) == 3          # floor(10/3)
    assert oracle.capacity(2.0, 7, 2, 4) == 7           # floor(28/4)


# --------------------------------------------------------------------------- top-k selection

def _integer_router(T, d, E, seed, lo=-3, hi=4):
    """One-hot tokens over an integer W_r: logits are exact integers with many ties."""
    r = _rng(seed)
    Wr = r.integers(lo, hi, size=(d, E)).astype(np.float32)
    return _onehot_x(T, d), Wr


def _brute_topk(keys, k):
    """Best k-subset by enumeration: max key sum, then lexicographically smallest."""
    best, best_sum = None, None
    for sub in itertools.combinations(range(len(keys)), k):
        s = sum(keys[e] for e in sub)
        if best is None or s > best_sum + 1e-12:
            best, best_sum = sub, s
    return sorted(best, key=lambda e: (-keys[e], e))


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (6, 3), (8, 2), (8, 3), (8, 8)])
def test_topk_softmax_matches_bruteforce(E, k):
    T, d = 48, 48
    x, Wr = _integer_router(T, d, E, seed=E * 10 + k)
    idx, w, gap = oracle.route_tc(x, Wr, k, "softmax", renorm=True)
    for t in range(T):
        u = Wr[t % d].astype(np.float64)          # softmax is monotone in the logits
        assert list(idx[t]) == _brute_topk(list(u), k), t


@pytest.mark.parametrize("E,k", [(5, 2), (8, 3)])
def test_topk_sigmoid_bias_matches_bruteforce(E, k):
    T, d = 40, 40
    x, Wr = _integer_router(T, d, E, seed=77 + E)
    b = (_rng(5).integers(-2, 3, size=E) * 0.25).astype(np.float32)
    idx, w, gap = oracle.route_tc(x, Wr, k, "sigmoid", sel_bias=b, renorm=True)
    for t in range(T):
        u = Wr[t % d].astype(np.float64)
        keys = list(expit(u) + b.astype(np.float64))
        want = _brute_topk(keys, k)
        assert list(idx[t]) == want, t
        s = expit(u[want])
        np.testing.assert_allclose(w[t], s / s.sum(), rtol=1e-13)   # weights ignore the bias


def test_ties_go_to_lowest_index():
    E, k, T, d = 8, 3, 4, 4
    x = _onehot_x(T, d)
    Wr = np.zeros((d, E), np.float32)                 # all logits equal
    idx, w, gap = oracle.route_tc(x, Wr, k, "softmax", renorm=True)
    assert (idx == np.array([0, 1, 2], np.int32)).all()
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-14)
    assert (gap == 0.0).all()
    Wr[:, 5] = 1.0                                      # one clear winner, then ties
    idx, _, _ = oracle.route_tc(x, Wr, k, "softmax")
    assert (idx == np.array([5, 0, 1], np.int32)).all()


# --------------------------------------------------------------------------- gate weights

def test_switch_top1_weight_is_softmax_max():
    T, d, E = 64, 32, 16
    r = _rng(3)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = (r.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    idx, w, gap = oracle.route_tc(x, Wr, 1, "softmax", renorm=False)
    p = softmax(x.astype(np.float64) @ Wr.astype(np.float64), axis=1)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(p, axis=1))
    np.testing.assert_allclose(w[:, 0], p.max(axis=1), rtol=1e-12)


def test_top2_renorm_is_sigmoid_of_logit_gap():
    # renormalised top-2 softmax weights: w0 = e^{u0} / (e^{u0} + e^{u1}) = expit(u0 - u1)
    T, d, E = 64, 32, 8
    r = _rng(4)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = (r.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    off = r.standard_normal(E).astype(np.float32)
    idx, w, gap = oracle.route_tc(x, Wr, 2, "softmax", logit_offset=off, renorm=True)
    u = x.astype(np.float64) @ Wr.astype(np.float64) + off
    u0 = u[np.arange(T), idx[:, 0]]
    u1 = u[np.arange(T), idx[:, 1]]
    np.testing.assert_allclose(w[:, 0], expit(u0 - u1), rtol=1e-12)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert (u0 >= u1).all()


def test_logit_offset_shift_invariance_and_renorm_sum():
    T, d, E, k = 50, 24, 12, 3
    r = _rng(6)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = (r.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    off = (np.round(r.standard_normal(E) * 1024) / 1024).astype(np.float32)   # +2 stays exact
    i1, w1, _ = oracle.route_tc(x, Wr, k, "softmax", logit_offset=off, renorm=True)
    i2, w2, _ = oracle.route_tc(x, Wr, k, "softmax", logit_offset=off + np.float32(2.0), renorm=True)
    np.testing.assert_array_equal(i1, i2)
    np.testing.assert_allclose(w1, w2, rtol=1e-12)
    np.testing.assert_allclose(w1.sum(axis=1), 1.0, atol=1e-12)
    # an offset changes the choice: a huge offset on expert 7 puts it first everywhere
    off2 = off.copy()
    off2[7] = 50.0
    i3, _, _ = oracle.route_tc(x, Wr, k, "softmax", logit_offset=off2)
    assert (i3[:, 0] == 7).all()


def test_selection_bias_forces_choice_but_not_weight():
    T, d, E, k = 30, 20, 10, 2
    r = _rng(8)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = (r.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    b = np.zeros(E, np.float32)
    b[3] = 5.0
    idx, w, _ = oracle.route_tc(x, Wr, k, "sigmoid", sel_bias=b, renorm=False)
    s = expit(x.astype(np.float64) @ Wr.astype(np.float64))
    assert (idx[:, 0] == 3).all()
    np.testing.assert_allclose(w[:, 0], s[:, 3], rtol=1e-13)   # raw unbiased score


# --------------------------------------------------------------------------- expert FFN

def test_swiglu_unit_values_are_silu():
    d, f = 4, 6
    a = np.array([-3.0, -0.5, 0.0, 0.25, 1.0, 4.0])
    W1 = np.zeros((d, f), np.float32)
    W1[0] = a
    W3 = np.zeros((d, f), np.float32)
    W3[0] = 1.0
    W2 = np.zeros((f, d), np.float32)
    W2[np.arange(d), np.arange(d)] = 1.0               # h_c for c < d copied to out_c
    x = np.zeros(d, np.float32)
    x[0] = 1.0
    out = oracle.swiglu_expert(x, W1, W3, W2)
    np.testing.assert_allclose(out, _silu(a[:d]), rtol=1e-14, atol=1e-300)


def test_swiglu_matches_dense_matrix_form_and_linearity():
    d, f = 24, 40
    r = _rng(9)
    x = r.standard_normal((3, d)).astype(np.float32)
    W1 = (r.standard_normal((d, f)) / math.sqrt(d)).astype(np.float32)
    W3 = (r.standard_normal((d, f)) / math.sqrt(d)).astype(np.float32)
    W2 = (r.standard_normal((f, d)) / math.sqrt(f)).astype(np.float32)
    ref = _dense_swiglu(x, W1, W3, W2)
    for t in range(3):
        np.testing.assert_allclose(oracle.swiglu_expert(x[t], W1, W3, W2), ref[t], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(oracle.swiglu_expert(x[t], W1, W3, 2 * W2),
                                   2 * oracle.swiglu_expert(x[t], W1, W3, W2), rtol=1e-13)
        assert not oracle.swiglu_expert(x[t], np.zeros_like(W1), W3, W2).any()   # SiLU(0) = 0
        # swapping W1 and W3 is NOT a symmetry (the gate is SiLU'd): a transposed role fails here
        assert np.abs(oracle.swiglu_expert(x[t], W3, W1, W2) - ref[t]).max() > 1e-3


# --------------------------------------------------------------------------- whole layer

def _layer_inputs(T, d, E, f, seed):
    r = _rng(seed)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = (r.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    W1 = (r.standard_normal((E, d, f)) / math.sqrt(d)).astype(np.float32)
    W3 = (r.standard_normal((E, d, f)) / math.sqrt(d)).astype(np.float32)
    W2 = (r.standard_normal((E, f, d)) / math.sqrt(f)).astype(np.float32)
    return x, Wr, W1, W3, W2


def test_single_expert_is_dense_swiglu():
    T, d, f = 20, 16, 32
    x, Wr, W1, W3, W2 = _layer_inputs(T, d, 1, f, seed=11)
    idx, w, _ = oracle.route_tc(x, Wr, 1, "softmax", renorm=False)
    np.testing.assert_allclose(w, 1.0, rtol=0, atol=0)
    off, cnt, slot, rows = oracle.dispatch_tc(idx, 1, -1)
    y = oracle.forward_tc(x, idx, w, slot, W1, W3, W2, np.arange(T))
    np.testing.assert_allclose(y, _dense_swiglu(x, W1[0], W3[0], W2[0]), rtol=1e-11, atol=1e-12)


def test_k_equals_E_is_full_softmax_mixture():
    T, d, E, f = 12, 16, 4, 24
    x, Wr, W1, W3, W2 = _layer_inputs(T, d, E, f, seed=12)
    for renorm in (True, False):
        idx, w, _ = oracle.route_tc(x, Wr, E, "softmax", renorm=renorm)
        off, cnt, slot, rows = oracle.dispatch_tc(idx, E, -1)
        y = oracle.forward_tc(x, idx, w, slot, W1, W3, W2, np.arange(T))
        p = softmax(x.astype(np.float64) @ Wr.astype(np.float64), axis=1)
        ref = sum(p[:, [e]] * _dense_swiglu(x, W1[e], W3[e], W2[e]) for e in range(E))
        np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_shared_experts_add_unweighted_and_drops_add_nothing():
    T, d, E, f, fs = 16, 8, 4, 12, 10
    x, Wr, W1, W3, W2 = _layer_inputs(T, d, E, f, seed=13)
    r = _rng(14)
    W1s = r.standard_normal((2, d, fs)).astype(np.float32)
    W3s = r.standard_normal((2, d, fs)).astype(np.float32)
    W2s = r.standard_normal((2, fs, d)).astype(np.float32)
    idx, w, _ = oracle.route_tc(x, Wr, 2, "softmax")
    cap = 3
    off, cnt, slot, rows = oracle.dispatch_tc(idx, E, cap)
    assert (slot < 0).any()
    y = oracle.forward_tc(x, idx, w, slot, W1, W3, W2, np.arange(T), W1s, W3s, W2s)
    ref = sum(_dense_swiglu(x, W1s[s], W3s[s], W2s[s]) for s in range(2))
    for t in range(T):
        for j in range(2):
            if slot[t, j] >= 0:
                e = idx[t, j]
                ref[t] += w[t, j] * _dense_swiglu(x[t:t + 1], W1[e], W3[e], W2[e])[0]
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-11)


# --------------------------------------------------------------------------- dispatch

def _check_dispatch(idx, E, cap, off, cnt_raw, slot, rows):
    T, k = idx.shape
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(cnt_raw, np.bincount(flat, minlength=E))
    kept_n = np.minimum(cnt_raw, cap) if cap >= 0 else cnt_raw
    np.testing.assert_array_equal(np.diff(off), kept_n)
    assert off[0] == 0
    s = slot.reshape(-1)
    assert (s >= 0).sum() == off[-1] == T * k - (s < 0).sum()
    kept = np.sort(s[s >= 0])
    np.testing.assert_array_equal(kept, np.arange(off[-1]))          # bijection onto rows
    for e in range(E):
        pos = np.nonzero(flat == e)[0]                                # (t, j) order
        sl = s[pos]
        n_keep = kept_n[e]
        assert (sl[:n_keep] >= 0).all() and (sl[n_keep:] < 0).all()  # first cap kept, rest dropped
        np.testing.assert_array_equal(sl[:n_keep], off[e] + np.arange(n_keep))
    for i in np.nonzero(s >= 0)[0]:
        assert rows[s[i]] == i // k


@pytest.mark.parametrize("T,E,k,cap,skew", [(200, 8, 2, -1, 0.0), (300, 8, 2, 40, 1.5),
                                            (257, 16, 1, 10, 2.0), (64, 4, 3, 0, 0.0),
                                            (64, 4, 3, 1000, 0.5), (1, 3, 2, 1, 0.0)])
def test_dispatch_invariants(T, E, k, cap, skew):
    r = _rng(T + E + k)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    p /= p.sum()
    idx = np.stack([r.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    off, cnt_raw, slot, rows = oracle.dispatch_tc(idx, E, cap)
    _check_dispatch(idx, E, cap, off, cnt_raw, slot, rows)


def test_dispatch_printed_capacity_drop_order():
    # 15 tokens pick one expert whose capacity is 10 (capacity example of the GPT-4
    # article, §3.2): the first 10 in token order are kept, the last 5 dropped
    idx = np.zeros((15, 1), np.int32)
    cap = oracle.capacity(1.25, 1024, 1, 128)
    off, cnt_raw, slot, rows = oracle.dispatch_tc(idx, 128, cap)
    assert cap == 10 and cnt_raw[0] == 15 and off[1] == 10 and off[-1] == 10
    np.testing.assert_array_equal(slot[:, 0], list(range(10)) + [-1] * 5)


# --------------------------------------------------------------------------- expert choice

def test_expert_choice_selection():
    T, d, E, cap = 96, 16, 6, 20
    r = _rng(20)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = (r.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    off = r.standard_normal(E).astype(np.float32)
    tok, w, gap, S = oracle.route_ec(x, Wr, cap, off, want_scores=True)
    ref_S = softmax(x.astype(np.float64) @ Wr.astype(np.float64) + off, axis=1)
    np.testing.assert_allclose(S, ref_S, rtol=1e-12)
    np.testing.assert_allclose(S.sum(axis=1), 1.0, atol=1e-13)
    for e in range(E):
        assert tok.shape[1] == cap                                   # exactly cap per expert
        assert (np.diff(tok[e]) > 0).all()                           # ascending, distinct
        want = np.sort(np.argsort(-ref_S[:, e], kind="stable")[:cap])
        np.testing.assert_array_equal(tok[e], want)
        np.testing.assert_allclose(w[e], ref_S[tok[e], e], rtol=1e-12)
        srt = np.sort(ref_S[:, e])[::-1]
        np.testing.assert_allclose(gap[e], srt[cap - 1] - srt[cap], rtol=1e-9, atol=1e-15)


def test_expert_choice_ties_take_lower_tokens_and_layer_sum():
    T, d, E, cap, f = 10, 4, 3, 4, 6
    x = np.ones((T, d), np.float32)                                  # identical tokens: all tie
    Wr = _rng(21).standard_normal((d, E)).astype(np.float32)
    tok, w, gap = oracle.route_ec(x, Wr, cap)
    np.testing.assert_array_equal(tok, np.tile(np.arange(cap), (E, 1)))
    assert (gap == 0).all()
    r = _rng(22)
    x = r.standard_normal((T, d)).astype(np.float32)
    W1 = r.standard_normal((E, d, f)).astype(np.float32)
    W3 = r.standard_normal((E, d, f)).astype(np.float32)
    W2 = r.standard_normal((E, f, d)).astype(np.float32)
    tok, w, gap, S = oracle.route_ec(x, Wr, cap, want_scores=True)
    y = oracle.forward_ec(x, tok, w, W1, W3, W2, np.arange(T))
    ref = np.zeros((T, d))
    for e in range(E):
        for t in tok[e]:
            ref[t] += S[t, e] * _dense_swiglu(x[t:t + 1], W1[e], W3[e], W2[e])[0]
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-11)
    untaken = sorted(set(range(T)) - set(tok.reshape(-1).tolist()))
    assert all(not y[t].any() for t in untaken)                      # 0 experts -> zero output


def test_threads_do_not_change_results():
    T, d, E = 300, 32, 16
    r = _rng(30)
    x = r.standard_normal((T, d)).astype(np.float32)
    Wr = r.standard_normal((d, E)).astype(np.float32)
    a = oracle.route_tc(x, Wr, 4, "sigmoid", nthreads=1)
    b = oracle.route_tc(x, Wr, 4, "sigmoid", nthreads=4)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


# --------------------------------------------------------------------------- streamed forms and combine

def test_streamed_forward_is_bitwise_equal_to_direct():
    T, d, E, f = 40, 16, 6, 24
    x, Wr, W1, W3, W2 = _layer_inputs(T, d, E, f, seed=40)
    r = _rng(41)
    W1s = r.standard_normal((2, d, 8)).astype(np.float32)
    W3s = r.standard_normal((2, d, 8)).astype(np.float32)
    W2s = r.standard_normal((2, 8, d)).astype(np.float32)
    idx, w, _ = oracle.route_tc(x, Wr, 3, "sigmoid", renorm=True)
    off, cnt, slot, rows = oracle.dispatch_tc(idx, E, 15)
    toks = np.array([0, 5, 7, 39, 12], np.int32)
    a = oracle.forward_tc(x, idx, w, slot, W1, W3, W2, toks, W1s, W3s, W2s, nthreads=3)
    b = oracle.forward_tc_streamed(x, idx, w, slot, W1, W3, W2, toks, W1s, W3s, W2s, nthreads=2)
    np.testing.assert_array_equal(a, b)
    tok, ew, gap = oracle.route_ec(x, Wr, 9)
    a = oracle.forward_ec(x, tok, ew, W1, W3, W2, toks, W1s, W3s, W2s)
    b = oracle.forward_ec_streamed(x, tok, ew, W1, W3, W2, toks, W1s, W3s, W2s, nthreads=4)
    np.testing.assert_array_equal(a, b)


def test_combine_definitions():
    T, k, d, E = 6, 2, 5, 4
    r = _rng(50)
    Y = r.standard_normal((T * k + T, d))
    slot = np.array([[0, 1], [2, -1], [3, 4], [-1, -1], [5, 6], [7, 8]], np.int32)
    w = np.zeros((T, k))
    w[0, 0] = 1.0                                          # one-hot weight picks a row
    y = oracle.combine_tc(Y, slot, w)
    np.testing.assert_array_equal(y[0], Y[0])
    assert not y[1:].any()
    w = r.random((T, k))
    ys = oracle.combine_tc(Y, slot, w, Y_shared=Y[T * k:])
    np.testing.assert_allclose(ys[3], Y[T * k + 3])        # all slots dropped: shared part only
    np.testing.assert_allclose(ys[1], w[1, 0] * Y[2] + Y[T * k + 1])
    y2 = oracle.combine_tc(2 * Y, slot, w)
    np.testing.assert_allclose(y2, 2 * oracle.combine_tc(Y, slot, w))   # linear in Y
    # expert choice: slot_of[t, e] = row, weight of a row = ec_w flat at that row
    cap = 2
    ec_tok = np.array([[0, 3], [1, 3], [2, 5], [0, 4]], np.int32)
    ec_w = r.random((E, cap))
    slot_ec = -np.ones((T, E), np.int32)
    for e in range(E):
        for rr, t in enumerate(ec_tok[e]):
            slot_ec[t, e] = e * cap + rr
    yec = oracle.combine_ec(Y, slot_ec, ec_w)
    np.testing.assert_allclose(yec[3], ec_w[0, 1] * Y[1] + ec_w[1, 1] * Y[3])
    np.testing.assert_allclose(yec[0], ec_w[0, 0] * Y[0] + ec_w[3, 0] * Y[6])


def test_forward_equals_combine_of_expert_rows():
    # the layer is the combine of per-row expert outputs: forward == combine(E(x_perm))
    T, d, E, f, k = 30, 16, 5, 20, 2
    x, Wr, W1, W3, W2 = _layer_inputs(T, d, E, f, seed=60)
    idx, w, _ = oracle.route_tc(x, Wr, k, "softmax", renorm=True)
    off, cnt, slot, row_token = oracle.dispatch_tc(idx, E, 10)
    Y = np.zeros((T * k, d))
    for e in range(E):
        rows = row_token[off[e]:off[e + 1]]
        Y[off[e]:off[e + 1]] = oracle.expert_rows(x[rows], W1[e], W3[e], W2[e])
    np.testing.assert_allclose(oracle.combine_tc(Y, slot, w), oracle.forward_tc(x, idx, w, slot, W1, W3, W2, np.arange(T)),
                               rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ load statistics
# "技术日报 2026-04-14" §4.4 states the balanced and collapsed values of the
# diagnostics (token fraction 1/E, LIF = 1 balanced and = E collapsed, CV = 0
# balanced, entropy largest for the uniform distribution); §4.2 states that the
# Switch term is optimal at f_i = P_i = 1/N, where N * sum f_i P_i = 1.

def test_load_stats_balanced_routing():
    E, T, k = 8, 64, 2
    idx = np.stack([np.arange(T) % E, (np.arange(T) + 3) % E], axis=1)
    cnt = np.bincount(idx.ravel(), minlength=E)
    f, P, s = oracle.load_stats(idx, cnt, np.full((T, E), 1.0 / E))
    assert np.allclose(f, 1.0 / E, rtol=0, atol=1e-15) and np.allclose(P, 1.0 / E, rtol=0, atol=1e-15)
    assert s[0] == pytest.approx(1.0, abs=1e-14) and s[1] == pytest.approx(0.0, abs=1e-14)
    assert s[2] == pytest.approx(np.log(E), abs=1e-14)
    assert s[3] == pytest.approx(1.0, abs=1e-14) and s[4] == pytest.approx(1.0, abs=1e-14)


@pytest.mark.parametrize("E", [2, 8, 64, 256])
def test_load_stats_collapsed_routing(E):
    T = 50
    idx = np.zeros((T, 1), np.int64)
    cnt = np.bincount(idx.ravel(), minlength=E)
    scores = np.zeros((T, E))
    scores[:, 0] = 1.0
    f, P, s = oracle.load_stats(idx, cnt, scores)
    # f = (1, 0, ..., 0): population std sqrt(E - 1) / E around the mean 1 / E
    assert s[0] == pytest.approx(E, rel=1e-15)
    assert s[1] == pytest.approx(np.sqrt(E - 1.0), rel=1e-14)
    assert s[2] == pytest.approx(0.0, abs=1e-15)
    assert s[3] == pytest.approx(E, rel=1e-15) and s[4] == pytest.approx(E, rel=1e-15)


def test_load_stats_hand_examples():
    # k = 1, E = 2: f = f1 = (3/4, 1/4), P = (0.6, 0.4)
    idx = np.array([[0], [0], [0], [1]])
    scores = np.array([[0.9, 0.1], [0.7, 0.3], [0.5, 0.5], [0.3, 0.7]])
    f, P, s = oracle.load_stats(idx, np.array([3, 1]), scores)
    assert np.allclose(f, [0.75, 0.25], rtol=0, atol=1e-15) and np.allclose(P, [0.6, 0.4], rtol=0, atol=1e-15)
    assert s[0] == pytest.approx(1.5) and s[1] == pytest.approx(0.5)          # std 0.25 / mean 0.5
    assert s[2] == pytest.approx(-(0.6 * np.log(0.6) + 0.4 * np.log(0.4)), rel=1e-14)
    assert s[3] == pytest.approx(2 * (0.75 * 0.6 + 0.25 * 0.4)) and s[4] == pytest.approx(1.1)
    # k = 2, E = 3: first choices all expert 0, assignments (2, 1, 1)
    idx = np.array([[0, 1], [0, 2]])
    scores = np.array([[0.5, 0.3, 0.2], [0.6, 0.1, 0.3]])
    f, P, s = oracle.load_stats(idx, np.array([2, 1, 1]), scores)
    assert np.allclose(P, [0.55, 0.2, 0.25], rtol=0, atol=1e-15)
    assert s[3] == pytest.approx(3 * 0.55, rel=1e-14)                          # f1 = (1, 0, 0)
    assert s[4] == pytest.approx(3 * (0.5 * 0.55 + 0.25 * 0.2 + 0.25 * 0.25), rel=1e-14)
    assert s[3] != pytest.approx(s[4])


def test_load_stats_entropy_matches_scipy():
    from scipy.stats import entropy
    rng = np.random.default_rng(5)
    for E in (4, 64, 256):
        scores = rng.random((300, E)) ** 3
        idx = np.argsort(-scores, axis=1, kind="stable")[:, :2]
        cnt = np.bincount(idx.ravel(), minlength=E)
        _, P, s = oracle.load_stats(idx, cnt, scores)
        assert s[2] == pytest.approx(entropy(P), rel=1e-12)   # scipy normalises P, natural log
        assert s[0] == pytest.approx(E * cnt.max() / cnt.sum(), rel=1e-14)


# ------------------------------------------------------------------ FP8 E4M3 weights
def _e4m3_table():
    """Every finite E4M3 value from the format's definition: sign, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN."""
    vals = []
    for code in range(256):
        sgn = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 7
        if e == 15 and m == 7:
            continue
        vals.append(sgn * (m / 8.0) * 2.0 ** -6 if e == 0 else sgn * (1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


def test_e4m3_round_fixes_every_code_and_the_extremes():
    t = _e4m3_table()
    assert np.array_equal(oracle.e4m3_round(t), t)
    assert t.max() == 448.0 and np.min(t[t > 0]) == 2.0 ** -9
    assert list(oracle.e4m3_round([500.0, -1e6, 2.0 ** -11, 0.0])) == [448.0, -448.0, 0.0, 0.0]


def test_e4m3_round_is_nearest_even():
    t = np.unique(np.abs(_e4m3_table()))
    mids = (t[:-1] + t[1:]) / 2                                     # exact ties
    r = oracle.e4m3_round(mids)
    lo, hi = t[:-1], t[1:]
    # the even neighbour: the one whose code's mantissa bit 0 is clear
    def mant_even(v):
        v = np.asarray(v)
        out = np.empty(v.shape, bool)
        for i, x in enumerate(v):
            if x < 2.0 ** -6:
                out[i] = int(round(x / 2.0 ** -9)) % 2 == 0
            else:
                e = np.floor(np.log2(x))
                out[i] = int(round((x / 2.0 ** e - 1) * 8)) % 2 == 0
        return out
    want = np.where(mant_even(lo), lo, hi)
    assert np.array_equal(r, want)
    # away from ties: the nearest neighbour
    rng = np.random.default_rng(3)
    x = rng.uniform(0, 448, 20000) * rng.choice([1, 2.0 ** -8, 2.0 ** -12], 20000)
    r = oracle.e4m3_round(x)
    idx = np.clip(np.searchsorted(t, x), 1, len(t) - 1)
    near = np.where(np.abs(t[idx] - x) < np.abs(t[idx - 1] - x), t[idx], t[idx - 1])
    tie = np.abs(np.abs(t[idx] - x) - np.abs(t[idx - 1] - x)) == 0
    assert np.array_equal(r[~tie], near[~tie])


def test_e4m3_round_matches_torch_float8():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.normal(0, 50, 50000), rng.normal(0, 1e-3, 20000), _e4m3_table(),
                        (_e4m3_table()[:-1] + _e4m3_table()[1:]) / 2])
    x = x[np.abs(x) <= 448].astype(np.float32)
    import torch
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_round(x), ref)


def test_quantize_e4m3_columns():
    rng = np.random.default_rng(6)
    W = rng.normal(0, 0.05, (64, 9)).astype(np.float32)
    W[:, 3] = 0.0                                                  # an all-zero channel
    q, s = oracle.quantize_e4m3_columns(W)
    assert s.dtype == np.float32 and s[3] == 0 and not q[:, 3].any()
    for n in (0, 1, 2, 4, 8):
        i = np.argmax(np.abs(W[:, n]))
        assert abs(q[i, n]) == 448.0                               # the channel's amax maps to the top code
        assert s[n] == np.float32(np.abs(W[:, n]).max() / np.float32(448))
    # dequantised weights stay within half an E4M3 step (relative 2^-4) of the input
    deq = q * s.astype(np.float64)
    big = np.abs(W) > s.astype(np.float64) * 2.0 ** -6 * 448 / 448
    assert np.all(np.abs(deq - W)[big] <= np.abs(W)[big] * 2.0 ** -4 + 1e-12)


def test_expert_rows_fp8_equals_expert_of_dequantised_weights():
    rng = np.random.default_rng(7)
    d, f, n = 32, 48, 5
    W1, W3 = rng.normal(0, 0.2, (d, f)), rng.normal(0, 0.2, (d, f))
    W2 = rng.normal(0, 0.2, (f, d))
    x = rng.normal(0, 1, (n, d))
    (q1, s1), (q3, s3), (q2, s2) = (oracle.quantize_e4m3_columns(w) for w in (W1, W3, W2))
    got = oracle.expert_rows_fp8(x, q1, s1, q3, s3, q2, s2)
    D1, D3, D2 = q1 * s1.astype(float), q3 * s3.astype(float), q2 * s2.astype(float)
    a = x @ D1
    ref = ((a / (1 + np.exp(-a))) * (x @ D3)) @ D2
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # and it tracks the unquantised expert to the E4M3 precision
    a0 = x @ W1
    full = ((a0 / (1 + np.exp(-a0))) * (x @ W3)) @ W2
    assert np.abs(got - full).max() <= 0.2 * np.abs(full).max()


def test_quantize_e4m3_rows_is_the_channel_quantiser_of_the_transpose():
    rng = np.random.default_rng(8)
    X = rng.normal(0, 1.5, (7, 40)).astype(np.float32)
    X[4] = 0.0                                                     # an all-zero token
    q, s = oracle.quantize_e4m3_rows(X)
    qt, st = oracle.quantize_e4m3_columns(X.T)
    assert np.array_equal(q, qt.T) and np.array_equal(s, st)
    assert s[4] == 0 and not q[4].any()
    for r in (0, 3, 6):                                            # each row's amax maps to the top code
        assert abs(q[r, np.argmax(np.abs(X[r]))]) == 448.0
    # a hand row: amax 7 -> scale 1/64; 3.5 -> 224 exactly; 0.05 -> 3.2 -> 3.25 (step 0.25 in [2, 4))
    q1, s1 = oracle.quantize_e4m3_rows(np.array([[7.0, -3.5, 0.05, 0.0]], np.float32))
    assert s1[0] == np.float32(7.0) / np.float32(448.0)
    assert list(q1[0]) == [448.0, -224.0, 3.25, 0.0]


def test_expert_rows_fp8up_reduces_to_the_plain_expert_when_exact():
    # operands on the E4M3 grid times a power of two, with row / column maxima of
    # 448 times that power: every scale is exactly the power of two and every
    # code the grid value, so the FP8 up projection is exact
    rng = np.random.default_rng(9)
    grid = _e4m3_table()
    d, f, n = 24, 16, 5
    x = rng.choice(grid, (n, d)) * 2.0 ** -10
    x[:, 0] = 448.0 * 2.0 ** -10
    W1, W3 = rng.choice(grid, (d, f)) * 2.0 ** -12, rng.choice(grid, (d, f)) * 2.0 ** -12
    W1[0], W3[1] = 448.0 * 2.0 ** -12, -448.0 * 2.0 ** -12
    W2 = rng.normal(0, 0.2, (f, d)).astype(np.float32).astype(np.float64)   # the C expert reads fp32
    got = oracle.expert_rows_fp8up(x, W1, W3, W2)
    ref = oracle.expert_rows(x, W1, W3, W2)
    assert np.abs(got - ref).max() <= 1e-12 * np.abs(ref).max()
    # with general operands it tracks the unquantised expert to the E4M3 precision
    x2, A1, A3 = rng.normal(0, 1, (n, d)), rng.normal(0, 0.2, (d, f)), rng.normal(0, 0.2, (d, f))
    full = oracle.expert_rows(x2, A1, A3, W2)
    got2 = oracle.expert_rows_fp8up(x2, A1, A3, W2)
    assert np.abs(got2 - full).max() <= 0.25 * np.abs(full).max()


# ------------------------------------------------------------------ affinity-ordered capacity drop
def test_affinity_drop_hand_example():
    # expert 0 gets 4 assignments with cap 2: it keeps the two largest weights (tokens 3
    # and 1; token 0 and 2 tie below them), rows in token order
    idx = np.array([[0, 1], [0, 2], [0, 1], [0, 2]])
    w = np.array([[0.3, 0.7], [0.6, 0.4], [0.3, 0.7], [0.9, 0.1]], np.float32)
    off, cnt, slot, rows = oracle.dispatch_tc_affinity(idx, w, 3, cap=2)
    assert list(cnt) == [4, 2, 2] and list(off) == [0, 2, 4, 6]
    assert list(slot[:, 0]) == [-1, 0, -1, 1]        # tokens 1 and 3 kept by expert 0
    assert list(rows) == [1, 3, 0, 2, 1, 3]
    # a tie at the boundary goes to the lower token
    w2 = w.copy()
    w2[3, 0] = 0.3
    off, cnt, slot, rows = oracle.dispatch_tc_affinity(idx, w2, 3, cap=2)
    assert list(slot[:, 0]) == [0, 1, -1, -1]         # 0.6 (token 1) and the lowest of the 0.3 ties (token 0)


@pytest.mark.parametrize("T,E,k,cap,skew", [(300, 8, 2, 60, 1.2), (500, 16, 1, 20, 1.5), (64, 4, 2, 0, 0.0),
                                            (200, 8, 2, 1000, 1.0)])
def test_affinity_drop_invariants(T, E, k, cap, skew):
    from workloads import random_assignment
    idx = random_assignment(T, E, k, seed=T + E, skew=skew).numpy()
    rng = np.random.default_rng(T)
    w = rng.choice(np.linspace(0.05, 0.95, 19), size=(T, k)).astype(np.float32)   # many ties
    off, cnt, slot, rows = oracle.dispatch_tc_affinity(idx, w, E, cap)
    t_off, t_cnt, t_slot, _ = oracle.dispatch_tc(idx, E, cap)
    assert np.array_equal(cnt, t_cnt) and np.array_equal(off, t_off)   # same counts, same segments
    if cap >= T * k:
        assert np.array_equal(slot, t_slot)                              # nothing dropped: token order
    for e in range(E):
        mine = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        kept = [(t, j) for t, j in mine if slot[t, j] >= 0]
        dropped = [(t, j) for t, j in mine if slot[t, j] < 0]
        assert len(kept) == min(len(mine), cap)
        # every kept assignment outranks every dropped one: larger weight, or equal and lower token
        for tk, jk in kept:
            for td, jd in dropped:
                assert (w[tk, jk], -tk) > (w[td, jd], -td)
        # kept rows of the segment in token order
        rws = sorted(slot[t, j] for t, j in kept)
        assert rws == list(range(off[e], off[e] + len(kept)))
        assert [rows[r] for r in rws] == sorted(t for t, _ in kept)
