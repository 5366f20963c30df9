"""Pins of the float64 oracle against facts fixed outside the oracle itself:
brute force on tiny inputs, closed forms, invariants, finite differences and
hand-derived MXFP8 values.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- router
def _bruteforce_topk(row, k):
    """Full sort of (expert, logit) pairs with pure-Python keys."""
    pairs = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return pairs[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (128, 8), (5, 5), (3, 1)])
def test_route_matches_bruteforce_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    # small integer logits force many ties
    lg = rng.integers(-3, 4, size=(64, E)).astype(np.float32)
    lg[0, :] = 0.0                                    # all tied
    idx, gate = O.route(lg, k)
    for t in range(lg.shape[0]):
        assert list(idx[t]) == _bruteforce_topk(lg[t], k)
    assert np.allclose(gate.sum(1), 1.0, rtol=0, atol=1e-15)
    assert (gate > 0).all() and (gate <= 1).all()


def test_route_gate_ratios_are_exp_of_logit_gaps():
    """g_i / g_j = exp(l_i - l_j) for selected i, j (closed form of a
    renormalised softmax), and slot order is non-increasing in gate."""
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((32, 128)).astype(np.float32)
    idx, gate = O.route(lg, 8)
    sel = np.take_along_axis(lg.astype(np.float64), idx.astype(np.int64), 1)
    for j in range(1, 8):
        assert np.allclose(gate[:, 0] / gate[:, j], np.exp(sel[:, 0] - sel[:, j]),
                           rtol=1e-12)
        assert (gate[:, j - 1] >= gate[:, j]).all()


def test_route_k_equals_E_is_softmax():
    """With k = E nothing is dropped: the gates are scipy's softmax, permuted
    into descending order."""
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((16, 12)).astype(np.float32)
    idx, gate = O.route(lg, 12)
    ref = scipy.special.softmax(lg.astype(np.float64), axis=1)
    assert np.allclose(gate, np.take_along_axis(ref, idx.astype(np.int64), 1),
                       rtol=1e-12, atol=0)


def test_route_neg_inf_experts_never_selected():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((50, 16)).astype(np.float32)
    lg[:, [2, 7, 11]] = -np.inf
    idx, gate = O.route(lg, 4)
    assert not np.isin(idx, [2, 7, 11]).any()
    assert np.isfinite(gate).all()


def test_route_inputs_outside_the_softmax_domain():
    """A token whose logits are all -inf is routed to experts 0..k-1 (equal
    keys, ascending index, as a full sort gives) with zero gates; a NaN logit
    routes like -inf; a token with fewer than k finite logits gives its -inf
    slots gate 0 and its finite ones the softmax of the finite logits."""
    lg = np.array([[-np.inf] * 6,
                   [0.5, np.nan, 2.0, np.nan, -1.0, 0.0],
                   [1.0, -np.inf, -np.inf, 3.0, -np.inf, -np.inf]], np.float32)
    idx, gate = O.route(lg, 3)
    assert list(idx[0]) == [0, 1, 2] and (gate[0] == 0).all()
    nan_as_inf = np.where(np.isnan(lg[1]), -np.inf, lg[1])
    i1, g1 = O.route(nan_as_inf[None], 3)
    assert list(idx[1]) == list(i1[0]) == _bruteforce_topk(nan_as_inf, 3)
    assert np.array_equal(gate[1], g1[0]) and np.isfinite(gate).all()
    assert list(idx[2]) == [3, 0, 1]
    assert gate[2, 2] == 0
    assert np.allclose(gate[2, :2], scipy.special.softmax([3.0, 1.0]), rtol=1e-15, atol=0)


def test_route_backward_finite_difference():
    """d(logits) through the renormalised top-k softmax vs central
    differences of sum(gate * w) with the selection held fixed."""
    rng = np.random.default_rng(4)
    T, E, k = 5, 10, 3
    lg = rng.standard_normal((T, E))
    idx, gate = O.route(lg, k)
    w = rng.standard_normal((T, k))
    dl = O.route_backward(gate, idx, w, E)
    h = 1e-6
    for t in range(T):
        for e in range(E):
            def loss(delta):
                l2 = lg.copy()
                l2[t, e] += delta
                sel = np.take_along_axis(l2, idx.astype(np.int64), 1)
                ex = np.exp(sel - sel.max(1, keepdims=True))
                g = ex / ex.sum(1, keepdims=True)
                return (g * w).sum()
            fd = (loss(h) - loss(-h)) / (2 * h)
            assert abs(fd - dl[t, e]) < 1e-8


# --------------------------------------------------------------- permute
def _bruteforce_perm(idx, E, align):
    flat = [int(v) for v in np.asarray(idx).reshape(-1)]
    order = sorted(range(len(flat)), key=lambda a: (flat[a], a))
    counts = [flat.count(e) for e in range(E)]
    row, rows = {}, []
    base = 0
    pos = 0
    for e in range(E):
        for r in range(counts[e]):
            row[order[pos]] = base + r
            pos += 1
        base += -(-counts[e] // align) * align
    return counts, [row[a] for a in range(len(flat))], base


@pytest.mark.parametrize("T,E,k,align", [(37, 8, 2, 128), (300, 16, 4, 8), (5, 4, 1, 1),
                                         (64, 6, 3, 32)])
def test_permute_against_bruteforce_and_invariants(T, E, k, align):
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 0] -= 10                     # expert 0 rarely / never picked
    idx, _ = O.route(lg, k)
    p = O.permute(idx, E, align)
    counts, rows, tpad = _bruteforce_perm(idx, E, align)
    assert list(p["counts"]) == counts
    assert list(p["row_of_assign"]) == rows
    assert p["padded_offsets"][-1] == tpad
    assert p["counts"].sum() == T * k
    assert (np.diff(p["offsets"]) == p["counts"]).all()
    assert (p["padded_offsets"] % align == 0).all()
    assert (np.diff(p["padded_offsets"]) >= p["counts"]).all()
    aor = p["assign_of_row"]
    # inverse maps; pad rows are -1
    assert (aor[p["row_of_assign"]] == np.arange(T * k)).all()
    assert (aor == -1).sum() == tpad - T * k
    # permute then unpermute is the identity
    x = rng.standard_normal((T, 7))
    xp = np.zeros((tpad, 7))
    xp[p["row_of_assign"]] = np.repeat(x, k, axis=0)
    back = O.unpermute_rows(xp, p["row_of_assign"], T, k)
    assert np.array_equal(back, np.repeat(x[:, None, :], k, axis=1))


# ----------------------------------------------------------- forward pins
def _tiny_layer(T=6, H=8, E=4, k=2, I=4, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, H))
    W13 = rng.standard_normal((E, H, 2 * I)) / math.sqrt(H)
    W2 = rng.standard_normal((E, I, H)) / math.sqrt(I)
    lg = rng.standard_normal((T, E))
    idx, gate = O.route(lg, k)
    dY = rng.standard_normal((T, H))
    return X, W13, W2, idx, gate, dY


def test_single_expert_is_dense_swiglu_ffn():
    """E = 1, k = 1: every gate is 1 and the layer is a dense SwiGLU FFN,
    evaluated here element by element with pure-Python loops."""
    T, H, I = 5, 6, 3
    rng = np.random.default_rng(7)
    X = rng.standard_normal((T, H))
    W13 = rng.standard_normal((1, H, 2 * I))
    W2 = rng.standard_normal((1, I, H))
    idx, gate = O.route(np.zeros((T, 1), np.float32), 1)
    assert (gate == 1.0).all()
    Y = O.forward(X, W13, W2, idx, gate)
    for t in range(T):
        act = []
        for i in range(I):
            u = sum(X[t, h] * W13[0, h, i] for h in range(H))
            v = sum(X[t, h] * W13[0, h, I + i] for h in range(H))
            act.append(u / (1.0 + math.exp(-u)) * v)
        for h in range(H):
            y = sum(act[i] * W2[0, i, h] for i in range(I))
            assert abs(Y[t, h] - y) < 1e-12 * max(1.0, abs(y))


def test_forward_is_gate_weighted_sum_of_experts_by_loops():
    """Y[t] = sum_j g_tj * expert(x_t) with the expert evaluated by loops."""
    X, W13, W2, idx, gate, _ = _tiny_layer(T=4, H=5, E=3, k=2, I=3, seed=11)
    Y = O.forward(X, W13, W2, idx, gate)
    T, H = X.shape
    I = W2.shape[1]
    for t in range(T):
        y = [0.0] * H
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            u = [sum(X[t, h] * W13[e, h, i] for h in range(H)) for i in range(I)]
            v = [sum(X[t, h] * W13[e, h, I + i] for h in range(H)) for i in range(I)]
            a = [u[i] / (1 + math.exp(-u[i])) * v[i] for i in range(I)]
            for h in range(H):
                y[h] += gate[t, j] * sum(a[i] * W2[e, i, h] for i in range(I))
        assert np.allclose(Y[t], y, rtol=1e-12, atol=1e-12)


def test_forward_token_subset_matches_full():
    X, W13, W2, idx, gate, _ = _tiny_layer(T=20, seed=3)
    Y = O.forward(X, W13, W2, idx, gate)
    sub = np.array([17, 2, 9])
    assert np.allclose(O.forward(X, W13, W2, idx, gate, tokens=sub), Y[sub], rtol=0, atol=1e-14)


# ---------------------------------------------------------- backward pins
def _loss(X, W13, W2, idx, gate, dY):
    return float((O.forward(X, W13, W2, idx, gate) * dY).sum())


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_central_differences(seed):
    X, W13, W2, idx, gate, dY = _tiny_layer(seed=seed)
    g = O.backward(X, W13, W2, idx, gate, dY)
    h = 1e-6

    def fd(arr, name):
        out = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            old = arr[i]
            arr[i] = old + h
            lp = _loss(**ctx)
            arr[i] = old - h
            lm = _loss(**ctx)
            arr[i] = old
            out[i] = (lp - lm) / (2 * h)
        return out

    ctx = dict(X=X, W13=W13, W2=W2, idx=idx, gate=gate, dY=dY)
    for name, key in [("X", "dX"), ("W13", "dW13"), ("W2", "dW2"), ("gate", "dgate")]:
        num = fd(ctx[name], name)
        ana = g[key]
        err = np.abs(num - ana).max() / max(np.abs(num).max(), 1e-30)
        assert err < 1e-6, (name, err)


def test_empty_expert_gets_zero_weight_gradient():
    X, W13, W2, idx, gate, dY = _tiny_layer(T=6, E=5, seed=5)
    idx = np.where(idx == 4, 3, idx)            # nobody picks expert 4
    idx[:, 1] = np.where(idx[:, 0] == idx[:, 1], (idx[:, 1] + 1) % 4, idx[:, 1])
    g = O.backward(X, W13, W2, idx, gate, dY)
    assert not (idx == 4).any()
    assert (g["dW13"][4] == 0).all() and (g["dW2"][4] == 0).all()


def test_dgate_identity_two_ways():
    """d(gate)_{t,j} = <z_{t,j}, dY_t> (ungated expert output against the
    upstream gradient) equals the backward's <A, D>."""
    X, W13, W2, idx, gate, dY = _tiny_layer(T=9, seed=8)
    _, saved = O.forward(X, W13, W2, idx, gate, keep=True)
    g = O.backward(X, W13, W2, idx, gate, dY)
    k = idx.shape[1]
    for e, s in saved.items():
        for r, a in enumerate(s["a"]):
            t, j = divmod(int(a), k)
            assert abs(g["dgate"][t, j] - s["z"][r] @ dY[t]) < 1e-12


def test_backward_subsets_match_full():
    X, W13, W2, idx, gate, dY = _tiny_layer(T=12, seed=9)
    full = O.backward(X, W13, W2, idx, gate, dY)
    sub = O.backward(X, W13, W2, idx, gate, dY, tokens=[3, 0], experts=[2, 1])
    assert np.allclose(sub["dX"], full["dX"][[3, 0]], atol=1e-14, rtol=0)
    assert np.allclose(sub["dgate"], full["dgate"][[3, 0]], atol=1e-14, rtol=0)
    assert np.allclose(sub["dW13"], full["dW13"][[2, 1]], atol=1e-14, rtol=0)
    assert np.allclose(sub["dW2"], full["dW2"][[2, 1]], atol=1e-14, rtol=0)


# -------------------------------------------------------------- MXFP8 pins
def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_e4m3_decode_golden_codes():
    for code, val in _load("e4m3_codes.json")["codes"]:
        got = O.e4m3_decode(int(code, 16))
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_all_finite_codes_round_trip():
    """Every finite E4M3 code decodes to a value that rounds and encodes back
    to itself; there are 253 distinct finite values (254 finite codes, +-0)."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_encode(O.e4m3_round(vals)), codes)
    assert len(set(vals.tolist())) == 253
    # strictly increasing over the positive codes 0x00..0x7E
    pos = O.e4m3_decode(np.arange(0x7F))
    assert (np.diff(pos) > 0).all()


def test_e4m3_round_is_nearest_on_the_grid():
    """For random reals in range, the rounded value is a grid point at least
    as close as both neighbours; ties go to the even code."""
    grid = O.e4m3_decode(np.arange(0x7F))               # 0 .. 448
    rng = np.random.default_rng(0)
    y = rng.uniform(0, 448, 20000)
    r = O.e4m3_round(y)
    d = np.abs(grid[None, :] - y[:, None]).min(1)
    assert np.allclose(np.abs(r - y), d, rtol=0, atol=1e-12)
    mids = (grid[:-1] + grid[1:]) / 2
    rm = O.e4m3_round(mids)
    codes = O.e4m3_encode(rm)
    assert ((codes & 1) == 0).all()


def test_mxfp8_golden_blocks():
    for case in _load("mxfp8_blocks.json")["cases"]:
        vals = [float(v) for v in case["values"]]
        blk = np.zeros((1, 32))
        blk[0, :len(vals)] = vals
        codes, scales = O.quantize_mxfp8(blk, 1)
        assert int(scales[0, 0]) == case["scale"], case["name"]
        want = [int(c, 16) for c in case["codes"]]
        assert list(codes[0, :len(vals)]) == want, case["name"]
        assert (codes[0, len(vals):] == 0).all()
        # column-wise quantisation of the transposed block agrees
        c0, s0 = O.quantize_mxfp8(blk.T, 0)
        assert np.array_equal(c0.T, codes) and int(s0[0, 0]) == case["scale"]


def test_mxfp8_exact_values_survive_round_trip():
    """Values of the form code * 2^s with a common s are reproduced exactly
    when the block's largest magnitude sits in the top binade [256, 448]."""
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, size=(64, 32)).astype(np.uint8)
    codes[:, 0] = rng.integers(0x78, 0x7F, size=64)    # amax in [256, 448]
    signs = rng.integers(0, 2, size=(64, 32)).astype(np.uint8) << 7
    s = rng.integers(-20, 20, size=(64, 1))
    x = O.e4m3_decode(codes | signs) * np.ldexp(1.0, s)
    c, sc = O.quantize_mxfp8(x, 1)
    assert np.array_equal(O.dequantize_mxfp8(c, sc, 1), x)


def test_mxfp8_quantisation_error_bound():
    """Rounding error bounds of 3 mantissa bits: with y = x / 2^s, elements in
    the normal range (2^-6 <= |y| <= 448) are within |x| * 2^-4, subnormal
    ones within 2^(s-10), and elements above 448 * 2^s map to +-448 * 2^s."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((128, 256)) * np.exp(rng.uniform(-8, 8, (128, 1)))
    c, sc = O.quantize_mxfp8(x, 1)
    xd = O.dequantize_mxfp8(c, sc, 1)
    s = np.repeat(sc.astype(np.int64) - 127, 32, axis=1)
    y = np.abs(x) / np.ldexp(1.0, s)
    err = np.abs(x - xd)
    normal = (y >= 2.0 ** -6) & (y <= 448)
    assert (err[normal] <= np.abs(x[normal]) * 2.0 ** -4).all()
    sub = y < 2.0 ** -6
    assert (err[sub] <= np.ldexp(1.0, s[sub] - 10)).all()
    sat = y > 448
    assert sat.any()
    assert np.array_equal(np.abs(xd[sat]), 448 * np.ldexp(1.0, s[sat]))
    assert (np.sign(xd[sat]) == np.sign(x[sat])).all()


def test_mxfp8_colwise_groups_restart_at_group_start():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((128, 64))
    x[64:96] *= 1000.0
    go = [0, 64, 96, 128]
    c, sc = O.quantize_mxfp8(x, 0, go)
    for g in range(3):
        cg, sg = O.quantize_mxfp8(x[go[g]:go[g + 1]], 0)
        assert np.array_equal(c[go[g]:go[g + 1]], cg)
        assert np.array_equal(sc[go[g] // 32:go[g + 1] // 32], sg)


def test_bf16_round_matches_torch_conversion():
    """The oracle's bf16 storage rounding equals torch's fp32 -> bf16
    conversion (round to nearest even) on random and tie values."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-20, 20, 50000))).astype(np.float32)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 256 + 1], np.float32)
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x), want)
    assert O.bf16_round(np.float32(1 + 2.0 ** -8)) == 1.0          # tie -> even
    assert O.bf16_round(np.float32(1 + 3 * 2.0 ** -8)) == 1 + 2.0 ** -6


def test_mxfp8_mode_equals_bf16_mode_on_representable_operands():
    """E=1, k=1 with inputs and weights that MXFP8 represents exactly and
    intermediates quantised from bf16: the mxfp8 forward equals the plain
    forward computed on the same quantise-dequantised operands."""
    rng = np.random.default_rng(9)
    T, H, I = 4, 64, 32
    def repr_(shape, axis):
        return O.mx_qdq(O.bf16_round(rng.standard_normal(shape)), axis)
    X = repr_((T, H), 1)
    W13 = repr_((H, 2 * I), 0)[None]
    W2 = repr_((I, H), 0)[None]
    idx, gate = O.route(np.zeros((T, 1)), 1)
    Ymx = O.forward(X, W13, W2, idx, gate, mode="mxfp8")
    h = X @ W13[0]
    A = O.silu(h[:, :I]) * h[:, I:]
    Yref = O.mx_qdq(O.bf16_round(A), 1) @ W2[0]
    assert np.allclose(Ymx, Yref, rtol=1e-12, atol=1e-12)
