"""Pins of the oracle's MXFP8 chain (modes ``mxfp8`` and ``fp8_bwd``, forward
and backward) against facts that hold outside the oracle.  CPU only.

1. Block locality.  MXFP8 quantisation along an axis commutes with scaling a
   whole block by a power of two (the shared exponent moves, the E4M3 codes
   stay), and so do bf16 rounding and every float product and sum.  So if an
   operand is blocked along its GEMM's contraction axis, scaling one row or
   column of an input by 4 scales exactly the outputs that depend on it
   linearly by 4 and leaves exactly the others bit for bit unchanged.  A
   block laid along the wrong axis mixes the scaled line with its neighbours
   and breaks one of these equalities.  Each test below names the operands
   whose axes it fixes.
2. A regime where every quantisation and every bf16 storage is exact
   (silu(u) = u once sigmoid(u) rounds to 1 in float64; powers of two; one
   non-zero term per dot product): there the MXFP8 backward must equal the
   plain float64 backward bit for bit, and both the definition evaluated with
   pure-Python loops.
3. Planted mistakes: each entry of the oracle's axis table is flipped in turn
   and some pin of part 1 must fail.
"""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O

MODES = ("mxfp8", "fp8_bwd")


def _layer(T=80, H=64, E=3, k=2, I=32, seed=0):
    """Random layer with ragged experts (more than 32 tokens each, counts not
    multiples of 32)."""
    rng = np.random.default_rng(seed)
    X = O.bf16_round(rng.standard_normal((T, H)))
    W13 = O.bf16_round(rng.standard_normal((E, H, 2 * I)) / math.sqrt(H))
    W2 = O.bf16_round(rng.standard_normal((E, I, H)) / math.sqrt(I))
    lg = rng.standard_normal((T, E))
    idx, gate = O.route(lg, k)
    dY = O.bf16_round(rng.standard_normal((T, H)))
    return dict(X=X, W13=W13, W2=W2, idx=idx, gate=gate, dY=dY)


def _bwd(L, mode, **over):
    a = dict(L, **over)
    return O.backward(a["X"], a["W13"], a["W2"], a["idx"], a["gate"], a["dY"], mode=mode)


def _eq(a, b):
    return np.array_equal(np.asarray(a), np.asarray(b))


def _others(n, i):
    return np.array([j for j in range(n) if j != i])


# ---------------------------------------------------------------- 1. locality
# Each pin returns True when its equalities hold, so the planted-mistake test
# can run them against a deliberately broken oracle.

def pin_fwd_token_rows(L, mode="mxfp8"):
    """Token t0's input row scaled by 4 leaves every other token's output
    unchanged bit for bit (X blocked along H, A along I: both per token).
    Fixes fwd.X, fwd.A."""
    t0 = 5
    X2 = L["X"].copy()
    X2[t0] *= 4.0
    Y = O.forward(L["X"], L["W13"], L["W2"], L["idx"], L["gate"], mode=mode)
    Y2 = O.forward(X2, L["W13"], L["W2"], L["idx"], L["gate"], mode=mode)
    o = _others(len(Y), t0)
    return _eq(Y2[o], Y[o]) and not _eq(Y2[t0], Y[t0])


def pin_fwd_w2_columns(L, mode="mxfp8"):
    """Column h0 of every W2_e scaled by 4 scales column h0 of Y by exactly 4
    and leaves the other columns unchanged (W2 blocked down I).  Fixes
    fwd.W2."""
    h0 = 7
    W22 = L["W2"].copy()
    W22[:, :, h0] *= 4.0
    Y = O.forward(L["X"], L["W13"], L["W2"], L["idx"], L["gate"], mode=mode)
    Y2 = O.forward(L["X"], L["W13"], W22, L["idx"], L["gate"], mode=mode)
    o = _others(Y.shape[1], h0)
    return _eq(Y2[:, h0], 4.0 * Y[:, h0]) and _eq(Y2[:, o], Y[:, o])


def pin_fwd_w13_columns(L, mode="mxfp8"):
    """Up-projection column I + i0 of W13_e scaled by 4 scales that column of
    the pre-activation h by exactly 4 and leaves the others unchanged (W13
    blocked down H).  Fixes fwd.W13."""
    I = L["W2"].shape[1]
    c = I + 3
    W132 = L["W13"].copy()
    W132[:, :, c] *= 4.0
    _, s1 = O.forward(L["X"], L["W13"], L["W2"], L["idx"], L["gate"], mode=mode, keep=True)
    _, s2 = O.forward(L["X"], W132, L["W2"], L["idx"], L["gate"], mode=mode, keep=True)
    o = _others(2 * I, c)
    return all(_eq(s2[e]["h"][:, c], 4.0 * s1[e]["h"][:, c]) and _eq(s2[e]["h"][:, o], s1[e]["h"][:, o])
               for e in s1)


def pin_bwd_dy_rows(L, mode):
    """dY of token t0 scaled by 4: dX[t0] and dgate[t0] scale by exactly 4,
    every other token's dX and dgate is unchanged (dY blocked along H for D,
    dh along 2I for dX: both per row).  Fixes bwd.dY, bwd.dh_dx."""
    t0 = 11
    dY2 = L["dY"].copy()
    dY2[t0] *= 4.0
    g1, g2 = _bwd(L, mode), _bwd(L, mode, dY=dY2)
    o = _others(len(dY2), t0)
    return (_eq(g2["dX"][t0], 4.0 * g1["dX"][t0]) and _eq(g2["dgate"][t0], 4.0 * g1["dgate"][t0])
            and _eq(g2["dX"][o], g1["dX"][o]) and _eq(g2["dgate"][o], g1["dgate"][o]))


def pin_bwd_dy_columns(L, mode):
    """Column h0 of dY scaled by 4: column h0 of every dW2_e scales by
    exactly 4 and the other columns are unchanged (gate * dY blocked down the
    expert's tokens).  Fixes bwd.gdY_dw."""
    h0 = 9
    dY2 = L["dY"].copy()
    dY2[:, h0] *= 4.0
    g1, g2 = _bwd(L, mode), _bwd(L, mode, dY=dY2)
    o = _others(dY2.shape[1], h0)
    return _eq(g2["dW2"][:, :, h0], 4.0 * g1["dW2"][:, :, h0]) and _eq(g2["dW2"][:, :, o], g1["dW2"][:, :, o])


def pin_bwd_w2_rows(L, mode):
    """Row i0 of W2_e0 scaled by 4: D's column i0 (hence dh's columns i0 and
    I + i0) scale by 4, so those two columns of dW13_e0 scale by exactly 4;
    every other column of dW13 and all of dW2 are unchanged (W2 blocked
    along H for D; dh blocked down the tokens for dW13).  Fixes bwd.W2,
    bwd.dh_dw."""
    e0, i0 = 1, 4
    I = L["W2"].shape[1]
    W22 = L["W2"].copy()
    W22[e0, i0] *= 4.0
    g1, g2 = _bwd(L, mode), _bwd(L, mode, W2=W22)
    cols = [i0, I + i0]
    o = _others(2 * I, i0)
    o = o[o != I + i0]
    oe = _others(W22.shape[0], e0)
    return (_eq(g2["dW13"][e0][:, cols], 4.0 * g1["dW13"][e0][:, cols])
            and _eq(g2["dW13"][e0][:, o], g1["dW13"][e0][:, o])
            and _eq(g2["dW13"][oe], g1["dW13"][oe]) and _eq(g2["dW2"], g1["dW2"]))


def pin_bwd_x_w13_rows(L, mode="fp8_bwd", f=4.0):
    """fp8_bwd (exact float64 forward): column h0 of X scaled by f and row h0
    of every W13_e by 1/f (f a power of two) leave X W13 unchanged bit for
    bit; then dX's column h0 scales by exactly 1/f and row h0 of every dW13_e
    by exactly f, all else unchanged (W13 blocked along 2I for dX; X blocked
    down the tokens for dW13).  The side scaled up becomes the maximum of
    most blocks laid across it, so f = 4 probes the X blocks and f = 1/4 the
    W13 blocks.  Fixes bwd.W13, bwd.X_dw."""
    h0 = 13
    X2 = L["X"].copy()
    X2[:, h0] *= f
    W132 = L["W13"].copy()
    W132[:, h0, :] /= f
    g1, g2 = _bwd(L, mode), _bwd(L, mode, X=X2, W13=W132)
    o = _others(X2.shape[1], h0)
    return (_eq(g2["dX"][:, h0], g1["dX"][:, h0] / f) and _eq(g2["dX"][:, o], g1["dX"][:, o])
            and _eq(g2["dW13"][:, h0], f * g1["dW13"][:, h0]) and _eq(g2["dW13"][:, o], g1["dW13"][:, o])
            and _eq(g2["dW2"], g1["dW2"]) and _eq(g2["dgate"], g1["dgate"]))


def pin_bwd_act_columns(L, mode):
    """Up-projection column I + i0 of W13_e0 scaled by 4: the stored
    activation's column i0 scales by 4, so row i0 of dW2_e0 scales by exactly
    4 and its other rows are unchanged (A blocked down the tokens for dW2;
    in mxfp8 also W13 blocked down H in the recomputed forward).  Fixes
    bwd.A_dw (and fwd.W13 in mxfp8)."""
    e0, i0 = 2, 6
    I = L["W2"].shape[1]
    W132 = L["W13"].copy()
    W132[e0, :, I + i0] *= 4.0
    g1, g2 = _bwd(L, mode), _bwd(L, mode, W13=W132)
    o = _others(I, i0)
    return (_eq(g2["dW2"][e0][i0], 4.0 * g1["dW2"][e0][i0]) and _eq(g2["dW2"][e0][o], g1["dW2"][e0][o]))


def pin_bwd_expert_groups(L, mode):
    """The weight gradients of expert e0 do not depend on tokens routed
    elsewhere: token-axis blocks restart at each expert's rows ([TE] 03,
    group-aware quantisation)."""
    e0 = 0
    t = int(np.nonzero(~(L["idx"] == e0).any(1))[0][0])
    dY2 = L["dY"].copy()
    dY2[t] *= 3.0
    X2 = L["X"].copy()
    X2[t] *= -2.0
    g1, g2 = _bwd(L, mode), _bwd(L, mode, dY=dY2, X=X2)
    return _eq(g2["dW13"][e0], g1["dW13"][e0]) and _eq(g2["dW2"][e0], g1["dW2"][e0])


FWD_PINS = [pin_fwd_token_rows, pin_fwd_w2_columns, pin_fwd_w13_columns]
BWD_PINS = [pin_bwd_dy_rows, pin_bwd_dy_columns, pin_bwd_w2_rows, pin_bwd_act_columns,
            pin_bwd_expert_groups]


@pytest.mark.parametrize("pin", FWD_PINS, ids=lambda f: f.__name__)
def test_forward_locality(pin):
    assert pin(_layer())


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda f: f.__name__)
def test_backward_locality(pin, mode):
    assert pin(_layer(seed=1), mode)


@pytest.mark.parametrize("f", [4.0, 0.25])
def test_backward_x_w13_locality(f):
    assert pin_bwd_x_w13_rows(_layer(seed=2), f=f)


def test_locality_pins_hold_trivially_in_bf16_mode():
    """Without quantisation every pin holds too (a control: the equalities
    themselves follow from float arithmetic, not from the blocking)."""
    L = _layer(seed=3)
    assert all(p(L, "bf16") for p in BWD_PINS)
    assert pin_bwd_x_w13_rows(L, "bf16", 4.0) and pin_bwd_x_w13_rows(L, "bf16", 0.25)


# ------------------------------------------------------------ 2. exact regime
def _exact_layer():
    """E = 2, k = 2 with equal logits (gates 1/2), T = H = I = 32.  X and dY
    are diagonal, every weight a power of two, u >= 64 (sigmoid(u) = 1 in
    float64, so silu(u) = u and silu'(u) = 1): every dot product has one
    non-zero term, every intermediate is a power of two (or 0) whose blocks
    span fewer than 17 binades, so MXFP8 and bf16 represent all of them."""
    T = H = I = 32
    E, k = 2, 2
    x = np.array([2.0 ** (t % 4 - 1) for t in range(T)])
    dy = np.array([2.0 ** (t % 3) for t in range(T)])
    X = np.diag(x)
    dY = np.diag(dy)
    W13 = np.zeros((E, H, 2 * I))
    W2 = np.zeros((E, I, H))
    for e in range(E):
        for h in range(H):
            for i in range(I):
                u = 2.0 ** (6 + (h + 2 * i + e) % 3)
                v = (-1) ** (h + i + e) * 2.0 ** ((h * i + e) % 4 - 2) if (h + i + e) % 5 else 0.0
                W13[e, h, i] = u / x[h]
                W13[e, h, I + i] = v / x[h]
                W2[e, i, h] = (-1) ** (i * h + e) * 2.0 ** ((i + 3 * h + e) % 3)
    idx, gate = O.route(np.zeros((T, E)), k)
    return X, W13, W2, idx, gate, dY


def _loops_backward(X, W13, W2, idx, gate, dY):
    """The backward's definition with pure-Python loops (silu(u) = u and
    silu'(u) = 1 in this regime, as checked by the caller)."""
    T, H = X.shape
    E, _, I2 = W13.shape
    I = I2 // 2
    k = idx.shape[1]
    dX = [[0.0] * H for _ in range(T)]
    dgate = [[0.0] * k for _ in range(T)]
    dW13 = [[[0.0] * I2 for _ in range(H)] for _ in range(E)]
    dW2 = [[[0.0] * H for _ in range(I)] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            e, g = int(idx[t, j]), float(gate[t, j])
            h = [sum(X[t, c] * W13[e, c, n] for c in range(H)) for n in range(I2)]
            u, v = h[:I], h[I:]
            D = [sum(dY[t, c] * W2[e, i, c] for c in range(H)) for i in range(I)]
            A = [u[i] * v[i] for i in range(I)]
            dgate[t][j] = sum(A[i] * D[i] for i in range(I))
            dh = [g * D[i] * v[i] for i in range(I)] + [g * D[i] * u[i] for i in range(I)]
            for c in range(H):
                dX[t][c] += sum(dh[n] * W13[e, c, n] for n in range(I2))
                for n in range(I2):
                    dW13[e][c][n] += X[t, c] * dh[n]
            for i in range(I):
                for c in range(H):
                    dW2[e][i][c] += A[i] * g * dY[t, c]
    return dict(dX=np.array(dX), dgate=np.array(dgate), dW13=np.array(dW13), dW2=np.array(dW2))


def test_exact_regime_mxfp8_backward_equals_definition():
    X, W13, W2, idx, gate, dY = _exact_layer()
    assert (gate == 0.5).all()
    h = X @ W13[0]
    assert (h[:, :32] >= 64).all() and (O.sigmoid(h[:, :32]) == 1.0).all()
    ref = O.backward(X, W13, W2, idx, gate, dY, mode="bf16")
    loops = _loops_backward(X, W13, W2, idx, gate, dY)
    for key in ref:
        assert _eq(ref[key], loops[key]), key
        assert np.abs(ref[key]).max() > 0, key
    for mode in MODES:
        got = O.backward(X, W13, W2, idx, gate, dY, mode=mode)
        for key in ref:
            assert _eq(got[key], ref[key]), (mode, key)
    Yb = O.forward(X, W13, W2, idx, gate, mode="bf16")
    assert _eq(O.forward(X, W13, W2, idx, gate, mode="mxfp8"), Yb)


def test_exact_regime_is_sensitive_to_one_inexact_operand():
    """Control: one weight moved off the E4M3 grid (a 5-bit mantissa) makes
    the MXFP8 backward differ from the plain one."""
    X, W13, W2, idx, gate, dY = _exact_layer()
    W2 = W2.copy()
    W2[1, 3, 5] *= 1.03125
    ref = O.backward(X, W13, W2, idx, gate, dY, mode="bf16")
    got = O.backward(X, W13, W2, idx, gate, dY, mode="mxfp8")
    assert not _eq(got["dX"], ref["dX"])


# --------------------------------------------------------- 3. planted mistakes
def _all_pins_hold(L):
    ok = all(p(L) for p in FWD_PINS)
    ok = ok and all(p(L, m) for p in BWD_PINS for m in MODES)
    return ok and pin_bwd_x_w13_rows(L, f=4.0) and pin_bwd_x_w13_rows(L, f=0.25)


@pytest.mark.parametrize("name", sorted(O.MX_AXES))
def test_flipped_axis_is_caught(name, monkeypatch):
    """Flipping the blocked axis of any one MXFP8 operand in the oracle makes
    at least one locality pin fail."""
    L = _layer(seed=4)
    assert _all_pins_hold(L)
    monkeypatch.setitem(O.MX_AXES, name, 1 - O.MX_AXES[name])
    assert not _all_pins_hold(L), name


@pytest.mark.parametrize("mode", MODES)
def test_sampled_subbatches_equal_full_layer(mode):
    """The per-expert sub-batches the full-size GPU tests give the oracle
    (only the sampled tokens' assignments, or all of an expert's for its
    weight gradients) reproduce the full layer's rows and weight gradients:
    every operand of Y, dX and d(gate) is blocked along a row, and the token
    blocks of the weight gradients see the whole expert."""
    import _oracle_jobs
    from workloads import MoEConfig, make_inputs
    cfg = MoEConfig("sub", 300, 64, 6, 3, 64, "bf16")
    inp = make_inputs(cfg, 3)
    idx, gate = O.route(inp["logits"], cfg.k)
    tokens = np.array([3, 77, 150, 299])
    full_in = {k: _f(v) for k, v in inp.items()}
    Yf = O.forward(full_in["X"], full_in["W13"], full_in["W2"], idx, gate, mode=mode)
    gf = O.backward(full_in["X"], full_in["W13"], full_in["W2"], idx, gate, full_in["dY"], mode=mode)
    Y, dX, dg, dws = _oracle_jobs.run_sampled(inp, idx, gate, tokens, [1, 4], mode, workers=2)
    assert np.allclose(Y, Yf[tokens], rtol=1e-12, atol=1e-12)
    assert np.allclose(dX, gf["dX"][tokens], rtol=1e-12, atol=1e-12)
    assert np.allclose(dg, gf["dgate"][tokens], rtol=1e-12, atol=1e-12)
    for e in (1, 4):
        assert np.allclose(dws[e][0], gf["dW13"][e], rtol=1e-12, atol=1e-12)
        assert np.allclose(dws[e][1], gf["dW2"][e], rtol=1e-12, atol=1e-12)


def _f(a):
    from workloads import bf16_bits_to_f32
    return bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a
