"""Float64 CPU oracle for the dropless MoE expert layer (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
table or constant with the CUDA library: the two are compared, never mixed.

Every function is the plain definition, written for reading, not for speed:
numpy float64, library matmuls as single steps, no blocking or fusion.

Sources (web pages on the method; cited by title and section):
  [MM]  "Prime Intellect releases Prime Mega MoE: a trainable fused MoE
        kernel" (MarkTechPost, Russian translation): 128 experts, top-8
        routing ("In brief"); two expert linears with SwiGLU and a combine
        ("How does the fused kernel work?"); precisions BF16 / MXFP8 and the
        fp8_bwd mode (same section).
  [OB]  "Prime Intellect Mega MoE" digest (neurobober), section "Overlapping
        Backward Pass": activation gradients need the weights, not the weight
        gradients, so the backward splits into two independent halves.
  [TE]  "Accelerating dropless MoE in JAX with NVIDIA Transformer Engine"
        (aikraft, rewrite of an NVIDIA Developer post): section 02 "Dropless
        MoE vs capacity-based MoE" (no token dropped or padded); section 03
        "Optimisation 1: grouped GEMM" (one GEMM per expert over its real
        token count), "Optimisation 2: dispatch and combine" (local reordering
        on dispatch, sum of expert outputs on combine) and group-aware MXFP8
        quantisation.
  [MX]  OCP Microscaling Formats (MX) v1.0: E4M3 elements, 32-element blocks,
        E8M0 shared scale.

Readings taken where the pages are silent:
  * top-k selects on the logits (same set as on softmax probabilities, since
    exp is monotone); equal logits go to the lower expert index; slot j is the
    j-th largest.  Gates are the softmax over all E renormalised over the k
    selected experts.
  * W13[e] = [W1 | W3]: columns [0, I) are the gate projection u, [I, 2I) the
    up projection v; A = silu(u) * v.
  * The gate multiplies each expert output before the per-token sum.
  * Rows of expert e are ordered by ascending assignment index a = t*k + j;
    each expert's row range starts at a multiple of ALIGN (=128) rows, with
    zero pad rows (a storage choice; logical counts stay dropless).
  * In the MXFP8 modes intermediates are stored in bf16 and quantised right
    before each GEMM, so codes are decided from bf16 values on both sides.
  * MXFP8 block scale: s = floor(log2(amax)) - 8 clamped to [-127, 127]
    (s = -127 for an all-zero block); elements are x / 2^s rounded to nearest
    even on the E4M3 grid, saturating to +-448.  The contraction axis of every
    GEMM is the blocked axis; token-axis blocks restart at each expert's start.
"""
from __future__ import annotations

import numpy as np

ALIGN = 128          # rows per expert group are padded to a multiple of this
MX_BLOCK = 32        # elements sharing one E8M0 scale [MX]
E4M3_MAX = 448.0     # largest finite E4M3 magnitude [MX]
E4M3_EMAX = 8        # exponent of the largest E4M3 binade [MX]


def f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Router  [MM "In brief": top-8 of 128 experts; TE 01: the router picks the
# top-K experts of each token]
# ---------------------------------------------------------------------------
def route(logits, k):
    """Top-k experts per token with gates renormalised to sum to one.

    Returns ``idx`` int32 [T,k] (slot order: descending logit, ties to the lower
    expert index) and ``gate`` float64 [T,k]: the softmax over all E
    probabilities of the chosen experts, divided by their sum.

    Inputs outside the softmax's domain (readings; the pages only speak of
    real logits): a NaN logit counts as -inf (never preferred to a number);
    a token whose logits are all -inf has no softmax and gets gate 0 in every
    slot, so it contributes nothing to the layer."""
    lg = f64(logits)
    lg = np.where(np.isnan(lg), -np.inf, lg)
    T, E = lg.shape
    # A stable sort on -logit keeps equal logits in ascending expert order.
    order = np.argsort(-lg, axis=1, kind="stable")
    idx = order[:, :k]
    m = lg.max(axis=1, keepdims=True)
    live = np.isfinite(m)                           # False: every logit is -inf
    p = np.exp(lg - np.where(live, m, 0.0))         # exp(-inf) = 0 on dead rows
    with np.errstate(invalid="ignore", divide="ignore"):
        p = p / p.sum(axis=1, keepdims=True)        # softmax over all E
        ps = np.take_along_axis(p, idx, axis=1)
        gate = ps / ps.sum(axis=1, keepdims=True)   # renormalise over top-k
    gate = np.where(live, gate, 0.0)
    return idx.astype(np.int32), gate


def route_backward(gate, idx, dgate, E):
    """d(logits) [T,E] from d(gate) [T,k] through the renormalised top-k
    softmax, with the selection held fixed.  For a selected expert i,
    g_i = exp(l_i) / sum_{j in sel} exp(l_j), so
    dl_i = g_i * (dg_i - sum_j g_j dg_j); unselected experts get zero."""
    g = f64(gate)
    dg = f64(dgate)
    T, k = g.shape
    dl = np.zeros((T, E))
    inner = (g * dg).sum(axis=1, keepdims=True)
    np.put_along_axis(dl, np.asarray(idx, np.int64), g * (dg - inner), axis=1)
    return dl


# ---------------------------------------------------------------------------
# Permutation builder  [TE 02: dropless, ragged per-expert groups;
# TE "Optimisation 2": local reordering of token copies by expert]
# ---------------------------------------------------------------------------
def permute(idx, E, align=ALIGN):
    """Index maps of the expert-major token order.

    counts[e]          assignments routed to expert e
    offsets[E+1]       exclusive scan of counts
    padded_offsets     exclusive scan of counts rounded up to ``align``
    row_of_assign[a]   storage row of assignment a = t*k + j
    assign_of_row[r]   inverse map over padded_offsets[E] rows, -1 on pad rows
    Within an expert, assignments keep ascending order of a (stable)."""
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    n_assign = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    padded = (counts + align - 1) // align * align
    padded_offsets = np.concatenate([[0], np.cumsum(padded)])
    row_of_assign = np.empty(n_assign, dtype=np.int64)
    for e in range(E):
        members = np.nonzero(flat == e)[0]          # ascending a
        row_of_assign[members] = padded_offsets[e] + np.arange(members.size)
    assign_of_row = np.full(padded_offsets[-1], -1, dtype=np.int64)
    assign_of_row[row_of_assign] = np.arange(n_assign)
    return dict(counts=counts, offsets=offsets, padded_offsets=padded_offsets,
                row_of_assign=row_of_assign, assign_of_row=assign_of_row)


def unpermute_rows(rows_perm, row_of_assign, T, k):
    """Token-order view [T,k,...] of rows stored in expert-major order."""
    return np.asarray(rows_perm)[np.asarray(row_of_assign).reshape(T, k)]


# ---------------------------------------------------------------------------
# MXFP8 (E4M3 elements, 32-element blocks, E8M0 scales)  [MM: MXFP8 on
# Blackwell; TE 03: group-aware MXFP8 quantisation; MX v1.0]
# ---------------------------------------------------------------------------
def e4m3_round(y):
    """Nearest-even E4M3 value of y, saturating to +-448 (finite inputs).

    E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; normal binades
    [2^e, 2^(e+1)) for e in [-6, 8] have spacing 2^(e-3); below 2^-6 the
    subnormal spacing is 2^-9."""
    y = f64(y)
    a = np.abs(y)
    _, ex = np.frexp(a)                   # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)            # binade exponent (subnormals: -6)
    q = np.ldexp(1.0, e - 3)              # grid spacing in that binade
    r = np.rint(a / q) * q                # rint: round half to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.signbit(y), -r, r)


def e4m3_encode(r):
    """Byte code of values already on the E4M3 grid (|r| <= 448)."""
    r = f64(r)
    sign = np.signbit(r).astype(np.uint8) << 7
    a = np.abs(r)
    _, ex = np.frexp(a)
    e = ex - 1
    normal = a >= 2.0 ** -6
    field = np.where(normal, e + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, np.where(normal, e, 0)) * 8 - 8,
                    a / 2.0 ** -9)
    mant = np.rint(mant).astype(np.int64)
    return (sign | (field.astype(np.uint8) << 3) | mant.astype(np.uint8)).astype(np.uint8)


def e4m3_decode(code):
    """Value of an E4M3 byte (0x7F / 0xFF are NaN; no infinities) [MX]."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 7) & 1
    f = (c >> 3) & 0xF
    m = c & 7
    val = np.where(f == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, f - 7))
    val = np.where((f == 15) & (m == 7), np.nan, val)
    return np.where(s == 1, -val, val)


def mx_block_exponent(amax):
    """Shared exponent s of a block: floor(log2(amax)) - 8, clamped to
    [-127, 127]; an all-zero block gets -127."""
    amax = f64(amax)
    _, ex = np.frexp(amax)
    s = np.where(amax > 0, (ex - 1) - E4M3_EMAX, -127)
    return np.clip(s, -127, 127).astype(np.int64)


def quantize_mxfp8(x, axis, group_offsets=None):
    """MXFP8-quantise a 2-D array along ``axis`` (1: 32-element blocks along
    each row; 0: 32-row blocks down each column).

    With ``group_offsets`` (axis 0 only) rows are treated as concatenated
    groups and blocks restart at every group start; offsets must be multiples
    of 32, so blocks stay inside one group and rows past the last offset are
    left untouched (codes 0, scale byte 0).
    Returns (codes uint8 same shape, scale bytes uint8: [R, C/32] for axis 1,
    [R/32, C] for axis 0) with scale byte = s + 127."""
    x = f64(x)
    R, C = x.shape
    if axis == 1:
        assert C % MX_BLOCK == 0
        blk = x.reshape(R, C // MX_BLOCK, MX_BLOCK)
        s = mx_block_exponent(np.abs(blk).max(axis=2))            # [R, C/32]
        y = blk / np.ldexp(1.0, s)[:, :, None]
        codes = e4m3_encode(e4m3_round(y)).reshape(R, C)
        return codes, (s + 127).astype(np.uint8)
    assert axis == 0 and R % MX_BLOCK == 0
    codes = np.zeros((R, C), dtype=np.uint8)
    scales = np.zeros((R // MX_BLOCK, C), dtype=np.uint8)
    if group_offsets is None:
        group_offsets = [0, R]
    go = [int(v) for v in group_offsets]
    for g in range(len(go) - 1):
        r0, r1 = go[g], go[g + 1]
        assert r0 % MX_BLOCK == 0 and r1 % MX_BLOCK == 0 and r1 <= R
        for b0 in range(r0, r1, MX_BLOCK):
            blk = x[b0:b0 + MX_BLOCK]                              # [32, C]
            s = mx_block_exponent(np.abs(blk).max(axis=0))         # [C]
            y = blk / np.ldexp(1.0, s)[None, :]
            codes[b0:b0 + MX_BLOCK] = e4m3_encode(e4m3_round(y))
            scales[b0 // MX_BLOCK] = (s + 127).astype(np.uint8)
    return codes, scales


def dequantize_mxfp8(codes, scales, axis):
    """Values represented by (codes, scale bytes) from quantize_mxfp8."""
    v = e4m3_decode(codes)
    sc = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    if axis == 1:
        return v * np.repeat(sc, MX_BLOCK, axis=1)
    return v * np.repeat(sc, MX_BLOCK, axis=0)


def mx_qdq(x, axis):
    """Quantise-dequantise round trip along ``axis`` (rows padded with zeros
    to a multiple of 32 for axis 0, then trimmed back)."""
    x = f64(x)
    if axis == 0:
        R = x.shape[0]
        Rp = -(-R // MX_BLOCK) * MX_BLOCK
        xp = np.zeros((Rp,) + x.shape[1:])
        xp[:R] = x
        c, s = quantize_mxfp8(xp, 0)
        return dequantize_mxfp8(c, s, 0)[:R]
    c, s = quantize_mxfp8(x, 1)
    return dequantize_mxfp8(c, s, 1)


# ---------------------------------------------------------------------------
# Expert layer  [MM "How does the fused kernel work?": dispatch, two expert
# linears, SwiGLU, combine; TE "Optimisation 1": per-expert GEMM over the real
# token count]
# ---------------------------------------------------------------------------
def silu(u):
    return u / (1.0 + np.exp(-u))


def sigmoid(u):
    return 1.0 / (1.0 + np.exp(-u))


def _members(idx, e, tokens=None):
    """Assignments a = t*k + j routed to expert e, ascending (restricted to the
    given tokens when ``tokens`` is not None)."""
    idx = np.asarray(idx)
    k = idx.shape[1]
    flat = idx.reshape(-1)
    a = np.nonzero(flat == e)[0]
    if tokens is not None:
        a = a[np.isin(a // k, tokens)]
    return a


def bf16_round(x):
    """Value of x as an fp32 number stored in bf16: nearest fp32, then the
    nearest bf16 (ties to even: add 0x7FFF plus the lowest kept bit to the
    fp32 bit pattern and drop the low 16 bits).  Finite inputs."""
    u = np.ascontiguousarray(f64(x).astype(np.float32)).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).astype(np.float64)


def _stored(mode, phase):
    """Storage of intermediates that a quantised GEMM reads.  In the MXFP8
    phases the layer keeps activations in BF16 and quantises them right
    before each GEMM ([MM]: BF16 storage, MXFP8 GEMMs), so the E4M3 codes are
    decided from bf16 values; the oracle takes the same decision from the same
    precision.  Identity elsewhere (the plain float64 definition)."""
    use_mx = mode == "mxfp8" or (mode == "fp8_bwd" and phase == "bwd")
    return bf16_round if use_mx else f64


# Blocked axis of each MXFP8 GEMM operand: the contraction axis of its GEMM
# ([TE] 03: MXFP8 GEMMs over ragged groups; [MX]: a block is 32 elements
# along the dot product).  Operands are 2-D: token-major activations have a
# row per assignment of one expert (1 = along the row, 0 = down the 32-row
# token blocks of that expert's rows); weights are W13[e] [H, 2I] and
# W2[e] [I, H] as stored.
MX_AXES = {
    # forward:  h = X W13_e (over H),  z = A W2_e (over I)
    "fwd.X": 1, "fwd.W13": 0, "fwd.A": 1, "fwd.W2": 0,
    # backward: D = dY W2_e^T (over H),  dX = dh W13_e^T (over 2I)
    "bwd.dY": 1, "bwd.W2": 1, "bwd.dh_dx": 1, "bwd.W13": 1,
    # weight gradients over the expert's tokens: dW13_e = X^T dh, dW2_e = A^T (g dY)
    "bwd.X_dw": 0, "bwd.dh_dw": 0, "bwd.A_dw": 0, "bwd.gdY_dw": 0,
}


def _gemm_operands(mode, phase):
    """Quantise-dequantise transform applied to a GEMM operand, called as
    q(x, name) with ``name`` a key of MX_AXES: identity for f32/bf16, MXFP8
    along MX_AXES[name] for mxfp8 (both phases) and for fp8_bwd (backward
    only) [MM: fp8_bwd = BF16 forward, FP8 backward]."""
    use_mx = mode == "mxfp8" or (mode == "fp8_bwd" and phase == "bwd")
    if not use_mx:
        return lambda x, name: f64(x)
    return lambda x, name: mx_qdq(x, MX_AXES[name])


def forward(X, W13, W2, idx, gate, tokens=None, mode="bf16", keep=False):
    """Layer output Y[t] = sum_j gate[t,j] * expert_{idx[t,j]}(x_t).

    expert_e(x) = (silu(x W1_e) * (x W3_e)) W2_e with [W1_e | W3_e] = W13[e].
    ``tokens`` restricts the computation to a subset of tokens (rows of the
    result follow ``tokens``).  In mxfp8 mode every GEMM operand is MXFP8
    quantised along its contraction axis first (activations per row, weights
    per column).  With ``keep`` the per-assignment h = x W13_e, A and the
    ungated expert output z are returned too (rows indexed by assignment)."""
    X = np.asarray(X)
    T, H = X.shape
    E, _, I2 = W13.shape
    I = I2 // 2
    k = np.asarray(idx).shape[1]
    q = _gemm_operands(mode, "fwd")
    st = _stored(mode, "fwd")
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    pos = {int(t): i for i, t in enumerate(tok)}
    Y = np.zeros((len(tok), H))
    saved = {}
    g_flat = f64(gate).reshape(-1)
    for e in range(E):
        a = _members(idx, e, None if tokens is None else tok)
        if a.size == 0:
            continue
        t = a // k
        x = q(X[t], "fwd.X")                             # rows blocked along H
        h = x @ q(W13[e], "fwd.W13")                     # W13_e blocked along H
        u, v = h[:, :I], h[:, I:]
        A = silu(u) * v
        z = q(st(A), "fwd.A") @ q(W2[e], "fwd.W2")       # blocked along I
        contrib = g_flat[a][:, None] * z
        for r, tt in enumerate(t):
            Y[pos[int(tt)]] += contrib[r]
        if keep:
            saved[e] = dict(a=a, h=h, A=A, z=z)
    return (Y, saved) if keep else Y


def backward(X, W13, W2, idx, gate, dY, tokens=None, experts=None, mode="bf16"):
    """Gradients of L = sum_t <Y[t], dY[t]> with the routing held fixed.

    For an assignment (t, j) to expert e with u, v, A, z as in ``forward``:
      D      = dY_t W2_e^T                   (ungated)
      dgate  = <z, dY_t> = <A, D>
      dA     = gate * D
      du     = dA * v * sig(u) * (1 + u * (1 - sig(u)))   (d silu / du)
      dv     = dA * silu(u)
      dh     = [du | dv]
      dX_t  += dh W13_e^T
      dW13_e = sum over e's assignments of x_t^T dh
      dW2_e  = sum over e's assignments of A^T (gate * dY_t)
    Experts with no assignment get zero weight gradients.

    ``tokens`` limits dX / dgate to a token subset (rows follow ``tokens``);
    ``experts`` limits dW13 / dW2 to an expert subset (leading axis follows
    ``experts``).  Either may be None (all).  In mxfp8 / fp8_bwd mode every
    backward GEMM operand is MXFP8-quantised along its contraction axis; the
    token-axis operands of the weight-gradient GEMMs are blocked in 32-row
    groups of the expert's rows in ascending assignment order, zero padded;
    the stored intermediates (h, A, dh, gate * dY) are bf16 values.
    Returns dict(dX, dgate, dW13, dW2)."""
    X = np.asarray(X)
    T, H = X.shape
    E, _, I2 = W13.shape
    I = I2 // 2
    k = np.asarray(idx).shape[1]
    qf = _gemm_operands(mode, "fwd")
    qb = _gemm_operands(mode, "bwd")
    stb = _stored(mode, "bwd")
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    exp_list = list(range(E)) if experts is None else [int(e) for e in experts]
    pos = {int(t): i for i, t in enumerate(tok)}
    tokset = set(pos)
    g_flat = f64(gate).reshape(-1)
    dX = np.zeros((len(tok), H))
    dgate = np.zeros((len(tok), k))
    dW13 = np.zeros((len(exp_list), H, I2))
    dW2 = np.zeros((len(exp_list), I, H))
    want_e = set(exp_list)
    for e in range(E):
        a_all = _members(idx, e)
        a = a_all if e in want_e else a_all[np.isin(a_all // k, tok)]
        if a.size == 0:
            continue
        t = a // k
        g = g_flat[a][:, None]
        # forward recomputation (the forward's own precision); in the MXFP8
        # backward the saved h and A are the stored (bf16) ones
        h = qf(X[t], "fwd.X") @ qf(W13[e], "fwd.W13")
        # two stored forms of the activation: the forward's own output A
        # (from the unrounded h, stored once) is the dW2 operand; dSwiGLU and
        # d(gate) recompute silu(u) * v from the stored pre-activation h
        A_saved = stb((h[:, :I] * sigmoid(h[:, :I])) * h[:, I:])
        h = stb(h)
        u, v = h[:, :I], h[:, I:]
        sg = sigmoid(u)
        A = u * sg * v
        dYt = f64(dY[t])
        D = qb(dYt, "bwd.dY") @ qb(W2[e], "bwd.W2").T   # contraction over H
        dA = g * D
        du = dA * v * sg * (1.0 + u * (1.0 - sg))
        dv = dA * (u * sg)
        dh = stb(np.concatenate([du, dv], axis=1))
        dgate_rows = (A * D).sum(axis=1)
        dx_rows = qb(dh, "bwd.dh_dx") @ qb(W13[e], "bwd.W13").T   # contraction over 2I
        for r, (aa, tt) in enumerate(zip(a, t)):
            if int(tt) in tokset:
                dX[pos[int(tt)]] += dx_rows[r]
                dgate[pos[int(tt)], int(aa) % k] = dgate_rows[r]
        if e in want_e:
            ei = exp_list.index(e)
            # contraction over the expert's tokens (column-wise blocks)
            dW13[ei] = qb(X[t], "bwd.X_dw").T @ qb(dh, "bwd.dh_dw")
            dW2[ei] = qb(A_saved, "bwd.A_dw").T @ qb(stb(g * dYt), "bwd.gdY_dw")
    return dict(dX=dX, dgate=dgate, dW13=dW13, dW2=dW2)


def rel_err(got, ref):
    """max |got - ref| / max |ref| (the tolerance measure of the parity tests)."""
    got = f64(got)
    ref = f64(ref)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / den)
