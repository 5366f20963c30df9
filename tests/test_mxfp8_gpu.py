"""MXFP8 (E4M3 / 32-element blocks / E8M0) and fp8_bwd (bf16 forward, MXFP8
backward) modes of the layer on the GPU vs the float64 oracle, whose GEMM
operands go through its own (bit-exact, separately tested) MXFP8 quantiser
along each GEMM's contraction axis."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from workloads import CONFIGS, MoEConfig, make_inputs

from _common import TOL_BF16, TOL_MXFP8, F32View, atom_byte, rel_err, tile_slot, to_device, to_f64

pytestmark = pytest.mark.gpu


def _run(cfg, inp, mode):
    import torch
    from mixture_experts_layer_18_gb300.layer import MoELayer
    L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.I, cfg.k, mode=mode)
    io = L.empty_io()
    dev = {k: to_device(v) for k, v in inp.items()}
    L.route(dev["logits"])
    L.forward(dev["X"], dev["W13"], dev["W2"], io["Y"])
    L.backward(dev["dY"], dev["W13"], dev["W2"], io["dX"], io["dW13"], io["dW2"], io["dgate"])
    torch.cuda.synchronize()
    assert L.device_status() == 0
    return L, io


def _oracle_inputs(inp):
    return {k: (F32View(v) if k != "logits" else v) for k, v in inp.items()}


# The block-scaled GEMMs run 192-column tiles over K stages of 128: I is a
# multiple of 384, and H = 256 / 512 leaves a ragged last tile on the H-wide
# outputs.
SMALL = [MoEConfig("mx_a", 512, 256, 8, 2, 384, "bf16"),
         MoEConfig("mx_b", 700, 512, 16, 4, 384, "bf16"),
         MoEConfig("mx_skew", 600, 256, 32, 4, 384, "bf16", skew=True)]


@pytest.mark.parametrize("mode", ["mxfp8", "fp8_bwd"])
@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_small_shapes_full(cfg, mode, x_scale=None):
    inp = make_inputs(cfg)
    if x_scale is not None:
        from workloads import bf16_bits_to_f32
        v = (bf16_bits_to_f32(inp["X"]) * np.float32(x_scale)).astype(np.float32)
        inp["X"] = (v.view(np.uint32) >> 16).astype(np.uint16)
    L, io = _run(cfg, inp, mode)
    oi = _oracle_inputs(inp)
    idx, gate = O.route(inp["logits"], cfg.k)
    Y, saved = O.forward(oi["X"], oi["W13"], oi["W2"], idx, gate, mode=mode, keep=True)
    g = O.backward(oi["X"], oi["W13"], oi["W2"], idx, gate, oi["dY"], mode=mode)
    tol_f = TOL_MXFP8 if mode == "mxfp8" else TOL_BF16
    roa = L.row_of_assign.cpu().numpy()
    h13 = to_f64(L.h13)
    for e, s in saved.items():
        assert rel_err(h13[roa[s["a"]]], s["h"]) <= tol_f, ("h13", e)
    errs = {"Y": rel_err(to_f64(io["Y"]), Y)}
    for k in ("dX", "dW13", "dW2", "dgate"):
        errs[k] = rel_err(to_f64(io[k]), g[k])
    assert errs["Y"] <= tol_f, errs
    for k in ("dX", "dW13", "dW2", "dgate"):
        assert errs[k] <= TOL_MXFP8, (k, errs)
    # the quantised path really differs from the bf16 one (the test would not
    # notice a silent bf16 fallback otherwise)
    gb = O.backward(oi["X"], oi["W13"], oi["W2"], idx, gate, oi["dY"], mode="bf16")
    assert rel_err(g["dW13"], gb["dW13"]) > 1e-3


@pytest.mark.parametrize("mode", ["mxfp8", "fp8_bwd"])
def test_large_preactivations(mode):
    """Inputs scaled by 32 (|u| ~ 150: exp(-u) overflows in the epilogues'
    SiLU and sigmoid; activations ~10^4, still far inside E4M3 x E8M0)."""
    test_small_shapes_full(SMALL[0], mode, x_scale=32.0)


@pytest.mark.parametrize("mode", ["mxfp8", "fp8_bwd"])
def test_small_shapes_single_cta_tiles(mode):
    """The block-scaled GEMMs on single-CTA 128-row tiles (instead of
    256-row tiles over an SM pair) give the same parity."""
    import mixture_experts_layer_18_gb300 as M
    M.moe_set_debug(M.MOE_DEBUG_SINGLE_CTA, 0)
    try:
        test_small_shapes_full(SMALL[1], mode)
    finally:
        M.moe_set_debug(0, 0)


def test_pair_and_single_cta_agree_bitwise():
    """Pair and single-CTA tiles run the same block-scaled MMAs over the same
    K order, so their GEMM results are bit-identical.  d(gate) sums each
    row's products over two column halves on pairs (two epilogue warps per
    row) and in one pass on single CTAs, so it agrees to rounding only."""
    import torch
    import mixture_experts_layer_18_gb300 as M
    cfg = SMALL[2]
    inp = make_inputs(cfg, 4)
    _, a = _run(cfg, inp, "mxfp8")
    M.moe_set_debug(M.MOE_DEBUG_SINGLE_CTA, 0)
    try:
        _, b = _run(cfg, inp, "mxfp8")
    finally:
        M.moe_set_debug(0, 0)
    for k in a:
        if k == "dgate":
            assert rel_err(to_f64(a[k]), to_f64(b[k])) <= 1e-6, k
        else:
            assert torch.equal(a[k], b[k]), k


def test_saved_encodings_bit_exact():
    """The mxfp8 forward leaves in `saved` the backward's encodings of
    X_perm (gathered and quantised in one pass, 32-row blocks per expert
    group) and of W13 / W2 (row-wise, from the same passes as the forward's
    column-wise ones).  Codes and scale bytes equal the oracle's quantiser
    applied to the oracle's own permutation of X and to the weights."""
    from workloads import bf16_bits_to_f32
    cfg = SMALL[2]
    inp = make_inputs(cfg, 6)
    L, _ = _run(cfg, inp, "mxfp8")
    lay, sv = L.layout, L.saved.cpu().numpy()
    rows = L.max_rows
    rp = (rows + 127) // 128 * 128
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    idx, _ = O.route(inp["logits"], k)
    pm = O.permute(idx, E)
    tpad = int(pm["padded_offsets"][-1])
    X = bf16_bits_to_f32(inp["X"]).astype(np.float64)
    aor = pm["assign_of_row"]
    xperm = np.zeros((tpad, H))
    xperm[aor >= 0] = X[aor[aor >= 0] // k]
    cq, cs = O.quantize_mxfp8(xperm, 0, pm["padded_offsets"])
    q = sv[lay.x_col_q: lay.x_col_q + rows * H].reshape(rows, H)[:tpad]
    assert np.array_equal(q, cq)
    rb, c = np.meshgrid(np.arange(tpad // 32), np.arange(H), indexing="ij")
    assert np.array_equal(sv[lay.x_col_sf + atom_byte(c, rb, rp // 128)], cs)
    for name, W, R, C, seg in (("w13_row", inp["W13"], E * H, 2 * I, H),
                               ("w2_row", inp["W2"], E * I, H, I)):
        rq, rs = O.quantize_mxfp8(bf16_bits_to_f32(W).reshape(R, C).astype(np.float64), 1)
        off_q, off_s = getattr(lay, name + "_q"), getattr(lay, name + "_sf")
        assert np.array_equal(sv[off_q: off_q + R * C].reshape(R, C), rq), name
        r, kb = np.meshgrid(np.arange(R), np.arange(C // 32), indexing="ij")
        assert np.array_equal(sv[off_s + atom_byte(tile_slot(r, seg), kb, C // 128)], rs), name


def test_activation_encodings_from_the_epilogue():
    """In mxfp8 mode the gate/up epilogue writes A's MXFP8 encodings itself
    (A is never stored in bf16).  Its column-wise encoding in `saved` (the
    dW2 operand: 32-row blocks per expert group) decodes to the oracle's A
    within the MXFP8 tolerance, and nearly all of its codes and scale bytes
    equal the oracle quantiser's on the oracle's bf16-rounded A (a wrong
    row, column, block or atom index would leave few equal; the rest differ
    where fp32 and fp64 sums round A to different bf16 values)."""
    cfg = SMALL[1]
    inp = make_inputs(cfg, 7)
    L, _ = _run(cfg, inp, "mxfp8")
    assert L.act is None
    lay, sv = L.layout, L.saved.cpu().numpy()
    rows = L.max_rows
    rp = (rows + 127) // 128 * 128
    I = cfg.I
    oi = _oracle_inputs(inp)
    idx, gate = O.route(inp["logits"], cfg.k)
    _, saved = O.forward(oi["X"], oi["W13"], oi["W2"], idx, gate, mode="mxfp8", keep=True)
    pm = O.permute(idx, cfg.E)
    tpad = int(pm["padded_offsets"][-1])
    A = np.zeros((tpad, I))
    for e, s in saved.items():
        A[pm["row_of_assign"][s["a"]]] = s["A"]
    cq, cs = O.quantize_mxfp8(O.bf16_round(A), 0, pm["padded_offsets"])
    q = sv[lay.act_col_q: lay.act_col_q + rows * I].reshape(rows, I)[:tpad]
    rb, c = np.meshgrid(np.arange(tpad // 32), np.arange(I), indexing="ij")
    sf = sv[lay.act_col_sf + atom_byte(c, rb, rp // 128)]
    assert (q == cq).mean() >= 0.95, (q == cq).mean()
    assert (sf == cs).mean() >= 0.98, (sf == cs).mean()
    # element error of the MX rule: at most 1/8 of the block maximum (values
    # past 448 * 2^s saturate: s = floor(log2(amax)) - 8), plus bf16 rounding
    assert rel_err(O.dequantize_mxfp8(q, sf, 0), A) <= 0.13


def _dw_experts(counts, rng):
    """The largest expert, the smallest non-empty one, one whose count is not
    a multiple of 32 (a partial token block) and a random non-empty one."""
    nz = np.nonzero(counts)[0]
    ex = [int(np.argmax(counts)), int(nz[np.argmin(counts[nz])])]
    odd = [int(e) for e in nz if counts[e] % 32 and int(e) not in ex]
    ex.append(odd[0])
    rest = [int(e) for e in nz if int(e) not in ex]
    ex.append(int(rng.choice(rest)))
    return ex


def _check_full_size(cfg, mode, n_tokens=64):
    """Full-size layer in an MXFP8 mode, in the launch configuration the
    benchmark times, against the oracle on sampled rows: Y, dX and d(gate)
    of ``n_tokens`` tokens (every slot of each) and dW13 / dW2 of four
    experts, element by element.  The oracle runs as per-expert sub-batches
    in a spawned process pool (``_oracle_jobs``)."""
    import _oracle_jobs
    inp = make_inputs(cfg)
    L, io = _run(cfg, inp, mode)
    idx, gate = O.route(inp["logits"], cfg.k)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    assert np.array_equal(L.counts.cpu().numpy(), counts)
    rng = np.random.default_rng(2)
    tokens = np.sort(rng.choice(cfg.T, n_tokens, replace=False))
    dw_experts = _dw_experts(counts, rng)
    Y, dX, dg, dws = _oracle_jobs.run_sampled(inp, idx, gate, tokens, dw_experts, mode)
    tol_f = TOL_MXFP8 if mode == "mxfp8" else TOL_BF16
    errs = {"Y": rel_err(to_f64(io["Y"][tokens]), Y),
            "dX": rel_err(to_f64(io["dX"][tokens]), dX),
            "dgate": rel_err(to_f64(io["dgate"][tokens]), dg)}
    for e in dw_experts:
        errs[f"dW13[{e}]"] = rel_err(to_f64(io["dW13"][e]), dws[e][0])
        errs[f"dW2[{e}]"] = rel_err(to_f64(io["dW2"][e]), dws[e][1])
    assert errs["Y"] <= tol_f, errs
    for k, v in errs.items():
        assert v <= TOL_MXFP8, (k, v, errs)
    for e in np.nonzero(counts == 0)[0]:
        assert (to_f64(io["dW13"][int(e)]) == 0).all() and (to_f64(io["dW2"][int(e)]) == 0).all()
    return errs


@pytest.mark.parametrize("mode", ["mxfp8", "fp8_bwd"])
def test_full_size_235b_sampled(mode):
    """235B layer shape: 64 tokens and four experts (largest, smallest, one
    with a partial 32-row token block, one at random)."""
    _check_full_size(CONFIGS["235b_mxfp8"], mode)


def test_full_size_30b_zipf_mxfp8():
    """30B shape with Zipf-skewed routing in mxfp8 mode: experts holding
    nearly every token and eight empty ones go through the block-scaled
    engine and the group-aware quantisers."""
    import dataclasses
    cfg = dataclasses.replace(CONFIGS["30b_zipf"], modes=("mxfp8",))
    counts = np.bincount(O.route(make_inputs(cfg, parts=("logits",))["logits"], cfg.k)[0].reshape(-1),
                         minlength=cfg.E)
    assert (counts == 0).sum() >= 8 and counts.max() > 16000
    _check_full_size(cfg, "mxfp8")
