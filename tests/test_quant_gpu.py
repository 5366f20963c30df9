"""MXFP8 quantiser on the GPU vs the float64 oracle's quantiser: E4M3 codes
and E8M0 scale bytes bit-exact, row-wise and column-wise, group-aware."""
import json
import os

import numpy as np
import pytest

import mixture_experts_layer_18_gb300 as M
from oracle import moe_oracle as O
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

from _common import atom_byte

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _quant(bits, axis, C=None, group_offsets=None):
    import torch
    R, ld = bits.shape
    C = C or ld
    src = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    q = torch.full((R, C), 0xAB, dtype=torch.uint8, device="cuda")
    sc_shape = (R, C // 32) if axis == 1 else (R // 32, C)
    sc = torch.full(sc_shape, 0xCD, dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    go = None
    G = 0
    if group_offsets is not None:
        go = torch.tensor(group_offsets, dtype=torch.int32, device="cuda")
        G = len(group_offsets) - 1
    rc = M.moe_quantize_mxfp8(src.data_ptr(), R, C, ld, axis, go.data_ptr() if go is not None else None,
                              G, q.data_ptr(), sc.data_ptr(), status.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == M.MOE_OK
    torch.cuda.synchronize()
    return q.cpu().numpy(), sc.cpu().numpy(), int(status[0].item())


def _draw(R, C, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, C)).astype(np.float32)
    x *= np.exp2(rng.integers(-40, 40, size=(R, 1))).astype(np.float32)   # wide range per row
    x[rng.random((R, C)) < 0.05] *= np.float32(2.0 ** -30)                # tiny values in blocks
    x[: min(R, 3), :32] = 0.0                                              # all-zero blocks
    return f32_to_bf16_bits(x)


@pytest.mark.parametrize("R,C", [(64, 256), (100, 96), (1, 32), (513, 4096)])
def test_rowwise_bit_exact(R, C):
    bits = _draw(R, C, R + C)
    q, sc, st = _quant(bits, 1)
    assert st == 0
    rq, rs = O.quantize_mxfp8(bf16_bits_to_f32(bits), 1)
    assert np.array_equal(sc, rs)
    assert np.array_equal(q, rq)


@pytest.mark.parametrize("R,C", [(64, 256), (96, 34), (4096, 512)])
def test_colwise_bit_exact(R, C):
    bits = _draw(R, C, 3 * R + C)
    q, sc, st = _quant(bits, 0)
    assert st == 0
    rq, rs = O.quantize_mxfp8(bf16_bits_to_f32(bits), 0)
    assert np.array_equal(sc, rs)
    assert np.array_equal(q, rq)


def test_row_pitch_larger_than_width():
    bits = _draw(64, 128, 7)
    q, sc, st = _quant(bits, 1, C=64)
    rq, rs = O.quantize_mxfp8(bf16_bits_to_f32(bits[:, :64]), 1)
    assert st == 0 and np.array_equal(q, rq) and np.array_equal(sc, rs)


def test_colwise_groups_stop_at_last_offset():
    bits = _draw(256, 64, 11)
    go = [0, 64, 64, 160]          # an empty group; rows >= 160 untouched
    q, sc, st = _quant(bits, 0, group_offsets=go)
    assert st == 0
    rq, rs = O.quantize_mxfp8(bf16_bits_to_f32(bits), 0, go)
    assert np.array_equal(q[:160], rq[:160]) and np.array_equal(sc[:5], rs[:5])
    assert (q[160:] == 0xAB).all() and (sc[5:] == 0xCD).all()


def test_colwise_unaligned_group_offset_reported():
    bits = _draw(128, 32, 12)
    _, _, st = _quant(bits, 0, group_offsets=[0, 40, 128])
    assert st == M.MOE_ERR_INVALID_ARG


def test_golden_blocks_on_gpu():
    """The hand-derived MXFP8 fixture, through the CUDA quantiser."""
    with open(os.path.join(GOLDEN, "mxfp8_blocks.json")) as f:
        cases = json.load(f)["cases"]
    rows = []
    for case in cases:
        vals = np.zeros(32, np.float32)
        vals[: len(case["values"])] = [float(v) for v in case["values"]]
        rows.append(vals)
    bits = f32_to_bf16_bits(np.stack(rows))
    assert np.array_equal(bf16_bits_to_f32(bits), np.stack(rows))   # fixture values are bf16-exact
    q, sc, st = _quant(bits, 1)
    assert st == 0
    for i, case in enumerate(cases):
        assert int(sc[i, 0]) == case["scale"], case["name"]
        want = [int(c, 16) for c in case["codes"]]
        assert list(q[i, : len(want)]) == want, case["name"]


def _dual(bits, rows_limit=None):
    import torch
    R, C = bits.shape
    src = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    Rp = (R + 127) // 128 * 128
    qr = torch.full((R, C), 0xAB, dtype=torch.uint8, device="cuda")
    qc = torch.full((R, C), 0xAB, dtype=torch.uint8, device="cuda")
    sr = torch.full((Rp * C // 32,), 0xCD, dtype=torch.uint8, device="cuda")
    sc = torch.full((Rp * C // 32,), 0xCD, dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    lim = torch.tensor([rows_limit], dtype=torch.int32, device="cuda") if rows_limit is not None else None
    rc = M.moe_quantize_mxfp8_dual(src.data_ptr(), R, C, C, lim.data_ptr() if lim is not None else None,
                                   qr.data_ptr(), sr.data_ptr(), qc.data_ptr(), sc.data_ptr(),
                                   status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == M.MOE_OK
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    return qr.cpu().numpy(), sr.cpu().numpy(), qc.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("R,C", [(32, 128), (256, 384), (96, 256), (1024, 1024)])
def test_dual_bit_exact(R, C):
    """Row-wise and column-wise encodings from the one-read kernel equal the
    oracle's, codes and scale bytes (unpacked from the atom layout)."""
    bits = _draw(R, C, 5 * R + C)
    x = bf16_bits_to_f32(bits)
    qr, sr, qc, sc = _dual(bits)
    rq, rs = O.quantize_mxfp8(x, 1)          # [R, C], [R, C/32]
    cq, cs = O.quantize_mxfp8(x, 0)          # [R, C], [R/32, C]
    assert np.array_equal(qr, rq)
    assert np.array_equal(qc, cq)
    r, kb = np.meshgrid(np.arange(R), np.arange(C // 32), indexing="ij")
    assert np.array_equal(sr[atom_byte(r, kb, C // 128)], rs)
    rb, c = np.meshgrid(np.arange(R // 32), np.arange(C), indexing="ij")
    assert np.array_equal(sc[atom_byte(c, rb, (R + 127) // 128)], cs)


def test_dual_rows_limit_leaves_the_rest():
    bits = _draw(256, 128, 9)
    qr, sr, qc, sc = _dual(bits, rows_limit=96)
    x = bf16_bits_to_f32(bits[:96])
    rq, _ = O.quantize_mxfp8(x, 1)
    cq, _ = O.quantize_mxfp8(x, 0)
    assert np.array_equal(qr[:96], rq) and np.array_equal(qc[:96], cq)
    assert (qr[96:] == 0xAB).all() and (qc[96:] == 0xAB).all()
