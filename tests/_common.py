"""Helpers shared by the GPU parity tests: moving seeded workload arrays to
the device and giving the oracle float views of bf16 bit arrays."""
from __future__ import annotations

import numpy as np

from workloads import bf16_bits_to_f32

TOL_BF16 = 2e-2     # max|err| / max|ref| for bf16 (and TF32) outputs and gradients
TOL_MXFP8 = 6e-2    # same measure for the MXFP8 GEMM paths
TOL_GATE = 2e-6     # absolute, fp32 gates in (0, 1]


class F32View:
    """Read-only float32 view of a uint16 bf16 array (or a float32 array):
    indexing converts only the selected part."""

    def __init__(self, arr):
        self.arr = arr
        self.shape = arr.shape

    def _conv(self, x):
        return bf16_bits_to_f32(x) if x.dtype == np.uint16 else np.asarray(x, np.float32)

    def __getitem__(self, idx):
        return self._conv(self.arr[idx])

    def __array__(self, dtype=None, copy=None):
        out = self._conv(self.arr)
        return out.astype(dtype) if dtype is not None else out


def to_device(arr, device="cuda"):
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_f64(t):
    """Device tensor -> float64 numpy."""
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / den)


def atom_byte(mn, kb, kgroups):
    """Byte of (MN index, 32-element K block) in the tensor-core scale atoms
    (512-byte atoms of 128 MN indices x 4 K blocks), as declared in moe.h."""
    mn = np.asarray(mn)
    kb = np.asarray(kb)
    return ((mn // 128) * kgroups + kb // 4) * 512 + (mn % 32) * 16 + ((mn // 32) % 4) * 4 + kb % 4


def tile_slot(mn, seg):
    """Scale slot of B-operand index mn of the block-scaled GEMMs, as declared
    in moe.h: each segment of `seg` indices is cut into 192-wide tiles and
    each tile owns 256 slots (two atoms)."""
    mn = np.asarray(mn)
    e, m = mn // seg, mn % seg
    return e * (-(-seg // 192) * 256) + (m // 192) * 256 + m % 192
