"""Seeded synthetic inputs for the dropless MoE expert layer.

This module only draws random numbers and stores them; it holds none of the
layer's arithmetic (no routing, no GEMM, no quantisation).  Both the float64
oracle (tests only) and the CUDA path are fed from here, so the two sides see
the same bytes.

Workloads (the shapes of the per-layer benchmark in "Prime Intellect releases
Prime Mega MoE" (MarkTechPost), table "One MoE layer": 128 experts, top-8,
random routing, 16 384-token sequences):

  tiny        T=256,   H=128,  E=8,   k=2, I=64,   fp32
  30b         T=16384, H=2048, E=128, k=8, I=768,  bf16  (Qwen3-30B-A3B shape)
  30b_zipf    as 30b, router logits skewed: Zipf(s=1.2) expert loads over a
              random expert permutation, 8 experts forced to zero tokens
  235b        T=16384, H=4096, E=128, k=8, I=1536, bf16  (Qwen3-235B-A22B shape)
  235b_mxfp8  235b shapes, run in the MXFP8 and fp8_bwd modes

Value recipe: X ~ N(0,1); W13 ~ N(0, 1/H); W2 ~ N(0, 1/I) (fan-in);
logits ~ N(0,1) in fp32; dY ~ N(0,1).  bf16 tensors are fp32 draws rounded to
nearest-even and are returned as uint16 bit patterns.  Every tensor has its
own stream, numpy ``default_rng([seed, tensor_id])``, so any one tensor can be
regenerated alone.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "MoEConfig", "CONFIGS", "make_inputs", "f32_to_bf16_bits",
    "bf16_bits_to_f32", "zipf_targets",
]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    dtype: str            # storage type of X, W13, W2, Y, dY: "f32" or "bf16"
    skew: bool = False    # Zipf-skewed router logits with forced-empty experts
    modes: tuple = ("bf16",)

    @property
    def n_assign(self) -> int:
        return self.T * self.k

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs: GEMM1 (2*N_a*H*2I) + GEMM2 (2*N_a*I*H)."""
        return 6.0 * self.n_assign * self.H * self.I

    def bwd_flops(self) -> float:
        """Algorithmic backward FLOPs: dH, dX, dW13, dW2 GEMMs (12*N_a*H*I)."""
        return 12.0 * self.n_assign * self.H * self.I


CONFIGS = {
    "tiny": MoEConfig("tiny", 256, 128, 8, 2, 64, "f32", modes=("f32",)),
    "30b": MoEConfig("30b", 16384, 2048, 128, 8, 768, "bf16"),
    "30b_zipf": MoEConfig("30b_zipf", 16384, 2048, 128, 8, 768, "bf16", skew=True),
    "235b": MoEConfig("235b", 16384, 4096, 128, 8, 1536, "bf16"),
    "235b_mxfp8": MoEConfig("235b_mxfp8", 16384, 4096, 128, 8, 1536, "bf16",
                            modes=("mxfp8", "fp8_bwd")),
}

_TENSOR_ID = {"logits": 1, "X": 2, "W13": 3, "W2": 4, "dY": 5, "skew": 6}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits.

    Inputs here are finite normal draws, so no NaN handling is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng([seed, _TENSOR_ID[name]])


def _normal(rng, shape, std, as_bf16, chunk_rows=None):
    """N(0, std^2) draws, fp32 or bf16 bits, generated in row chunks."""
    shape = tuple(shape)
    out = np.empty(shape, dtype=np.uint16 if as_bf16 else np.float32)
    rows = shape[0]
    step = chunk_rows or rows
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        v = rng.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(v) if as_bf16 else v
    return out


def zipf_targets(n_live: int, total: int, cap: int, s: float = 1.2) -> np.ndarray:
    """Per-expert target loads proportional to rank^-s, water-filled so that no
    expert exceeds ``cap`` rows (a token can pick an expert at most once)."""
    w = np.arange(1, n_live + 1, dtype=np.float64) ** (-s)
    tgt = np.zeros(n_live)
    free = np.ones(n_live, dtype=bool)
    remaining = float(total)
    while True:
        share = remaining * w * free / w[free].sum()
        over = free & (share > cap)
        if not over.any():
            tgt[free] = share[free]
            return tgt
        tgt[over] = cap
        free &= ~over
        remaining = total - tgt[~free].sum()


def _skew_bias(noise: np.ndarray, k: int, seed: int, n_empty: int = 8,
               iters: int = 120) -> np.ndarray:
    """Per-expert logit bias giving Zipf(1.2) loads and ``n_empty`` experts
    that are never picked.  The bias is tuned by damped fixed-point steps on the
    same noise; the loads are counted with numpy's argpartition.  Only the
    resulting logits matter downstream (they are the parity input)."""
    T, E = noise.shape
    perm = _rng(seed, "skew").permutation(E)
    empty, live = perm[:n_empty], perm[n_empty:]
    target = np.zeros(E)
    target[live] = zipf_targets(len(live), T * k, T)
    b = np.zeros(E, dtype=np.float64)
    b[empty] = -np.inf
    for _ in range(iters):
        lg = noise + b.astype(np.float32)
        sel = np.argpartition(-lg, k - 1, axis=1)[:, :k]
        cnt = np.bincount(sel.reshape(-1), minlength=E).astype(np.float64)
        b[live] += 0.5 * np.log((target[live] + 1.0) / (cnt[live] + 1.0))
        b[live] -= b[live].mean()
    return b.astype(np.float32)


def make_inputs(cfg: MoEConfig, seed: int = 0,
                parts=("logits", "X", "W13", "W2", "dY")) -> dict:
    """Draw the requested tensors of one workload.

    Returns numpy arrays: ``logits`` fp32 [T,E]; ``X`` [T,H], ``W13`` [E,H,2I],
    ``W2`` [E,I,H], ``dY`` [T,H] as fp32 (cfg.dtype == "f32") or uint16 bf16
    bits (cfg.dtype == "bf16")."""
    bf = cfg.dtype == "bf16"
    T, H, E, I = cfg.T, cfg.H, cfg.E, cfg.I
    out = {}
    for name in parts:
        rng = _rng(seed, name)
        if name == "logits":
            lg = rng.standard_normal((T, E), dtype=np.float32)
            if cfg.skew:
                lg = lg + _skew_bias(lg, cfg.k, seed)[None, :]
            out[name] = np.ascontiguousarray(lg, dtype=np.float32)
        elif name == "X":
            out[name] = _normal(rng, (T, H), 1.0, bf, 4096)
        elif name == "W13":
            out[name] = _normal(rng, (E, H, 2 * I), H ** -0.5, bf, 4)
        elif name == "W2":
            out[name] = _normal(rng, (E, I, H), I ** -0.5, bf, 4)
        elif name == "dY":
            out[name] = _normal(rng, (T, H), 1.0, bf, 4096)
        else:
            raise KeyError(name)
    return out
