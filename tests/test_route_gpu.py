"""Router and permutation builder on the GPU vs the float64 oracle: indices,
counts, offsets and row maps bit-exact; gates within fp32 rounding."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from workloads import CONFIGS, make_inputs

from _common import TOL_GATE, to_device

pytestmark = pytest.mark.gpu


def _run_route(logits_np, E, k, H=64, I=64, status=0):
    import torch
    from mixture_experts_layer_18_gb300.layer import MoELayer
    T = logits_np.shape[0]
    L = MoELayer(T, H, E, I, k, mode="bf16", backward=False)
    L.assign_of_row.fill_(12345)
    lg = to_device(logits_np) if T else torch.empty((0, E), device="cuda")
    L.route(lg)
    torch.cuda.synchronize()
    assert L.device_status() == status
    return L


def _check(L, logits_np, E, k):
    idx, gate = O.route(logits_np, k)
    p = O.permute(idx, E)
    T = logits_np.shape[0]
    assert np.array_equal(L.topk_idx.cpu().numpy(), idx)
    if T:
        assert np.abs(L.gate.cpu().numpy() - gate).max() <= TOL_GATE
    assert np.array_equal(L.counts.cpu().numpy(), p["counts"])
    assert np.array_equal(L.offsets.cpu().numpy(), p["offsets"])
    assert np.array_equal(L.padded_offsets.cpu().numpy(), p["padded_offsets"])
    assert np.array_equal(L.row_of_assign.cpu().numpy(), p["row_of_assign"])
    aor = L.assign_of_row.cpu().numpy()
    tpad = int(p["padded_offsets"][-1])
    assert np.array_equal(aor[:tpad], p["assign_of_row"])
    assert (aor[tpad:] == -1).all()


@pytest.mark.parametrize("name", ["tiny", "30b", "30b_zipf", "235b"])
def test_route_workloads_bit_exact(name):
    cfg = CONFIGS[name]
    lg = make_inputs(cfg, parts=("logits",))["logits"]
    L = _run_route(lg, cfg.E, cfg.k)
    _check(L, lg, cfg.E, cfg.k)
    if cfg.skew:
        assert (L.counts.cpu().numpy() == 0).sum() >= 8


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (130, 16, 4), (129, 128, 8), (300, 3, 3),
                                   (77, 1, 1), (513, 64, 1), (200, 256, 8), (64, 1000, 32)])
def test_route_edge_shapes(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    L = _run_route(lg, E, k)
    _check(L, lg, E, k)


def test_route_ties_and_neg_inf():
    rng = np.random.default_rng(5)
    lg = rng.integers(-2, 3, size=(400, 32)).astype(np.float32)   # many exact ties
    lg[:, 7] = -np.inf
    lg[:10] = 0.0                                                   # rows of all-equal logits
    lg[10:20, :] = -np.inf
    lg[10:20, 3] = 1.0                                              # one finite expert
    L = _run_route(lg, 32, 4)
    _check(L, lg, 32, 4)


def test_route_empty_batch():
    L = _run_route(np.zeros((0, 16), np.float32), 16, 2)
    assert (L.counts.cpu().numpy() == 0).all()
    assert (L.padded_offsets.cpu().numpy() == 0).all()
    assert (L.assign_of_row.cpu().numpy() == -1).all()


def test_route_is_deterministic():
    cfg = CONFIGS["30b"]
    lg = make_inputs(cfg, parts=("logits",))["logits"]
    a = _run_route(lg, cfg.E, cfg.k)
    b = _run_route(lg, cfg.E, cfg.k)
    for name in ("topk_idx", "gate", "row_of_assign", "assign_of_row", "padded_offsets"):
        assert np.array_equal(getattr(a, name).cpu().numpy(), getattr(b, name).cpu().numpy())


def test_route_inputs_outside_the_softmax_domain():
    """Tokens whose logits are all -inf (zero gates), NaN logits (read as
    -inf) and tokens with fewer than k finite logits: indices and gates as
    the oracle gives them, MOE_ERR_BAD_INPUT in the status word, and the
    permutation still bit-exact."""
    import mixture_experts_layer_18_gb300 as M
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((300, 40)).astype(np.float32)
    lg[3] = -np.inf
    lg[150] = -np.inf
    lg[7, [1, 5, 30]] = np.nan
    lg[200, :] = -np.inf
    lg[200, [9, 2]] = [0.5, 0.5]
    L = _run_route(lg, 40, 4, status=M.MOE_ERR_BAD_INPUT)
    _check(L, lg, 40, 4)
    gate = L.gate.cpu().numpy()
    assert (gate[[3, 150]] == 0).all() and np.isfinite(gate).all()
    assert list(L.topk_idx.cpu().numpy()[3]) == [0, 1, 2, 3]
