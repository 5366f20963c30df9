"""Router backward (d(logits) from d(gate) through the renormalised top-k
softmax) on the GPU vs the float64 oracle (pinned by finite differences)."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from workloads import CONFIGS, make_inputs

from _common import to_device

pytestmark = pytest.mark.gpu


def _run(logits, k, dgate):
    import torch
    from mixture_experts_layer_18_gb300.layer import MoELayer
    T, E = logits.shape
    L = MoELayer(T, 64, E, 64, k, mode="bf16", backward=False)
    L.route(to_device(logits))
    dl = torch.full((T, E), 7.0, dtype=torch.float32, device="cuda")
    L.route_backward(to_device(dgate.astype(np.float32)), dl)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    return dl.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(300, 8, 2), (129, 128, 8), (64, 1000, 32), (77, 3, 1)])
def test_route_backward_matches_oracle(T, E, k):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    dg = rng.standard_normal((T, k))
    got = _run(lg, k, dg)
    idx, gate = O.route(lg, k)
    ref = O.route_backward(gate, idx, dg.astype(np.float32), E)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()
    assert (got[ref == 0] == 0).all()          # unselected experts exactly zero


def test_route_backward_workload_30b_zipf():
    cfg = CONFIGS["30b_zipf"]
    lg = make_inputs(cfg, parts=("logits",))["logits"]
    dg = np.random.default_rng(3).standard_normal((cfg.T, cfg.k))
    got = _run(lg, cfg.k, dg)
    idx, gate = O.route(lg, cfg.k)
    ref = O.route_backward(gate, idx, dg.astype(np.float32), cfg.E)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()
    # softmax-Jacobian property: each row of d(logits) sums to zero
    assert np.abs(got.astype(np.float64).sum(1)).max() <= 1e-5 * np.abs(ref).max() * cfg.k
