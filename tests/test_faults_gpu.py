"""Device-side failure reporting without a GPU fault: bounded waits that run
out report MOE_ERR_TIMEOUT and return; corrupted index maps are caught by the
kernels' own bounds checks (MOE_ERR_BAD_INDEX, access skipped).  After each
case the context must still run a correct step."""
import numpy as np
import pytest

import mixture_experts_layer_18_gb300 as M
from oracle import moe_oracle as O
from workloads import MoEConfig, make_inputs

from _common import TOL_BF16, F32View, rel_err, to_device, to_f64

pytestmark = pytest.mark.gpu

CFG = MoEConfig("fault", 512, 256, 8, 2, 256, "bf16")


def _setup():
    from mixture_experts_layer_18_gb300.layer import MoELayer
    inp = make_inputs(CFG)
    L = MoELayer(CFG.T, CFG.H, CFG.E, CFG.I, CFG.k, mode="bf16")
    io = L.empty_io()
    dev = {k: to_device(v) for k, v in inp.items()}
    return inp, L, io, dev


def _step(L, io, dev):
    L.route(dev["logits"])
    L.forward(dev["X"], dev["W13"], dev["W2"], io["Y"])
    L.backward(dev["dY"], dev["W13"], dev["W2"], io["dX"], io["dW13"], io["dW2"], io["dgate"])


def _check_correct(inp, io):
    oi = {k: (F32View(v) if k != "logits" else v) for k, v in inp.items()}
    idx, gate = O.route(inp["logits"], CFG.k)
    Y = O.forward(oi["X"], oi["W13"], oi["W2"], idx, gate)
    g = O.backward(oi["X"], oi["W13"], oi["W2"], idx, gate, oi["dY"])
    assert rel_err(to_f64(io["Y"]), Y) <= TOL_BF16
    for k in ("dX", "dW13", "dW2", "dgate"):
        assert rel_err(to_f64(io[k]), g[k]) <= TOL_BF16, k


@pytest.mark.parametrize("flags", [0, M.MOE_DEBUG_SINGLE_CTA])
def test_wait_that_never_ends_reports_timeout(flags):
    import torch
    inp, L, io, dev = _setup()
    try:
        M.moe_set_debug(flags | M.MOE_DEBUG_NEVER_READY, 2_000_000)   # 2 ms limit
        L.clear_status()
        _step(L, io, dev)
        torch.cuda.synchronize()
        assert L.device_status() == M.MOE_ERR_TIMEOUT
    finally:
        M.moe_set_debug(flags, 0)
    L.clear_status()
    _step(L, io, dev)
    torch.cuda.synchronize()
    M.moe_set_debug(0, 0)
    assert L.device_status() == 0
    _check_correct(inp, io)


def test_corrupted_maps_report_bad_index():
    import torch
    inp, L, io, dev = _setup()
    L.route(dev["logits"])
    torch.cuda.synchronize()
    roa_ok = L.row_of_assign.clone()
    aor_ok = L.assign_of_row.clone()
    L.row_of_assign[5] = 1 << 30                          # read by the combines, d(gate) reduce
    L.assign_of_row[int(roa_ok[9])] = CFG.T * CFG.k + 7   # read by the gathers and epilogues
    L.clear_status()
    L.forward(dev["X"], dev["W13"], dev["W2"], io["Y"])
    L.backward(dev["dY"], dev["W13"], dev["W2"], io["dX"], io["dW13"], io["dW2"], io["dgate"])
    torch.cuda.synchronize()
    assert L.device_status() == M.MOE_ERR_BAD_INDEX
    assert bool(torch.isfinite(io["Y"].float()).all())
    # the context is intact: a clean step is exact again
    L.row_of_assign.copy_(roa_ok)
    L.assign_of_row.copy_(aor_ok)
    L.clear_status()
    _step(L, io, dev)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    _check_correct(inp, io)


def test_invalid_arguments_rejected_before_launch():
    import torch
    inp, L, io, dev = _setup()
    d = M.moe_dims(CFG.T, CFG.H, CFG.E, CFG.I, CFG.k, M.MOE_BF16, 1)
    # misaligned output pointer
    rc = M.moe_forward(d, dev["X"].data_ptr(), dev["W13"].data_ptr(), dev["W2"].data_ptr(),
                       L.route_out, io["Y"].data_ptr() + 2, L.saved.data_ptr(), L.saved.numel(),
                       L.ws_fwd.data_ptr(), L.ws_fwd.numel(), L.status.data_ptr(), None)
    assert rc == M.MOE_ERR_INVALID_ARG
    # short workspace
    rc = M.moe_backward(d, dev["dY"].data_ptr(), dev["W13"].data_ptr(), dev["W2"].data_ptr(),
                        L.route_out, L.saved.data_ptr(), L.saved.numel(), io["dX"].data_ptr(),
                        io["dW13"].data_ptr(), io["dW2"].data_ptr(), io["dgate"].data_ptr(),
                        L.ws_bwd.data_ptr(), 1024, L.status.data_ptr(), None)
    assert rc == M.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert L.device_status() == 0


@pytest.mark.parametrize("flags", [0, M.MOE_DEBUG_ONE_LAUNCH_BACKWARD])
def test_backward_while_half_the_gpu_is_busy(flags):
    """A bounded side kernel on another stream holds about half of the SMs
    (one block with 200 KB of shared memory per SM, 76 blocks, 300 ms) while
    a whole step runs with a 20 ms device wait limit: status 0 and oracle
    parity, both for the default backward (two co-scheduled launches, no
    tile waits on another CTA) and for the one-launch form, whose dX / dW13
    tiles wait on D tiles of other CTAs, so its launch must not start on the
    SMs that happen to be free and then wait for CTAs that cannot be placed
    (a cooperative launch)."""
    import torch
    from mixture_experts_layer_18_gb300.layer import MoELayer
    cfg = MoEConfig("busy", 4096, 1024, 16, 4, 512, "bf16")
    inp = make_inputs(cfg, 1)
    L = MoELayer(cfg.T, cfg.H, cfg.E, cfg.I, cfg.k, mode="bf16")
    io = L.empty_io()
    dev = {k: to_device(v) for k, v in inp.items()}
    _step(L, io, dev)
    torch.cuda.synchronize()
    assert L.device_status() == 0
    side = torch.cuda.Stream()
    try:
        M.moe_set_debug(flags, 20_000_000)
        L.clear_status()
        torch.cuda.synchronize()
        assert M.moe_debug_occupy(76, 200 * 1024, 300_000_000, side.cuda_stream) == M.MOE_OK
        _step(L, io, dev)
        torch.cuda.synchronize()
    finally:
        M.moe_set_debug(0, 0)
    assert L.device_status() == 0
    oi = {k: (F32View(v) if k != "logits" else v) for k, v in inp.items()}
    idx, gate = O.route(inp["logits"], cfg.k)
    tokens = np.arange(0, cfg.T, 97)
    Y = O.forward(oi["X"], oi["W13"], oi["W2"], idx, gate, tokens=tokens)
    g = O.backward(oi["X"], oi["W13"], oi["W2"], idx, gate, oi["dY"], tokens=tokens,
                   experts=[0, 9])
    assert rel_err(to_f64(io["Y"][tokens]), Y) <= TOL_BF16
    assert rel_err(to_f64(io["dX"][tokens]), g["dX"]) <= TOL_BF16
    assert rel_err(to_f64(io["dgate"][tokens]), g["dgate"]) <= TOL_BF16
    for i, e in enumerate([0, 9]):
        assert rel_err(to_f64(io["dW13"][e]), g["dW13"][i]) <= TOL_BF16
        assert rel_err(to_f64(io["dW2"][e]), g["dW2"][i]) <= TOL_BF16


def test_occupy_hook_rejects_unbounded_requests():
    assert M.moe_debug_occupy(0, 0, 1000, None) == M.MOE_ERR_INVALID_ARG
    assert M.moe_debug_occupy(4, 300 * 1024, 1000, None) == M.MOE_ERR_INVALID_ARG
    assert M.moe_debug_occupy(4, 1024, 2_000_000_000, None) == M.MOE_ERR_INVALID_ARG


def test_one_launch_backward_matches_two_launches():
    """The one-launch co-scheduled backward (readiness counters) and the
    default two launches run the same tiles on the same operands: identical
    results bit for bit."""
    import torch
    inp, L, io, dev = _setup()
    _step(L, io, dev)
    torch.cuda.synchronize()
    a = {k: v.clone() for k, v in io.items()}
    try:
        M.moe_set_debug(M.MOE_DEBUG_ONE_LAUNCH_BACKWARD, 0)
        _step(L, io, dev)
        torch.cuda.synchronize()
    finally:
        M.moe_set_debug(0, 0)
    assert L.device_status() == 0
    for k in a:
        assert torch.equal(a[k], io[k]), k
