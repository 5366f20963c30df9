"""The library's timing hooks (moe_set_gemm_events, moe_set_gemm_launch_events)
record the caller's CUDA events around the grouped-GEMM launches of exactly
the next call of a kind, and nothing after it."""
import pytest

from workloads import MoEConfig, make_inputs

from _common import to_device

pytestmark = pytest.mark.gpu

CFG = MoEConfig("hooks", 512, 256, 8, 2, 384, "bf16")


@pytest.mark.parametrize("mode", ["bf16", "mxfp8"])
def test_bracket_and_per_launch_events(mode):
    import torch

    import mixture_experts_layer_18_gb300 as M
    from mixture_experts_layer_18_gb300.layer import MoELayer
    L = MoELayer(CFG.T, CFG.H, CFG.E, CFG.I, CFG.k, mode=mode)
    io = L.empty_io()
    d = {k: to_device(v) for k, v in make_inputs(CFG).items()}

    def step():
        L.route(d["logits"])
        L.forward(d["X"], d["W13"], d["W2"], io["Y"])
        L.backward(d["dY"], d["W13"], d["W2"], io["dX"], io["dW13"], io["dW2"], io["dgate"])

    step()
    torch.cuda.synchronize()

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record()             # materialise the handle
        return e

    for which in (M.MOE_WS_FORWARD, M.MOE_WS_BACKWARD):
        br = (ev(), ev())
        per = [(ev(), ev()) for _ in range(2)]
        spare = (ev(), ev())   # a third pair: only two launches per call, never recorded
        torch.cuda.synchronize()
        M.moe_set_gemm_events(which, br[0].cuda_event, br[1].cuda_event)
        M.moe_set_gemm_launch_events(which, [a.cuda_event for a, _ in per + [spare]],
                                     [b.cuda_event for _, b in per + [spare]])
        mark = ev()            # recorded on the stream before the call
        step()
        torch.cuda.synchronize()
        assert L.device_status() == 0
        bracket = br[0].elapsed_time(br[1])
        launches = [a.elapsed_time(b) for a, b in per]
        assert all(t > 0 for t in launches)
        assert sum(launches) <= bracket * 1.01 + 1e-3
        assert per[0][1].elapsed_time(per[1][0]) >= 0   # in launch order
        assert mark.elapsed_time(br[0]) >= 0             # recorded by this call
        assert spare[0].elapsed_time(spare[1]) >= 0 and spare[1].elapsed_time(mark) >= 0
        # the hooks fired once: a further call records nothing
        stamp = [b.elapsed_time(br[1]) for b in (br[0],)]
        step()
        torch.cuda.synchronize()
        assert [b.elapsed_time(br[1]) for b in (br[0],)] == stamp
