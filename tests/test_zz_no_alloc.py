"""moe_route_noalloc: the router / permutation builder for callers that
cannot allocate device memory (for example a plugin inside a framework that
owns all device allocations and offers no workspace, or a latency-critical
loop that must not call cudaMalloc after start-up).  Its scratch is a
library-owned device array, so it must give exactly what moe_route gives with
a caller workspace - on consecutive calls, since the array keeps the previous
call's contents.  Collected last on purpose (file name)."""
import numpy as np
import pytest

import mixture_experts_layer_18_gb300 as M

from _common import to_device

FIELDS = ("topk_idx", "gate", "counts", "offsets", "padded_offsets", "row_of_assign",
          "assign_of_row")


def _bufs(T, E, k):
    import torch
    from mixture_experts_layer_18_gb300.layer import MoELayer
    L = MoELayer(T, 64, E, 64, k, mode="bf16", backward=False)
    for f in FIELDS:
        getattr(L, f).fill_(-7)
    return L


def _noalloc(L, logits):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    lp = logits.data_ptr() if logits.numel() else None
    return M.moe_route_noalloc(L.dims, lp, L.route_out, L.status.data_ptr(), stream)


@pytest.mark.gpu
def test_noalloc_route_matches_workspace_route_twice():
    import torch
    cases = [(16384, 128, 8, 0), (1000, 64, 4, 1)]   # a large call, then a smaller one
    for T, E, k, seed in cases:
        lg = to_device(np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32))
        ref = _bufs(T, E, k)
        ref.route(lg)
        got = _bufs(T, E, k)
        assert _noalloc(got, lg) == M.MOE_OK
        torch.cuda.synchronize()
        assert ref.device_status() == 0 and got.device_status() == 0
        # the same kernels on the same logits: every field, gates included,
        # is identical bit for bit
        for f in FIELDS:
            a = getattr(ref, f).cpu().numpy()
            b = getattr(got, f).cpu().numpy()
            assert np.array_equal(a, b), (T, f)


@pytest.mark.gpu
def test_noalloc_route_rejects_sizes_beyond_its_scratch():
    import torch
    # 2 * E * ceil(T/128) = 2 * 1024 * 128 int32 > 131072: refused before any launch
    L = _bufs(16384, 1024, 8)
    lg = torch.zeros((16384, 1024), device="cuda")
    assert _noalloc(L, lg) == M.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (L.topk_idx == -7).all()
