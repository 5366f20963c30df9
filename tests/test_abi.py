"""The C-ABI library builds, loads and exports every function include/moe.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes

import pytest

import mixture_experts_layer_18_gb300 as M


def test_library_exports_every_header_function():
    names = M.header_functions()
    assert {"moe_route", "moe_forward", "moe_backward", "moe_quantize_mxfp8"} <= set(names)
    lib = M.lib()
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def _dims(**kw):
    base = dict(T=256, H=128, E=8, I=64, top_k=2, mode=M.MOE_F32, save_for_backward=1)
    base.update(kw)
    return M.moe_dims(**base)


@pytest.mark.parametrize("bad", [dict(H=100), dict(I=0), dict(E=0), dict(E=2000), dict(top_k=0),
                                 dict(top_k=9), dict(top_k=40, E=64), dict(T=-1), dict(mode=7)])
def test_invalid_dims_rejected_on_host(bad):
    d = _dims(**bad)
    assert M.moe_max_rows(d) == -1
    assert M.moe_workspace_size(d, M.MOE_WS_FORWARD) == 0
    with pytest.raises(M.MoEError):
        M.moe_saved_layout_of(d)
    out = M.moe_route_out()
    assert M.moe_route(d, None, out, None, 0, None, None) == M.MOE_ERR_INVALID_ARG


def test_sizes_follow_the_documented_layout():
    d = _dims(T=16384, H=4096, E=128, I=1536, top_k=8, mode=M.MOE_BF16)
    rows = 16384 * 8 + 128 * 128
    assert M.moe_max_rows(d) == rows
    lay = M.moe_saved_layout_of(d)
    assert lay.x_perm == 0
    assert lay.h13 >= rows * 4096 * 2 and lay.act >= lay.h13 + rows * 3072 * 2
    assert lay.total >= lay.act + rows * 1536 * 2
    assert M.moe_workspace_size(d, M.MOE_WS_FORWARD) >= rows * 4096 * 2
    # dY_perm, dh13, dXp (bf16 saves gate * A, so no gated copy of dY)
    assert M.moe_workspace_size(d, M.MOE_WS_BACKWARD) >= rows * (2 * 4096 + 3072) * 2
    assert M.moe_workspace_size(d, 99) == 0
    # MXFP8: no X_perm (the dispatch gather writes MXFP8 encodings directly)
    lay8 = M.moe_saved_layout_of(_dims(T=16384, H=4096, E=128, I=1536, top_k=8,
                                       mode=M.MOE_MXFP8))
    assert lay8.x_perm == 0 and lay8.h13 == 0


def _span(lay, name, following):
    """Bytes between a saved-layout field and the next one."""
    return getattr(lay, following) - getattr(lay, name)


@pytest.mark.parametrize("mode, x_perm, act", [
    ("MOE_BF16", True, True), ("MOE_F32", True, True),
    ("MOE_FP8_BWD", True, True),       # its MXFP8 backward quantises X_perm and A
    ("MOE_MXFP8", False, False),       # both exist only as MXFP8 encodings
])
def test_saved_tensors_per_mode(mode, x_perm, act):
    """Which bf16 / fp32 intermediates each mode keeps in `saved` (the
    MXFP8 forward gathers X into its encodings and encodes A in the SwiGLU
    epilogue; moe.h documents the zero-sized fields)."""
    T, H, E, I, k = 1024, 256, 8, 128, 2
    d = _dims(T=T, H=H, E=E, I=I, top_k=k, mode=getattr(M, mode))
    rows = T * k + 128 * E
    es = 4 if mode == "MOE_F32" else 2
    lay = M.moe_saved_layout_of(d)
    assert (_span(lay, "x_perm", "h13") >= rows * H * es) == x_perm
    assert (_span(lay, "x_perm", "h13") == 0) == (not x_perm)
    assert _span(lay, "h13", "act") >= rows * 2 * I * es
    nxt = "x_col_q" if mode == "MOE_MXFP8" else "total"
    assert (_span(lay, "act", nxt) >= rows * I * es) == act
    if mode == "MOE_MXFP8":
        rp = (rows + 127) // 128 * 128
        assert lay.act == lay.x_col_q               # A: no bf16 copy
        assert lay.act_col_q - lay.x_col_q >= rows * H + rp * H // 32
        assert lay.total - lay.w2_row_q >= E * I * H + E * I * H // 32


def test_backward_workspace_per_mode():
    """bf16 gathers dY once (the forward left gate * A for dW2); fp32 keeps
    dY_perm and gate * dY_perm; the MXFP8 modes gather dY into encodings."""
    T, H, E, I, k = 1024, 256, 8, 128, 2
    rows = T * k + 128 * E
    ws = {m: M.moe_workspace_size(_dims(T=T, H=H, E=E, I=I, top_k=k, mode=getattr(M, m)),
                                  M.MOE_WS_BACKWARD)
          for m in ("MOE_BF16", "MOE_F32")}
    # dY_perm + dh13 + dXp (+ partials, counters) in bf16; two dY copies in fp32
    assert ws["MOE_BF16"] >= rows * (2 * H + 2 * I) * 2
    assert ws["MOE_BF16"] < rows * (3 * H + 2 * I) * 2
    assert ws["MOE_F32"] >= rows * (3 * H + 2 * I) * 4


def test_null_and_misaligned_pointers_rejected_on_host():
    d = _dims()
    out = M.moe_route_out(*([256] * 7))        # 16-byte aligned but fake; never launched
    # workspace too small -> rejected before any launch
    assert M.moe_route(d, 256, out, 256, 1, 256, None) == M.MOE_ERR_INVALID_ARG
    out_bad = M.moe_route_out(*([8] * 7))
    assert M.moe_route(d, 256, out_bad, 256, 1 << 20, 256, None) == M.MOE_ERR_INVALID_ARG
    assert M.moe_quantize_mxfp8(None, 32, 30, 30, 1, None, 0, None, None, 256, None) == \
        M.MOE_ERR_INVALID_ARG
    assert M.moe_quantize_mxfp8(None, 31, 32, 32, 0, None, 0, None, None, 256, None) == \
        M.MOE_ERR_INVALID_ARG


def test_status_strings():
    for code in range(7):
        assert M.moe_status_string(code)
    assert M.moe_status_string(42) == "unknown status"
