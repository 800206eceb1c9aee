"""Device memory a layer keeps, against the bytes of the weights it was given.

By default a bf16 layer keeps the decode kernel's per-feature records and the
grouped GEMMs' row layouts (about twice the expert bytes). With
MOE_FLAG_ONE_WEIGHT_COPY a bf16 layer the record-streaming kernel serves
(hidden <= 2048) keeps the records alone, which the grouped tensor-core path then
reads too: resident weight bytes within 1.1x the logical weight bytes (fp32
router, bf16 routed and shared experts), both paths still matching the oracle.
The layer's own count is checked against the device's free memory.
"""
import pytest

import moe_inputs as mi
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ONE_COPY = 0x2   # MOE_FLAG_ONE_WEIGHT_COPY
FORCE = 0x1      # MOE_FLAG_FORCE_GROUPED


def _logical_bytes(sp):
    return sp.H * sp.E * 4 + sp.E * 3 * sp.I * sp.H * 2 + 3 * sp.Is * sp.H * 2


def _create_measured(sp, S, max_tokens, flags):
    """(layer, device bytes the create took) with the caller's weights already resident."""
    from sparse_mixture_experts_gemv_gb300 import MoeLayer
    w = G.weights_of(S)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()   # blocks cached by earlier tests would be released inside the window
    free0 = torch.cuda.mem_get_info()[0]
    L = MoeLayer(sp.H, sp.E, sp.k, sp.I, sp.Is, w, fmt=sp.fmt, max_tokens=max_tokens, flags=flags)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free1 = torch.cuda.mem_get_info()[0]
    return L, free0 - free1


def test_qwen_bf16_one_weight_copy():
    sp = mi.QWEN_LAYER
    S = G.synth(sp)
    logical = _logical_bytes(sp)
    for flags in (ONE_COPY, ONE_COPY | FORCE):
        L, taken = _create_measured(sp, S, 256, flags)
        try:
            wb, ws = L.memory()
            assert wb <= 1.1 * logical, (wb, logical, wb / logical)
            # the count covers what the create took from the device (allocation granularity aside)
            assert abs(taken - (wb + ws)) <= 64 * 2 ** 20 + 0.01 * (wb + ws), (taken, wb, ws)
            assert "one weight copy" in L.describe()
            for T in ((1, 4) if not flags & FORCE else (40, 256)):
                x = mi.tokens(sp, T, stream=9100 + T)
                out, idx, wt = G.run_cuda(L, x)
                G.compare(S, x, out, idx, wt)
        finally:
            L.close()


def test_qwen_bf16_default_keeps_both_layouts():
    sp = mi.QWEN_LAYER
    S = G.synth(sp)
    L, taken = _create_measured(sp, S, 256, 0)
    try:
        wb, ws = L.memory()
        logical = _logical_bytes(sp)
        assert 1.9 * logical <= wb <= 2.1 * logical, wb / logical
        assert abs(taken - (wb + ws)) <= 64 * 2 ** 20 + 0.01 * (wb + ws), (taken, wb, ws)
    finally:
        L.close()


def test_small_bf16_one_weight_copy_every_path():
    """A small layer with one weight copy at several T (ragged expert groups), through
    the decode kernel, the grouped GEMMs, and the chunked driver."""
    from sparse_mixture_experts_gemv_gb300 import MoeLayer
    sp = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, seed=21).spec
    S = G.synth(sp)
    L = MoeLayer(sp.H, sp.E, sp.k, sp.I, sp.Is, G.weights_of(S), max_tokens=300, flags=ONE_COPY)
    try:
        wb, _ = L.memory()
        assert wb <= 1.1 * _logical_bytes(sp)
        for T in (1, 3, 8, 9, 37, 300):
            x = mi.tokens(sp, T, stream=9200 + T)
            out, idx, wt = G.run_cuda(L, x)
            G.compare(S, x, out, idx, wt)
    finally:
        L.close()


def test_mxfp4_layer_memory_is_reported():
    sp = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=22).spec
    L = G.cuda_layer(sp, max_tokens=64)
    wb, ws = L.memory()
    assert wb > 0 and ws > 0
