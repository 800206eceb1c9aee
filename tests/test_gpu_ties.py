"""Exact logit ties go to the lower expert index, on every routing path.

The layer's contract (include/moe_layer.h) selects the k largest router logits in
descending order with exact ties broken towards the lower expert index. Random
routers almost never tie, so here the router has repeated columns: expert e uses
column e mod U of a U-column router, so groups of experts far apart in index (and
in different lanes of a warp top-k) have mathematically equal logits. The
expected selection is computed from the U distinct logits and expanded, so the
ties in it are exact; tokens where two different groups come within 1e-5 of each
other near the selection are left out of the strict check (at most a few).

Paths: the bf16 record-streaming decode kernel (T=1, T=4), the MXFP4 one, the
three-phase decode kernel (int4 layer), the grouped tensor-core path, and the
allocation-free routing entry point.
"""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as o
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FORCE = 0x1  # MOE_FLAG_FORCE_GROUPED


class TiedRouter:
    """A synthetic layer whose router column e is column e mod U of its own router."""

    def __init__(self, base, U):
        self.spec = base.spec
        self._base = base
        self.U = U
        self.col = np.arange(base.spec.E) % U
        self.unique = np.ascontiguousarray(base.router()[:, :U])
        self._router = np.ascontiguousarray(self.unique[:, self.col])

    def router(self):
        return self._router

    def router_bias(self):
        return None

    def expert_raw(self, e):
        return self._base.expert_raw(e)

    def shared_raw(self):
        return self._base.shared_raw()


def expected_selection(S: TiedRouter, x_bits):
    """(idx [T, k] by (-logit, index), mask of tokens checked strictly)."""
    k = S.spec.k
    lu = o.router_logits(o.bf16_bits_to_f64(x_bits), S.unique.astype(np.float64))   # [T, U]
    logits = lu[:, S.col]                                                            # exact ties
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int64)
    ok = np.ones(T, dtype=bool)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))
        idx[t] = order[:k]
        # groups met down to the (k+1)-th position must be at least 1e-5 apart
        g = S.col[order[:k + 1]]
        vals = lu[t, np.unique(g)]
        vals.sort()
        if len(vals) > 1 and np.diff(vals).min() < G.NEAR_TIE:
            ok[t] = False
    return idx, ok


def _layer(S, fmt, max_tokens, flags=0):
    from sparse_mixture_experts_gemv_gb300 import MoeLayer, weights_from_raw
    sp = S.spec
    w = weights_from_raw(S.router(), None, S._base.stacked(), S.shared_raw())
    return MoeLayer(sp.H, sp.E, sp.k, sp.I, sp.Is, w, fmt=fmt, max_tokens=max_tokens, flags=flags)


def _check(S, L, x_bits, fmt):
    out, idx, wt = G.run_cuda(L, x_bits)
    want, ok = expected_selection(S, x_bits)
    assert ok.mean() >= 0.75, ok.mean()
    assert (idx[ok] == want[ok]).all(), np.nonzero((idx != want).any(1) & ok)[0][:5]
    # tied experts among the selected get bitwise equal weights
    for t in np.nonzero(ok)[0]:
        g = S.col[idx[t]]
        for a in range(S.spec.k):
            for b in range(a + 1, S.spec.k):
                if g[a] == g[b]:
                    assert wt[t, a] == wt[t, b]
    # count the tokens whose k-th pick ties with an expert left out (the lower index won)
    E = S.spec.E
    boundary = 0
    for t in np.nonzero(ok)[0]:
        left_out = (S.col == S.col[want[t, -1]]) & ~np.isin(np.arange(E), want[t])
        boundary += int(left_out.any())
    G.compare(S, x_bits, out, idx, wt, fmt=fmt)
    return boundary


def test_ties_bf16_stream_kernel():
    """Qwen-shaped router (H=2048, E=256: one or two router rows per CTA), groups of 3."""
    base = mi.custom_layer(H=2048, E=256, k=8, I=128, Is=128, seed=61)
    S = TiedRouter(base, U=86)
    L = _layer(S, "bf16", max_tokens=8)
    try:
        assert "moe_decode_stream_kernel" in L.describe()
        nb = 0
        for T in (1, 4):
            for c in range(6):
                nb += _check(S, L, mi.tokens(base.spec, T, stream=7000 + 10 * T + c), "bf16")
        assert nb > 0
    finally:
        L.close()


def test_ties_mxfp4_stream_kernel():
    base = mi.custom_layer(H=512, E=320, k=8, I=128, Is=128, fmt="mxfp4", seed=62)
    S = TiedRouter(base, U=107)
    L = _layer(S, "mxfp4", max_tokens=8)
    try:
        assert "moe_decode_stream_mx_kernel" in L.describe()
        nb = 0
        for T in (1, 4):
            for c in range(6):
                nb += _check(S, L, mi.tokens(base.spec, T, stream=7100 + 10 * T + c), "mxfp4")
        assert nb > 0
    finally:
        L.close()


def test_ties_three_phase_kernel():
    """MXFP4 with H = 768 (not a multiple of 512) runs on the three-phase kernel."""
    base = mi.custom_layer(H=768, E=320, k=8, I=128, Is=128, fmt="mxfp4", seed=63)
    S = TiedRouter(base, U=107)
    L = _layer(S, "mxfp4", max_tokens=8)
    try:
        assert "moe_decode_fused_kernel" in L.describe()
        nb = 0
        for T in (1, 3):
            for c in range(4):
                nb += _check(S, L, mi.tokens(base.spec, T, stream=7200 + 10 * T + c), "mxfp4")
        assert nb > 0
    finally:
        L.close()


def test_ties_int4_stream_kernel():
    base = mi.custom_layer(H=512, E=320, k=8, I=128, Is=128, fmt="int4", seed=65)
    S = TiedRouter(base, U=107)
    L = _layer(S, "int4", max_tokens=8)
    try:
        assert "moe_decode_stream_mx_kernel<int4>" in L.describe()
        nb = 0
        for T in (1, 4):
            for c in range(4):
                nb += _check(S, L, mi.tokens(base.spec, T, stream=7500 + 10 * T + c), "bf16")
        assert nb > 0
    finally:
        L.close()


@pytest.mark.parametrize("T", [5, 300])
def test_ties_grouped_path(T):
    base = mi.custom_layer(H=2048, E=256, k=8, I=128, Is=128, seed=61)
    S = TiedRouter(base, U=86)
    L = _layer(S, "bf16", max_tokens=512, flags=FORCE)
    try:
        assert _check(S, L, mi.tokens(base.spec, T, stream=7300 + T), "bf16") > 0
    finally:
        L.close()


@pytest.mark.parametrize("E,U", [(256, 86), (512, 171)])
def test_ties_noalloc_entry_point(E, U):
    from sparse_mixture_experts_gemv_gb300 import _native as N
    base = mi.custom_layer(H=1024, E=E, k=8, I=128, Is=128, seed=64)
    S = TiedRouter(base, U=U)
    router_t = torch.from_numpy(np.ascontiguousarray(S.router().T)).cuda()
    T = 8
    x_bits = mi.tokens(base.spec, T, stream=7400 + E)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    idx = torch.full((T, 8), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, 8), dtype=torch.float32, device="cuda")
    st = N.moe_route_topk_noalloc(x.data_ptr(), router_t.data_ptr(), None, None, T, 1024, E, 8, idx.data_ptr(),
                                  w.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == N.MOE_OK
    torch.cuda.synchronize()
    want, ok = expected_selection(S, x_bits)
    got = idx.cpu().numpy().astype(np.int64)
    assert ok.mean() >= 0.75
    assert (got[ok] == want[ok]).all()
