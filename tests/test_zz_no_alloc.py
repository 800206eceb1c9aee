"""The allocation-free routing entry point (moe_route_topk_noalloc) against the
routing moe_layer_forward computes, through the C ABI, on two calls in a row,
and its weights against the fp64 oracle's renormalised softmax.

Callers that cannot allocate device memory (a host framework that owns all
device memory through its own pool, or a real-time path that must not allocate
once running) use this entry point; its only scratch is a fixed array inside the
library, shared by all calls. This file is collected last so that a run stopping
at the first failure has already run every other test; it also passes on its own
in a fresh process.
"""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as o
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("H,E", [(1024, 128), (2560, 512)])
def test_noalloc_routing_matches_layer_forward_twice(H, E):
    """E=512 is the scratch array's limit and takes the 16-keys-per-lane top-k."""
    from sparse_mixture_experts_gemv_gb300 import MoeLayer, _native as N
    S = mi.custom_layer(H=H, E=E, k=8, I=128, Is=128, seed=21)
    L = MoeLayer(H, E, 8, 128, 128, G.weights_of(S), max_tokens=8)
    router_t = torch.from_numpy(np.ascontiguousarray(S.router().T)).cuda()   # [E, H] fp32
    for call, T in enumerate((4, 1, 8)):
        x_bits = mi.tokens(S.spec, T, stream=900 + call)
        lb_np = mi.logit_bias(S.spec, T, 0.5, stream=900 + call)
        x = torch.from_numpy(x_bits.view(np.int16)).cuda()
        lb = torch.from_numpy(lb_np).cuda()
        L.forward(x, logit_bias=lb)
        ref_idx, ref_w = L.routing(T)
        idx = torch.full((T, 8), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, 8), dtype=torch.float32, device="cuda")
        st = N.moe_route_topk_noalloc(x.data_ptr(), router_t.data_ptr(), None, lb.data_ptr(), T, H, E, 8,
                                      idx.data_ptr(), w.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == N.MOE_OK, N.moe_status_string(st)
        torch.cuda.synchronize()
        # expert sets must agree away from near-ties of the fp64 router logits
        logits = o.router_logits(o.bf16_bits_to_f64(x_bits), S.router().astype(np.float64), None, lb_np)
        firm = o.topk_boundary_gap(logits, 8) >= G.NEAR_TIE
        a, b = idx.cpu().numpy(), ref_idx.cpu().numpy()
        for t in np.nonzero(firm)[0]:
            assert set(a[t].tolist()) == set(b[t].tolist())
        assert o.valid_topk(logits, a.astype(np.int64), G.NEAR_TIE).all()
        same = (a == b).all(axis=1)
        assert np.abs(w.cpu().numpy()[same] - ref_w.cpu().numpy()[same]).max() <= 1e-5
        # weights against the oracle: the renormalised softmax of the selected fp64 logits
        wref = o.routing_weights(logits, a.astype(np.int64))
        assert np.abs(w.cpu().numpy() - wref).max() < 1e-5
        np.testing.assert_allclose(w.cpu().numpy().sum(1), 1.0, atol=1e-5)
    L.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from sparse_mixture_experts_gemv_gb300 import _native as N
    x = torch.zeros((16, 256), dtype=torch.int16, device="cuda")
    r = torch.zeros((1024, 256), dtype=torch.float32, device="cuda")
    idx = torch.zeros((16, 8), dtype=torch.int32, device="cuda")
    w = torch.zeros((16, 8), dtype=torch.float32, device="cuda")
    assert N.moe_route_topk_noalloc(x.data_ptr(), r.data_ptr(), None, None, 9, 256, 16, 2, idx.data_ptr(),
                                    w.data_ptr(), 0) == N.MOE_ERR_UNSUPPORTED       # T > 8
    assert N.moe_route_topk_noalloc(x.data_ptr(), r.data_ptr(), None, None, 2, 256, 1024, 2, idx.data_ptr(),
                                    w.data_ptr(), 0) == N.MOE_ERR_UNSUPPORTED       # E > 512
    assert N.moe_route_topk_noalloc(x.data_ptr(), r.data_ptr(), None, None, 2, 256, 16, 17, idx.data_ptr(),
                                    w.data_ptr(), 0) == N.MOE_ERR_INVALID_ARG       # k > E
