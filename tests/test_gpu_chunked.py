"""Long-prompt forward in chunks (moe_layer_forward_chunked) on the GPU: every chunk
runs the grouped path, so the output must be bit-identical for every chunk size and
equal to one forced-grouped call over all rows, which is itself checked against the
fp64 oracle."""
import numpy as np
import pytest

import moe_inputs as mi
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FORCE = 0x1  # MOE_FLAG_FORCE_GROUPED


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _chunked(L, x_bits, chunk, lb=None):
    out = L.forward_chunked(_dev(x_bits), chunk=chunk,
                            logit_bias=None if lb is None else torch.from_numpy(lb).cuda())
    assert L.sync_status() == 0
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp4"])
def test_chunk_size_does_not_change_a_bit(fmt):
    if fmt == "bf16":
        spec = mi.WORKLOADS["tiny"].layer
    else:
        spec = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=5).spec
    T = 1000
    x = mi.tokens(spec, T, stream=4242)
    # one call over all rows on the grouped path: parity against the oracle
    Lf = G.cuda_layer(spec, max_tokens=1024, flags=FORCE)
    ref_bits, idx, wt = G.run_cuda(Lf, x)
    G.compare(G.synth(spec), x, ref_bits, idx, wt, fmt=fmt)
    # a layer whose workspace holds only 256 rows serves all 1000 in chunks
    Lc = G.cuda_layer(spec, max_tokens=256)
    for chunk in (0, 256, 255, 100, 7):
        got = _chunked(Lc, x, chunk)
        assert (got == ref_bits).all(), f"chunk {chunk}: {(got != ref_bits).sum()} values differ"


def test_chunked_with_logit_bias():
    spec = mi.WORKLOADS["tiny"].layer
    T = 300
    x = mi.tokens(spec, T, stream=77)
    lb = mi.logit_bias(spec, T, sigma=2.0, stream=78)
    Lf = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    ref_bits, idx, wt = G.run_cuda(Lf, x, logit_bias=lb)
    G.compare(G.synth(spec), x, ref_bits, idx, wt, logit_bias=lb)
    Lc = G.cuda_layer(spec, max_tokens=64)
    assert (_chunked(Lc, x, 0, lb) == ref_bits).all()
    assert (_chunked(Lc, x, 33, lb) == ref_bits).all()


def test_chunked_arguments():
    from sparse_mixture_experts_gemv_gb300 import _native as N
    spec = mi.WORKLOADS["tiny"].layer
    L = G.cuda_layer(spec, max_tokens=64)
    x = _dev(mi.tokens(spec, 100, stream=5))
    out = torch.empty_like(x)
    f = N.moe_layer_forward_chunked
    assert f(L.handle, x.data_ptr(), out.data_ptr(), 100, 65, None, 0) == N.MOE_ERR_INVALID_ARG   # chunk > max
    assert f(L.handle, x.data_ptr(), out.data_ptr(), 100, -1, None, 0) == N.MOE_ERR_INVALID_ARG   # chunk < 0
    assert f(L.handle, x.data_ptr(), out.data_ptr(), -1, 0, None, 0) == N.MOE_ERR_INVALID_ARG     # T < 0
    assert f(L.handle, x.data_ptr(), x.data_ptr(), 100, 0, None, 0) == N.MOE_ERR_INVALID_ARG      # aliasing
    assert f(L.handle, x.data_ptr() + 2, out.data_ptr(), 10, 0, None, 0) == N.MOE_ERR_INVALID_ARG  # misaligned
    assert f(L.handle, 0, 0, 0, 0, None, 0) == N.MOE_OK                                            # T == 0
    assert f(L.handle, x.data_ptr(), out.data_ptr(), 100, 0, None, 0) == N.MOE_OK
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    assert L.stats().path == N.MOE_PATH_GROUPED and L.stats().tokens == 100 - 64   # the last chunk
