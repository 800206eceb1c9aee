"""Activations beyond the f16 range on the layers whose kernels hold x (or the
routed SwiGLU outputs) in f16: MXFP4 and int4 routed experts. A call either
matches the fp64 oracle or reports MOE_ERR_DEVICE_CHECK; it never returns
infinities silently. bf16 layers take the whole bf16 range and must match.
"""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as o
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FORCE = 0x1  # MOE_FLAG_FORCE_GROUPED
DEVICE_CHECK = 6


def _big_rows(spec, T, stream, scale):
    """Seeded bf16 rows; every third row has a few entries scaled up to ~scale."""
    x = o.bf16_bits_to_f64(mi.tokens(spec, T, stream=stream))
    rng = np.random.default_rng(stream)
    for t in range(0, T, 3):
        cols = rng.choice(spec.H, size=4, replace=False)
        x[t, cols] = scale * np.sign(x[t, cols] + 1e-9)
    return mi.f32_to_bf16_bits(x.astype(np.float32))


def _run(L, S, x_bits, fmt):
    xt = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    out = L.forward(xt)
    st = L.sync_status()
    if st == DEVICE_CHECK:
        return "reported"
    assert st == 0, st
    got = G.bits_to_f64(out.cpu().numpy().view(np.uint16))
    assert np.isfinite(got).all()
    ref = o.moe_forward(S, x_bits)["out"]
    diff = got - ref
    rel = np.linalg.norm(diff) / np.linalg.norm(ref)
    rms = np.sqrt((ref ** 2).mean())
    if fmt == "bf16":
        assert rel <= G.BF16_REL_L2, rel
    else:
        assert rel <= G.MXFP4_REL_L2 and np.abs(diff).max() / rms <= G.MXFP4_MAX_ABS_NORM, (rel, np.abs(diff).max() / rms)
    return "matched"


@pytest.mark.parametrize("fmt,flags,T", [("mxfp4", 0, 3), ("mxfp4", FORCE, 40), ("int4", 0, 3), ("int4", FORCE, 40),
                                         ("bf16", 0, 3), ("bf16", FORCE, 40)])
def test_large_activations_match_or_report(fmt, flags, T):
    spec = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt=fmt, seed=5).spec
    S = G.synth(spec)
    L = G.cuda_layer(spec, max_tokens=512 if flags else 8, flags=flags)
    outcomes = []
    for scale in (3e3, 1e6):
        outcomes.append(_run(L, S, _big_rows(spec, T, 8100 + T, scale), fmt))
    if fmt == "bf16":
        assert outcomes == ["matched", "matched"]
    else:
        # |x| = 1e6 cannot be held in f16: it must be reported
        assert outcomes[1] == "reported", outcomes
    # the layer is usable again after the report was read
    x = mi.tokens(spec, T, stream=8200 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(S, x, out, idx, wt, fmt="mxfp4" if fmt == "mxfp4" else "bf16")
