"""Parity of the grouped (prefill) path -- tcgen05 router, GPU dispatch, grouped
tcgen05 GEMMs, combine -- against the fp64 oracle, on the GPU."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as o
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FORCE = 0x1  # MOE_FLAG_FORCE_GROUPED


def _check_dispatch(L, T, k, E, idx):
    hist, offs, perm, pos = (a.cpu().numpy().astype(np.int64) for a in L.dispatch(T))
    ref = o.dispatch(idx, E, 128)
    assert (hist == ref["hist"]).all()
    assert (offs == ref["offsets"]).all()
    assert (perm == ref["perm"]).all()           # bit-exact: token order within each expert
    assert (pos == ref["pos"].reshape(-1)).all()


def test_tiny_forced_grouped_t8():
    w = mi.WORKLOADS["tiny"]
    L = G.cuda_layer(w.layer, max_tokens=512, flags=FORCE)
    S = G.synth(w.layer)
    x = mi.workload_tokens(w, 0)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 2
    G.compare(S, x, out, idx, wt)
    _check_dispatch(L, 8, 2, 16, idx)


@pytest.mark.parametrize("T", [1, 9, 100, 129, 300, 512])
def test_tiny_grouped_ragged(T):
    spec = mi.WORKLOADS["tiny"].layer
    L = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, T, stream=1000 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(G.synth(spec), x, out, idx, wt)
    _check_dispatch(L, T, 2, 16, idx)


def test_grouped_deterministic():
    spec = mi.WORKLOADS["tiny"].layer
    L = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, 300, stream=77)
    a = G.run_cuda(L, x)[0]
    b = G.run_cuda(L, x)[0]
    assert (a == b).all()


def test_qwen_grouped_small_t():
    """Just above the weight-streaming limit: T=9 and T=64 take the grouped path."""
    w = mi.WORKLOADS["qwen_decode"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    S = G.synth(w.layer)
    for T in (9, 64):
        x = mi.tokens(w.layer, T, stream=500 + T)
        out, idx, wt = G.run_cuda(L, x)
        assert L.stats().path == 2
        G.compare(S, x, out, idx, wt)


def test_qwen_prefill_4096_sampled_rows():
    """Full-size prefill chunk (T=4096, Zipf-skewed routing): dispatch checked on all
    rows, outputs on a seeded sample of 256 rows (the layer is token-independent,
    so the oracle on a subset of rows is exact for those rows)."""
    w = mi.WORKLOADS["qwen_prefill"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    S = G.synth(w.layer)
    x = mi.workload_tokens(w, 0)
    out, idx, wt = G.run_cuda(L, x)
    st = L.stats()
    assert st.path == 2
    _check_dispatch(L, 4096, 8, 256, idx)
    rows = np.sort(np.random.default_rng(0).choice(4096, size=256, replace=False))
    ref = o.moe_forward(S, x[rows])
    r = G.compare(S, x[rows], out[rows], idx[rows], wt[rows], ref=ref)
    print("prefill sampled rows", r, "touched", st.distinct_experts, "max rows", st.max_expert_rows)
    assert st.max_expert_rows > 4 * 4096 * 8 / 256   # the Zipf bias skews the load


def test_grouped_matches_decode_path():
    """The two paths agree on the same tokens (T=8 on the tiny layer)."""
    spec = mi.WORKLOADS["tiny"].layer
    Ld = G.cuda_layer(spec, max_tokens=64)
    Lg = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, 8, stream=31)
    a, ia, _ = G.run_cuda(Ld, x)
    b, ib, _ = G.run_cuda(Lg, x)
    assert (ia == ib).all()
    assert np.abs(G.bits_to_f64(a) - G.bits_to_f64(b)).max() <= 2 * G.BF16_MAX_ABS
