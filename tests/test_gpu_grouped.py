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
    from sparse_mixture_experts_gemv_gb300 import _native as N
    ref = o.dispatch(idx, E, N.MOE_GROUPED_BLOCK_ROWS)
    assert (hist == ref["hist"]).all()
    assert (offs == ref["offsets"]).all()
    assert (perm == ref["perm"]).all()           # bit-exact: token order within each expert
    assert (pos == ref["pos"].reshape(-1)).all()
    # the block map the grouped GEMMs take as M tiles: (expert, first grouped row), bit-exact,
    # and the oracle's tile plan by expert load gives the same blocks
    blocks, nb = L.block_map(T)
    assert nb == len(ref["blocks"]), (nb, len(ref["blocks"]))
    assert (blocks.cpu().numpy().astype(np.int64) == ref["blocks"]).all()
    plan = o.tile_plan(hist, N.MOE_GROUPED_BLOCK_ROWS, N.MOE_GROUPED_BLOCK_ROWS)
    assert (plan[:, :2] == blocks.cpu().numpy().astype(np.int64)).all()


def test_tiny_forced_grouped_t8():
    w = mi.WORKLOADS["tiny"]
    L = G.cuda_layer(w.layer, max_tokens=512, flags=FORCE)
    S = G.synth(w.layer)
    x = mi.workload_tokens(w, 0)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 2
    G.compare(S, x, out, idx, wt)
    _check_dispatch(L, 8, 2, 16, idx)


@pytest.mark.parametrize("T", [1, 9, 100, 127, 128, 129, 255, 256, 257, 300, 512])
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


# ---------------------------------------------------------------- MXFP4 routed experts
def _mx_small():
    return mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=5).spec


@pytest.mark.parametrize("T", [1, 8, 9, 100, 129, 300])
def test_small_mxfp4_grouped(T):
    """MXFP4 routed experts decoded inside the grouped tcgen05 GEMMs (forced grouped
    path at small T, ragged 128-row blocks), against the oracle."""
    spec = _mx_small()
    L = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, T, stream=3000 + T)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 2
    G.compare(G.synth(spec), x, out, idx, wt, fmt="mxfp4")
    _check_dispatch(L, T, spec.k, spec.E, idx)


def test_mxfp4_grouped_wide_scale_range():
    """Scale exponents spread over 24 binades inside each row (the in-kernel f16
    stage holds e2m1 x 2^(s - largest scale of the row), exact down to 2^-23),
    on both gate/up and down rows."""
    from sparse_mixture_experts_gemv_gb300 import MoeLayer, weights_from_raw
    from tests.layer_helpers import ModifiedLayer

    base = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=9)
    spec = base.spec

    def widen(r):
        out = dict(r)
        for name in ("gate_scales", "up_scales", "down_scales"):
            s = r[name].astype(np.int64)
            rows, nb = s.shape
            spread = (np.arange(rows)[:, None] * 7 + np.arange(nb)[None, :] * 5) % 24
            out[name] = (127 - 2 - spread).astype(np.uint8)   # exponents -2 ... -25
        return out

    S = ModifiedLayer(base, expert_fn=widen)
    raws = [S.expert_raw(e) for e in range(spec.E)]
    stacked = {n: np.stack([r[n] for r in raws]) for n in raws[0]}
    weights = weights_from_raw(S.router(), S.router_bias(), stacked, S.shared_raw())
    L = MoeLayer(spec.H, spec.E, spec.k, spec.I, spec.Is, weights, fmt="mxfp4", max_tokens=512, flags=FORCE)
    try:
        x = mi.tokens(spec, 200, stream=41)
        out, idx, wt = G.run_cuda(L, x)
        G.compare(S, x, out, idx, wt, fmt="mxfp4")
    finally:
        L.close()


def test_mxfp4_grouped_matches_decode_path():
    """T=7 MXFP4 window: the record-streaming decode kernel and the grouped GEMMs
    select the same experts and agree to a few output roundings."""
    spec = _mx_small()
    Ld = G.cuda_layer(spec, max_tokens=64)
    Lg = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, 7, stream=32)
    a, ia, _ = G.run_cuda(Ld, x)
    b, ib, _ = G.run_cuda(Lg, x)
    assert (ia == ib).all()
    da, db = G.bits_to_f64(a), G.bits_to_f64(b)
    rms = np.sqrt((da ** 2).mean())
    assert np.abs(da - db).max() / rms <= 2 * G.MXFP4_MAX_ABS_NORM


def test_ling_mxfp4_prefill_sampled_rows():
    """Ling-shaped MXFP4 prefill chunk (T=4096, H=2560, E=512, top-8, I=768):
    dispatch checked on all rows, outputs on a seeded sample of 64 rows."""
    w = mi.WORKLOADS["ling_mxfp4_prefill"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    S = G.synth(w.layer)
    x = mi.workload_tokens(w, 0)
    out, idx, wt = G.run_cuda(L, x)
    st = L.stats()
    assert st.path == 2
    _check_dispatch(L, 4096, 8, 512, idx)
    rows = np.sort(np.random.default_rng(1).choice(4096, size=64, replace=False))
    ref = o.moe_forward(S, x[rows])
    r = G.compare(S, x[rows], out[rows], idx[rows], wt[rows], fmt="mxfp4", ref=ref)
    print("ling mxfp4 prefill sampled rows", r, "touched", st.distinct_experts)


# ---------------------------------------------------------------- int4 routed experts
@pytest.mark.parametrize("T", [9, 100, 300])
def test_small_int4_grouped(T):
    """int4 routed experts decoded to f16 (one rounding of q * s + b) inside the
    grouped tcgen05 GEMMs, against the oracle."""
    spec = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="int4", seed=5).spec
    L = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, T, stream=8000 + T)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 2
    G.compare(G.synth(spec), x, out, idx, wt)
    _check_dispatch(L, T, spec.k, spec.E, idx)


def test_int4_grouped_deterministic_and_matches_decode():
    spec = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="int4", seed=5).spec
    Lg = G.cuda_layer(spec, max_tokens=512, flags=FORCE)
    x = mi.tokens(spec, 300, stream=99)
    a = G.run_cuda(Lg, x)[0]
    b = G.run_cuda(Lg, x)[0]
    assert (a == b).all()
    Ld = G.cuda_layer(spec, max_tokens=64)
    xs = x[:6]
    d, i_d, _ = G.run_cuda(Ld, xs)
    g, i_g, _ = G.run_cuda(Lg, xs)
    assert (i_d == i_g).all()
    assert np.abs(G.bits_to_f64(d) - G.bits_to_f64(g)).max() <= 2 * G.BF16_MAX_ABS


def test_qwen_int4_prefill_sampled_rows():
    w = mi.WORKLOADS["qwen_int4_prefill"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    S = G.synth(w.layer)
    x = mi.workload_tokens(w, 0)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 2
    _check_dispatch(L, 4096, 8, 256, idx)
    rows = np.sort(np.random.default_rng(2).choice(4096, size=128, replace=False))
    r = G.compare(S, x[rows], out[rows], idx[rows], wt[rows], ref=o.moe_forward(S, x[rows]))
    print("qwen int4 prefill sampled rows", r)


@pytest.mark.parametrize("max_tokens,T", [(10000, 9000), (10000, 4865), (10000, 33)])
def test_dispatch_several_chunks_per_cta(max_tokens, T):
    """The cooperative dispatch kernel runs a fixed grid of min(SMs, chunks of
    max_tokens) CTAs; with 10000 tokens of capacity each CTA owns two 32-token
    chunks (9000 tokens), a CTA boundary falls inside a chunk pair (4865), or most
    CTAs own none (33). hist/offsets/perm/pos and the block map stay bit-exact."""
    spec = mi.custom_layer(H=256, E=64, k=4, I=128, Is=128, seed=31).spec
    L = G.cuda_layer(spec, max_tokens=max_tokens, flags=FORCE)
    x = mi.tokens(spec, T, stream=3100 + T)
    out, idx, wt = G.run_cuda(L, x)
    _check_dispatch(L, T, spec.k, spec.E, idx)
    rows = np.random.default_rng(T).choice(T, size=min(T, 64), replace=False)
    G.compare(G.synth(spec), x, out, idx, wt, rows=np.sort(rows))


def test_dispatch_three_kernel_form_for_huge_capacity():
    """With 240000 tokens in one call and 512 experts, 50 chunks per CTA: the per-CTA
    mask table of the cooperative dispatch (50 x 512 words + its count table) would
    not fit in its shared memory, so the three-kernel form runs (top-k + histogram,
    scan, scatter) and gives the same bit-exact dispatch."""
    spec = mi.custom_layer(H=256, E=512, k=2, I=128, Is=128, seed=32).spec
    L = G.cuda_layer(spec, max_tokens=240000, flags=FORCE)
    T = 240000
    x = mi.tokens(spec, T, stream=3200)
    out, idx, wt = G.run_cuda(L, x)
    _check_dispatch(L, T, spec.k, spec.E, idx)
    rows = np.random.default_rng(5).choice(T, size=48, replace=False)
    G.compare(G.synth(spec), x, out, idx, wt, rows=np.sort(rows))
