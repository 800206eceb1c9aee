"""Parity of the weight-streaming (decode / verify) path against the fp64 oracle, on the GPU."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as o
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _x(spec, n, stream):
    return mi.tokens(spec, n, stream=stream)


def test_tiny_t8_decode_path():
    w = mi.WORKLOADS["tiny"]
    L = G.cuda_layer(w.layer, max_tokens=64)
    S = G.synth(w.layer)
    x = mi.workload_tokens(w, 0)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 1
    G.compare(S, x, out, idx, wt)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_tiny_every_window_size(T):
    spec = mi.WORKLOADS["tiny"].layer
    L = G.cuda_layer(spec, max_tokens=64)
    x = _x(spec, T, stream=100 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(G.synth(spec), x, out, idx, wt)


def test_qwen_decode_64_tokens():
    w = mi.WORKLOADS["qwen_decode"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    S = G.synth(w.layer)
    worst = 0.0
    for call in range(w.calls):
        x = mi.workload_tokens(w, call)
        out, idx, wt = G.run_cuda(L, x)
        r = G.compare(S, x, out, idx, wt)
        worst = max(worst, r["max_abs"])
    print("qwen_decode worst max-abs", worst)


def test_qwen_verify_windows():
    w = mi.WORKLOADS["qwen_verify"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    S = G.synth(w.layer)
    distinct = []
    for call in range(w.calls):
        x = mi.workload_tokens(w, call)
        lb = mi.workload_logit_bias(w, call)
        out, idx, wt = G.run_cuda(L, x, lb)
        G.compare(S, x, out, idx, wt, logit_bias=lb)
        distinct.append(L.stats().distinct_experts)
        assert distinct[-1] == len(set(idx.reshape(-1).tolist()))
    assert max(distinct) <= 32 and min(distinct) >= 20
    print("verify distinct experts per window", distinct)


@pytest.mark.parametrize("name", ["ling_mxfp4_t1", "ling_mxfp4_t4"])
def test_ling_mxfp4(name):
    w = mi.WORKLOADS[name]
    L = G.cuda_layer(w.layer, max_tokens=8)
    S = G.synth(w.layer)
    for call in range(4):
        x = mi.workload_tokens(w, call)
        out, idx, wt = G.run_cuda(L, x)
        r = G.compare(S, x, out, idx, wt, fmt="mxfp4")
    print(name, r)


@pytest.mark.parametrize("T", [5, 6, 8])
def test_qwen_windows_beyond_four(T):
    """Qwen-shaped windows of 5-8 tokens on the weight-streaming kernel (5 tokens keep
    two 8-record ring groups beside x; 6 and 8 take three 4-record groups)."""
    spec = mi.QWEN_LAYER
    L = G.cuda_layer(spec, max_tokens=4096)
    S = G.synth(spec)
    for call in range(2):
        x = mi.tokens(spec, T, stream=6000 + 10 * T + call)
        out, idx, wt = G.run_cuda(L, x)
        assert L.stats().path == 1
        G.compare(S, x, out, idx, wt)


def test_ling_mxfp4_window_of_seven():
    """The largest weight-streaming window of the Ling-shaped MXFP4 layer (7 tokens,
    16-record MXFP4 groups)."""
    w = mi.WORKLOADS["ling_mxfp4_t4"]
    L = G.cuda_layer(w.layer, max_tokens=8)
    S = G.synth(w.layer)
    x = mi.tokens(w.layer, 7, stream=6070)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 1
    G.compare(S, x, out, idx, wt, fmt="mxfp4")


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_small_mxfp4_every_window_size(T):
    """A small MXFP4 layer (E=16, k=4, so windows share experts and groups cross
    expert and 32-feature scale-block boundaries) at every window size."""
    S = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=5)
    L = G.cuda_layer(S.spec, max_tokens=8)
    x = mi.tokens(S.spec, T, stream=200 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(S, x, out, idx, wt, fmt="mxfp4")


@pytest.mark.parametrize("H,T", [(1024, 1), (1536, 3), (2048, 2)])
def test_mxfp4_stream_every_tile_count(H, T):
    """The MXFP4 stream kernel is compiled per H / 256 (2, 4, 6, 8, 10 output tiles per
    warp); H = 512 and 2560 are covered above, these are the other three."""
    S = mi.custom_layer(H=H, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=17)
    L = G.cuda_layer(S.spec, max_tokens=8)
    assert "moe_decode_stream_mx_kernel" in L.describe()
    x = mi.tokens(S.spec, T, stream=400 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(S, x, out, idx, wt, fmt="mxfp4")


def test_single_routed_expert_window():
    """k = 1, T = 1: one routed expert of 128 features spread over 152 CTAs, so most
    CTAs have no routed record and the group holding their shared tail has no routed
    part; the rest have one or two."""
    S = mi.custom_layer(H=512, E=8, k=1, I=128, Is=256, seed=21)
    L = G.cuda_layer(S.spec, max_tokens=8)
    for stream in range(3):
        x = mi.tokens(S.spec, 1, stream=500 + stream)
        out, idx, wt = G.run_cuda(L, x)
        G.compare(S, x, out, idx, wt)


@pytest.mark.parametrize("H,fmt,T", [(4096, "bf16", 1), (4096, "bf16", 5), (768, "mxfp4", 1), (768, "mxfp4", 3)])
def test_three_phase_kernel_shapes(H, fmt, T):
    """Shapes the record-streaming kernels do not take (bf16 with H > 2048, MXFP4 with H not a
    multiple of 512) run on the three-phase decode kernel; same parity bar."""
    S = mi.custom_layer(H=H, E=8, k=2, I=128, Is=128, fmt=fmt, seed=11)
    L = G.cuda_layer(S.spec, max_tokens=8)
    assert "moe_decode_fused_kernel" in L.describe()
    x = mi.tokens(S.spec, T, stream=300 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(S, x, out, idx, wt, fmt=fmt)


def test_deterministic_and_batch_invariant():
    w = mi.WORKLOADS["qwen_verify"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    x = mi.workload_tokens(w, 3)
    a, ia, _ = G.run_cuda(L, x)
    b, ib, _ = G.run_cuda(L, x)
    assert (a == b).all() and (ia == ib).all()
    singles = np.concatenate([G.run_cuda(L, x[t:t + 1])[0] for t in range(4)])
    d = np.abs(G.bits_to_f64(singles) - G.bits_to_f64(a)).max()
    assert d <= G.BF16_MAX_ABS


def test_forward_host_matches_device_forward():
    w = mi.WORKLOADS["qwen_verify"]
    L = G.cuda_layer(w.layer, max_tokens=4096)
    x = mi.workload_tokens(w, 5)
    lb = mi.workload_logit_bias(w, 5)
    dev, _, _ = G.run_cuda(L, x, lb)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    lbh = torch.from_numpy(lb).pin_memory()
    L.forward_host(xh, oh, lbh)
    assert (oh.numpy().view(np.uint16) == dev).all()


@pytest.mark.parametrize("E,k,Is", [(4, 4, 128), (8, 1, 128), (16, 2, 0)])
def test_degenerate_shapes(E, k, Is):
    """k == E (dense softmax mixture), k == 1, and a layer without a shared expert."""
    S = mi.custom_layer(H=256, E=E, k=k, I=128, Is=Is, seed=3)
    from sparse_mixture_experts_gemv_gb300 import MoeLayer
    L = MoeLayer(256, E, k, 128, Is, G.weights_of(S) if Is else _no_shared(S), max_tokens=8)
    x = mi.tokens(S.spec, 5, stream=7)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(S, x, out, idx, wt)
    L.close()


def _no_shared(S):
    from sparse_mixture_experts_gemv_gb300 import weights_from_raw
    w = weights_from_raw(S.router(), S.router_bias(), S.stacked(), {"gate": None, "up": None, "down": None})
    return w


def test_zero_tokens_is_a_noop():
    spec = mi.WORKLOADS["tiny"].layer
    L = G.cuda_layer(spec, max_tokens=64)
    from sparse_mixture_experts_gemv_gb300 import _native as N
    assert N.moe_layer_forward(L.handle, 0, 0, 0, 0) == N.MOE_OK


def test_invalid_arguments_rejected():
    from sparse_mixture_experts_gemv_gb300 import _native as N
    spec = mi.WORKLOADS["tiny"].layer
    L = G.cuda_layer(spec, max_tokens=64)
    x = torch.zeros((8, 256), dtype=torch.int16, device="cuda")
    out = torch.zeros((8, 256), dtype=torch.int16, device="cuda")
    h = L.handle
    assert N.moe_layer_forward(h, x.data_ptr(), out.data_ptr(), 65, 0) == N.MOE_ERR_INVALID_ARG  # > max_tokens
    assert N.moe_layer_forward(h, x.data_ptr(), out.data_ptr(), -1, 0) == N.MOE_ERR_INVALID_ARG
    assert N.moe_layer_forward(h, 0, out.data_ptr(), 8, 0) == N.MOE_ERR_INVALID_ARG               # null
    assert N.moe_layer_forward(h, x.data_ptr() + 2, out.data_ptr(), 4, 0) == N.MOE_ERR_INVALID_ARG  # misaligned
    assert N.moe_layer_forward(h, x.data_ptr(), x.data_ptr() + 512, 8, 0) == N.MOE_ERR_INVALID_ARG  # overlap
    assert N.moe_layer_forward(0, x.data_ptr(), out.data_ptr(), 8, 0) == N.MOE_ERR_INVALID_ARG
    cfg = N.moe_layer_config_t(256, 16, 17, 128, 128, 8, 0, 0)  # k > E
    st, hh = N.moe_layer_create_status(cfg, N.moe_layer_weights_t())
    assert st == N.MOE_ERR_INVALID_ARG and hh is None
    cfg = N.moe_layer_config_t(200, 16, 2, 128, 128, 8, 0, 0)  # H not a multiple of 256
    w = N.moe_layer_weights_t(router_dev=1, gate_dev=1, up_dev=1, down_dev=1, shared_gate_dev=1,
                              shared_up_dev=1, shared_down_dev=1)
    st, hh = N.moe_layer_create_status(cfg, w)
    assert st == N.MOE_ERR_UNSUPPORTED and hh is None


def test_forced_device_wait_timeout_reports_status():
    """A bounded device wait on a flag nothing sets runs out; the status says so and the
    context stays usable."""
    from sparse_mixture_experts_gemv_gb300 import MoeLayer, _native as N
    S = G.synth(mi.WORKLOADS["tiny"].layer)
    L = MoeLayer(256, 16, 2, 128, 128, G.weights_of(S), max_tokens=8,
                 flags=N.MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT)
    assert "forced wait timeout" in L.describe()
    x = torch.from_numpy(mi.tokens(S.spec, 2, 9).view(np.int16)).cuda()
    L.forward(x)
    torch.cuda.synchronize()
    # later calls fail fast: each would otherwise wait ~2 ms on the forced flag again
    import time
    t0 = time.perf_counter()
    for _ in range(8):
        L.forward(x)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 8e-3
    assert L.sync_status() == N.MOE_ERR_TIMEOUT
    assert L.sync_status() == N.MOE_OK   # cleared
    L.close()
    # the context still works
    good = G.cuda_layer(mi.WORKLOADS["tiny"].layer, max_tokens=64)
    xx = mi.tokens(S.spec, 3, 11)
    out, idx, wt = G.run_cuda(good, xx)
    G.compare(S, xx, out, idx, wt)


def test_describe_names_the_active_path():
    L = G.cuda_layer(mi.WORKLOADS["tiny"].layer, max_tokens=64)
    d = L.describe()
    assert "decode GEMV path" in d and "moe_decode_stream_kernel" in d
    S = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="mxfp4", seed=5)
    assert "moe_decode_stream_mx_kernel" in G.cuda_layer(S.spec, max_tokens=8).describe()


# ---------------------------------------------------------------- int4 routed experts
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_small_int4_every_window_size(T):
    """Groupwise affine int4 routed experts on the record-streaming kernel
    (codes as exact f16 integers on the tensor cores, s * sum(q x) + b * sum(x)
    per block), against the oracle."""
    S = mi.custom_layer(H=512, E=16, k=4, I=256, Is=128, fmt="int4", seed=5)
    L = G.cuda_layer(S.spec, max_tokens=64)
    x = mi.tokens(S.spec, T, stream=7000 + T)
    out, idx, wt = G.run_cuda(L, x)
    assert L.stats().path == 1
    G.compare(G.synth(S.spec), x, out, idx, wt)
    assert "moe_decode_stream_mx_kernel<int4>" in L.describe()


@pytest.mark.parametrize("H,I,T", [(1024, 384, 1), (1024, 384, 7), (2560, 128, 4)])
def test_int4_stream_shapes(H, I, T):
    """int4 records at other hidden sizes (other per-H instantiations), with
    intermediate sizes whose 16-record groups straddle the 64-feature boundaries
    of the down (scale, bias) vectors."""
    S = mi.custom_layer(H=H, E=24, k=6, I=I, Is=128, fmt="int4", seed=H + I)
    L = G.cuda_layer(S.spec, max_tokens=8)
    assert "moe_decode_stream_mx_kernel<int4>" in L.describe()
    x = mi.tokens(S.spec, T, stream=7100 + T)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(G.synth(S.spec), x, out, idx, wt)


def test_int4_three_phase_kernel_outside_stream_limits():
    """H not a multiple of 512: int4 decode runs on the three-phase kernel."""
    S = mi.custom_layer(H=768, E=16, k=4, I=256, Is=128, fmt="int4", seed=6)
    L = G.cuda_layer(S.spec, max_tokens=8)
    assert "moe_decode_fused_kernel<int4>" in L.describe()
    for T in (1, 5):
        x = mi.tokens(S.spec, T, stream=7200 + T)
        out, idx, wt = G.run_cuda(L, x)
        G.compare(G.synth(S.spec), x, out, idx, wt)


def test_qwen_int4_decode():
    w = mi.WORKLOADS["qwen_int4_decode"]
    L = G.cuda_layer(w.layer, max_tokens=8)
    S = G.synth(w.layer)
    assert "moe_decode_stream_mx_kernel<int4>" in L.describe()
    for call in range(3):
        x = mi.workload_tokens(w, call)
        out, idx, wt = G.run_cuda(L, x)
        r = G.compare(S, x, out, idx, wt)
    print("qwen int4 decode", r)
    # a verify window on the same layer
    x = mi.tokens(w.layer, 4, stream=7300)
    out, idx, wt = G.run_cuda(L, x)
    G.compare(S, x, out, idx, wt)
