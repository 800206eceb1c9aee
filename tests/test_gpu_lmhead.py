"""Online-FP8 LM head on the GPU: the create-time quantizer is bit-exact against the
oracle's (E4M3 round-to-nearest-even with saturation, per-row fp32 scales), and
the GEMV matches the fp64 oracle on the quantized weights within an fp32
dot-product bound."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import lmhead_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _check_logits(codes, scales, x_bits, got):
    """fp32 accumulation bound: |err| <= 2e-5 * sum_h |s * q * x| (+ tiny absolute)."""
    ref = O.forward(codes, scales, x_bits)
    wq = O.decode_e4m3(codes) * scales[:, None].astype(np.float64)
    mag = np.abs(O.bf16_bits_to_f64(x_bits)) @ np.abs(wq).T
    err = np.abs(got.astype(np.float64) - ref)
    assert (err <= 2e-5 * mag + 1e-30).all(), float((err / np.maximum(mag, 1e-30)).max())
    return float((err / np.maximum(mag, 1e-30)).max())


@pytest.mark.parametrize("V,H", [(999, 512), (1024, 256), (333, 2560)])
def test_small_heads(V, H):
    from sparse_mixture_experts_gemv_gb300 import LmHead
    spec = mi.LmHeadSpec(V=V, H=H, seed=V)
    w = mi.lmhead_rows(spec, 0, V)
    w[3] = 0                                          # all-zero row: scale 1, codes 0
    w[5, :7] = [0x3F80, 0xBF80, 0x0001, 0x8001, 0x5F80, 0x0000, 0x8000]  # 1, -1, subnormals, 2^64, +-0
    head = LmHead(w)
    try:
        codes, scales = (a.cpu().numpy() for a in head.weights())
        rq, rs = O.quantize_rows(w)
        assert (scales == rs).all()
        bad = np.argwhere(codes != rq)
        assert len(bad) == 0, [(int(r), int(c), int(codes[r, c]), int(rq[r, c])) for r, c in bad[:5]]
        for T in (1, 2, 3, 4):
            x = mi.lmhead_tokens(spec, T, stream=T)
            got = head.forward(_dev(x)).cpu().numpy()
            _check_logits(codes, scales, x, got)
    finally:
        head.close()


def test_full_size_head_sampled_rows():
    """157,184 x 2,560 head, T=4: quantized codes of 512 sampled rows and their
    logits against the oracle."""
    from sparse_mixture_experts_gemv_gb300 import LmHead
    spec = mi.LMHEAD
    head = LmHead(mi.lmhead_weights(spec))
    try:
        x = mi.lmhead_tokens(spec, 4, stream=11)
        got = head.forward(_dev(x)).cpu().numpy()
        codes, scales = head.weights()
        rows = np.sort(np.random.default_rng(5).choice(spec.V, size=512, replace=False))
        idx = torch.from_numpy(rows).cuda()
        c = codes[idx].cpu().numpy()
        s = scales[idx].cpu().numpy()
        w_rows = np.stack([mi.lmhead_rows(spec, int(r), int(r) + 1)[0] for r in rows])
        rq, rs = O.quantize_rows(w_rows)
        assert (s == rs).all() and (c == rq).all()
        r = _check_logits(c, s, x, got[:, rows])
        print("full-size head: max error / fp32 bound", r)
        # T=1 equals the first row of T=4
        g1 = head.forward(_dev(x[:1])).cpu().numpy()
        assert (g1[0] == got[0]).all()
    finally:
        head.close()


def test_lmhead_arguments():
    from sparse_mixture_experts_gemv_gb300 import _native as N, LmHead
    spec = mi.LmHeadSpec(V=64, H=256, seed=1)
    w = _dev(mi.lmhead_rows(spec, 0, 64))
    assert N.moe_lmhead_create(250, 64, w.data_ptr())[0] == N.MOE_ERR_UNSUPPORTED   # H % 256
    assert N.moe_lmhead_create(256, 0, w.data_ptr())[0] == N.MOE_ERR_INVALID_ARG
    assert N.moe_lmhead_create(256, 64, 0)[0] == N.MOE_ERR_INVALID_ARG
    head = LmHead(mi.lmhead_rows(spec, 0, 64))
    try:
        x = _dev(mi.lmhead_tokens(spec, 5, stream=2))
        out = torch.empty((5, 64), dtype=torch.float32, device="cuda")
        f = N.moe_lmhead_forward
        assert f(head.handle, x.data_ptr(), out.data_ptr(), 5, 0) == N.MOE_ERR_INVALID_ARG      # T > 4
        assert f(head.handle, x.data_ptr() + 2, out.data_ptr(), 1, 0) == N.MOE_ERR_INVALID_ARG  # misaligned
        assert f(head.handle, 0, 0, 0, 0) == N.MOE_OK
        assert f(head.handle, x.data_ptr(), out.data_ptr(), 4, 0) == N.MOE_OK
        torch.cuda.synchronize()
    finally:
        head.close()
