"""Pins of the FP8 LM-head oracle (CPU): the E4M3 format's anchor values, the
encoder against a brute-force nearest-code search, the quantizer's invariants and
the GEMV's closed forms. A plausible mistake in the oracle (wrong bias, rounding
halves away from zero, no saturation, a dropped scale, a transposed product)
fails at least one of these."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import lmhead_oracle as L


def test_e4m3_anchor_values():
    d = L.decode_e4m3(np.arange(256))
    assert d[0x38] == 1.0 and d[0x40] == 2.0 and d[0x3F] == 1.875
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0                 # largest finite
    assert d[0x08] == 2.0 ** -6                                    # smallest normal
    assert d[0x01] == 2.0 ** -9 and d[0x06] == 0.75 * 2.0 ** -6    # subnormals
    assert d[0x00] == 0.0 and d[0x80] == 0.0 and np.signbit(d[0x80])
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    fin = d[:0x7F]
    assert (np.diff(fin) > 0).all()                                # monotone positive half
    assert (d[0x80:0xFF] == -fin).all()                            # sign bit
    assert len(set(d[~np.isnan(d)].tolist())) == 253


def _brute_force(v):
    """Nearest finite code, ties to the code with an even mantissa, saturating."""
    d = L.decode_e4m3(np.arange(256))
    out = []
    for x in np.asarray(v, dtype=np.float64):
        sign = 0x80 if np.signbit(x) else 0x00          # the code keeps the sign of x (-0 for small negatives)
        codes = np.array([c for c in range(sign, sign + 0x7F)])
        vals = d[codes]
        x = min(max(x, -448.0), 448.0)
        err = np.abs(vals - x)
        best = codes[err == err.min()]
        if len(best) > 1:
            best = [c for c in best if c % 2 == 0]      # ties: the even code
        out.append(best[0])
    return np.array(out, dtype=np.uint8)


def test_encoder_matches_brute_force():
    rng = np.random.default_rng(11)
    d = L.decode_e4m3(np.arange(0x7F))
    mids = (d[1:] + d[:-1]) / 2                      # exact ties between neighbours
    v = np.concatenate([
        rng.standard_normal(3000) * 50,
        np.exp2(rng.uniform(-12, 9.5, 3000)) * rng.choice([-1, 1], 3000),
        mids, -mids, d, [449.0, 460.0, 464.0, 470.0, 1e6, -1e6, 2.0 ** -11, 2.0 ** -10, 3 * 2.0 ** -11],
    ]).astype(np.float32)
    got = L.encode_e4m3(v)
    ref = _brute_force(v.astype(np.float64))
    bad = np.nonzero(got != ref)[0]
    assert len(bad) == 0, [(float(v[i]), int(got[i]), int(ref[i])) for i in bad[:5]]


def test_quantized_rows():
    spec = mi.LmHeadSpec(V=300, H=512, seed=3)
    w = mi.lmhead_rows(spec, 0, 300)
    w[7] = 0                                          # an all-zero row
    q, s = L.quantize_rows(w)
    dq = L.decode_e4m3(q) * s[:, None].astype(np.float64)
    wf = L.bf16_bits_to_f64(w)
    assert s[7] == 1.0 and (q[7] == 0).all()
    nz = np.abs(wf).max(axis=1) > 0
    # the largest element of every nonzero row lands on +-448
    assert (np.abs(L.decode_e4m3(q[nz])).max(axis=1) == 448.0).all()
    # round to nearest: within half a quantum (2^-4 relative for normals, s * 2^-10 below)
    err = np.abs(dq - wf)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, s[:, None] * 2.0 ** -10)
    assert (err <= bound * (1 + 1e-12)).all()
    # scales: amax / 448 in fp32
    amax = np.abs(wf).max(axis=1).astype(np.float32)
    assert (s[nz] == (amax[nz] / np.float32(448.0))).all()


def test_forward_closed_forms():
    spec = mi.LmHeadSpec(V=64, H=256, seed=4)
    q, s = L.quantize_rows(mi.lmhead_rows(spec, 0, 64))
    col = L.decode_e4m3(q) * s[:, None]
    onehot = np.zeros((1, 256), dtype=np.uint16)
    onehot[0, 17] = 0x3F80                            # x = e_17 (bf16 1.0)
    assert np.array_equal(L.forward(q, s, onehot)[0], col[:, 17])
    x = mi.lmhead_tokens(spec, 3, stream=1)
    y = L.forward(q, s, x)
    assert y.shape == (3, 64)
    for t in range(3):                                # rows independent of each other
        assert np.allclose(L.forward(q, s, x[t:t + 1])[0], y[t], rtol=0, atol=1e-12)
    # an explicit dot product for one logit
    xf = L.bf16_bits_to_f64(x)
    assert abs(y[2, 5] - sum(col[5, h] * xf[2, h] for h in range(256))) < 1e-9


@pytest.mark.parametrize("mutation", ["bias8", "half_away", "no_saturation"])
def test_planted_mistakes_are_caught(mutation, monkeypatch):
    orig_decode, orig_encode = L.decode_e4m3, L.encode_e4m3
    if mutation == "bias8":
        monkeypatch.setattr(L, "decode_e4m3", lambda c: orig_decode(c) / 2.0)
        with pytest.raises(AssertionError):
            test_e4m3_anchor_values()
    elif mutation == "half_away":
        def enc(v):
            x = np.asarray(v, dtype=np.float64)
            out = orig_encode(v)
            d = L.decode_e4m3(np.arange(0x7F))
            mids = (d[1:] + d[:-1]) / 2
            hit = np.isin(np.abs(x), mids)
            up = np.searchsorted(d, np.abs(x)) & 0x7F     # the larger neighbour
            return np.where(hit, (up | (out & 0x80)).astype(np.uint8), out)
        monkeypatch.setattr(L, "encode_e4m3", enc)
        with pytest.raises(AssertionError):
            test_encoder_matches_brute_force()
    else:
        def enc(v):
            x = np.asarray(v, dtype=np.float64)
            out = orig_encode(v)
            return np.where(np.abs(x) > 464, np.uint8(0x7F) | (out & 0x80), out).astype(np.uint8)
        monkeypatch.setattr(L, "encode_e4m3", enc)
        with pytest.raises(AssertionError):
            test_encoder_matches_brute_force()
