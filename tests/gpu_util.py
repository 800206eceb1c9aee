"""Helpers for the GPU parity tests: build layers from the seeded generator, run the
CUDA path through the C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import functools

import numpy as np

import moe_inputs as mi
from oracle import moe_oracle as o

# Tolerances on the bf16 outputs against the unrounded fp64 oracle.
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
# MXFP4 layers have outputs with RMS ~15 (a bf16 ulp there is 0.06-0.25), so the
# max-abs bound applies to outputs normalised by the oracle RMS.
MXFP4_MAX_ABS_NORM = 5e-2
MXFP4_REL_L2 = 1e-2
NEAR_TIE = 1e-5


def bits_to_f64(bits):
    return o.bf16_bits_to_f64(bits)


@functools.lru_cache(maxsize=4)
def synth(spec: mi.LayerSpec) -> mi.SynthLayer:
    return mi.SynthLayer(spec)


def weights_of(S: mi.SynthLayer) -> dict:
    from sparse_mixture_experts_gemv_gb300 import weights_from_raw
    return weights_from_raw(S.router(), S.router_bias(), S.stacked(), S.shared_raw())


_layers = {}


def cuda_layer(spec: mi.LayerSpec, max_tokens: int, flags: int = 0):
    """MoeLayer for a synthetic layer (cached per (spec, max_tokens, flags) in this process)."""
    from sparse_mixture_experts_gemv_gb300 import MoeLayer
    key = (spec, max_tokens, flags)
    if key in _layers:   # most recently used last, so eviction takes the least recently used
        _layers[key] = _layers.pop(key)
    else:
        # keep at most two big layers alive
        if len(_layers) >= 3:
            _layers.pop(next(iter(_layers))).close()
        S = synth(spec)
        _layers[key] = MoeLayer(spec.H, spec.E, spec.k, spec.I, spec.Is, weights_of(S), fmt=spec.fmt,
                                max_tokens=max_tokens, flags=flags)
    return _layers[key]


def run_cuda(layer, x_bits: np.ndarray, logit_bias=None):
    import torch
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    lb = torch.from_numpy(np.ascontiguousarray(logit_bias, dtype=np.float32)).cuda() if logit_bias is not None else None
    out = layer.forward(x, logit_bias=lb)
    idx, w = layer.routing(x.shape[0])
    st = layer.sync_status()
    assert st == 0, f"device status {st}"
    return (out.cpu().numpy().view(np.uint16), idx.cpu().numpy().astype(np.int64), w.cpu().numpy())


def compare(S, x_bits, out_bits, gpu_idx, gpu_w=None, logit_bias=None, fmt="bf16", ref=None,
            rows=None):
    """Compare CUDA results with the oracle. Returns a dict of error figures; asserts the bars.

    Token rows whose k-th/(k+1)-th oracle logit gap is below NEAR_TIE may pick either
    side of the tie: the CUDA selection must then be a valid top-k within NEAR_TIE,
    and those rows are compared with the oracle evaluated on the CUDA selection.
    rows: compare only these token rows (the layer treats rows independently), so
    that large calls are checked on a sample the oracle computes quickly.
    """
    k = S.spec.k
    if rows is not None:
        assert ref is None
        rows = np.asarray(rows)
        x_bits, out_bits, gpu_idx = x_bits[rows], out_bits[rows], gpu_idx[rows]
        gpu_w = None if gpu_w is None else gpu_w[rows]
        logit_bias = None if logit_bias is None else logit_bias[rows]
    if ref is None:
        ref = o.moe_forward(S, x_bits, logit_bias=logit_bias)
    logits = ref["logits"]
    gap = o.topk_boundary_gap(logits, k)
    near = gap < NEAR_TIE
    firm = ~near
    # selected expert indices: exact set equality away from ties, order where gaps allow
    for t in np.nonzero(firm)[0]:
        assert set(gpu_idx[t].tolist()) == set(ref["idx"][t].tolist()), f"token {t}: idx {gpu_idx[t]} vs {ref['idx'][t]}"
        sel = logits[t, ref["idx"][t]]
        for j in range(k):
            lo_gap = np.inf if j == 0 else sel[j - 1] - sel[j]
            hi_gap = np.inf if j == k - 1 else sel[j] - sel[j + 1]
            if min(lo_gap, hi_gap) >= NEAR_TIE:
                assert gpu_idx[t, j] == ref["idx"][t, j], f"token {t} slot {j}"
    ref_out = ref["out"].copy()
    if near.any():
        assert o.valid_topk(logits[near], gpu_idx[near], NEAR_TIE).all()
        alt = o.moe_forward(S, x_bits[near], logit_bias=None if logit_bias is None else logit_bias[near],
                            force_idx=gpu_idx[near])
        ref_out[near] = alt["out"]
    if gpu_w is not None:
        # weights: renormalised softmax of the selected (oracle) logits, fp32 on the GPU
        wref = o.routing_weights(logits, gpu_idx)
        assert np.abs(gpu_w - wref).max() < 1e-5, np.abs(gpu_w - wref).max()
        assert np.abs(gpu_w.sum(-1) - 1).max() < 1e-5
    got = bits_to_f64(out_bits)
    diff = got - ref_out
    max_abs = float(np.abs(diff).max())
    rel_l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(ref_out), 1e-30))
    rms = float(np.sqrt((ref_out ** 2).mean()))
    res = {"max_abs": max_abs, "rel_l2": rel_l2, "rms": rms, "near_ties": int(near.sum())}
    if fmt == "mxfp4":
        assert max_abs / rms <= MXFP4_MAX_ABS_NORM, res
        assert rel_l2 <= MXFP4_REL_L2, res
    else:
        assert max_abs <= BF16_MAX_ABS, res
        assert rel_l2 <= BF16_REL_L2, res
    return res
