"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch them.

Each mutation replaces one oracle function with a subtly wrong version; the
pins of test_oracle_pins are then run and at least one must fail.
"""
import numpy as np
import pytest

from oracle import moe_oracle as o
from tests import test_oracle_pins as pins

_orig = {name: getattr(o, name) for name in
         ("swiglu_expert", "routing_weights", "select_topk", "mxfp4_to_f64", "e8m0_value",
          "bf16_bits_to_f64", "router_logits", "moe_forward", "dispatch", "e2m1_value", "silu",
         "int4_affine_to_f64")}


def _silu_on_up(X, wg, wu, wd):
    return (_orig["silu"](X @ wu.T) * (X @ wg.T)) @ wd.T


def _no_renorm(logits, idx):
    return np.take_along_axis(o.softmax(logits), idx, -1)   # softmax over all E, not renormalised


def _topk_ascending(logits, k):
    return np.argsort(logits, axis=-1, kind="stable")[:, :k]


def _topk_ties_high(logits, k):
    E = logits.shape[-1]
    rev = logits[:, ::-1]
    order = np.argsort(-rev, axis=-1, kind="stable")
    return (E - 1 - order)[:, :k]


def _nibbles_swapped(codes, scales):
    c = np.asarray(codes)
    return _orig["mxfp4_to_f64"](((c & 0x0F) << 4) | (c >> 4), scales)


def _scale_bias_128(scale):
    return _orig["e8m0_value"](scale) / 2.0


def _e2m1_no_subnormal(code):
    c = np.asarray(code).astype(np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    return sign * np.ldexp(1.0 + 0.5 * m, (e - 1)) * (c & 7 != 0)


def _bf16_wrong_shift(bits):
    b = np.asarray(bits).astype(np.uint32) << np.uint32(15)
    return b.view(np.float32).astype(np.float64)


def _router_no_bias(x, w, router_bias=None, logit_bias=None):
    return x @ w


def _no_shared(layer, x_bits, logit_bias=None, force_idx=None, shared=True):
    return _orig["moe_forward"](layer, x_bits, logit_bias, force_idx, shared=False)


def _dispatch_reverse_tokens(idx, E, block_rows):
    d = _orig["dispatch"](idx[::-1], E, block_rows)
    T, k = idx.shape
    perm = d["perm"]
    t = perm // k
    d["perm"] = (T - 1 - t) * k + perm % k
    return d


def _int4_nibbles_swapped(codes, scales, biases):
    c = np.asarray(codes)
    return _orig["int4_affine_to_f64"](((c & 0x0F) << 4) | (c >> 4), scales, biases)


def _int4_group_32(codes, scales, biases):
    c = np.asarray(codes)
    q = np.stack([c & 0x0F, c >> 4], axis=-1).reshape(c.shape[:-1] + (c.shape[-1] * 2,)).astype(np.float64)
    s = np.repeat(o.bf16_bits_to_f64(scales), 32, axis=-1)
    b = np.repeat(o.bf16_bits_to_f64(biases), 32, axis=-1)
    n = min(q.shape[-1], s.shape[-1])
    return q[..., :n] * s[..., :n] + b[..., :n]


def _int4_signed_codes(codes, scales, biases):
    c = np.asarray(codes)
    q = np.stack([c & 0x0F, c >> 4], axis=-1).reshape(c.shape[:-1] + (c.shape[-1] * 2,)).astype(np.float64)
    q = np.where(q >= 8, q - 16, q)                  # read as two's complement
    s = np.repeat(o.bf16_bits_to_f64(scales), 64, axis=-1)
    b = np.repeat(o.bf16_bits_to_f64(biases), 64, axis=-1)
    return q * s + b


MUTATIONS = {
    "int4_nibbles_swapped": ("int4_affine_to_f64", _int4_nibbles_swapped),
    "int4_group_of_32": ("int4_affine_to_f64", _int4_group_32),
    "int4_signed_codes": ("int4_affine_to_f64", _int4_signed_codes),
    "silu_on_up": ("swiglu_expert", _silu_on_up),
    "weights_not_renormalised": ("routing_weights", _no_renorm),
    "topk_smallest": ("select_topk", _topk_ascending),
    "topk_ties_to_higher_index": ("select_topk", _topk_ties_high),
    "mxfp4_nibbles_swapped": ("mxfp4_to_f64", _nibbles_swapped),
    "e8m0_bias_128": ("e8m0_value", _scale_bias_128),
    "e2m1_subnormal_dropped": ("e2m1_value", _e2m1_no_subnormal),
    "bf16_wrong_shift": ("bf16_bits_to_f64", _bf16_wrong_shift),
    "router_bias_dropped": ("router_logits", _router_no_bias),
    "shared_expert_dropped": ("moe_forward", _no_shared),
    "dispatch_reverse_token_order": ("dispatch", _dispatch_reverse_tokens),
}

PIN_TESTS = [
    lambda: pins.test_bf16_decode_known_patterns(),
    lambda: pins.test_e2m1_table_exhaustive(),
    lambda: pins.test_mxfp4_decode_all_bytes_and_scales(),
    lambda: pins.test_topk_brute_force_with_ties(6, 2),
    lambda: pins.test_routing_weights_closed_form(),
    lambda: pins.test_router_logits_orientation(),
    lambda: pins.test_worked_examples_bf16("k1_two_experts"),
    lambda: pins.test_worked_examples_bf16("k2_softmax_weights"),
    lambda: pins.test_worked_example_mxfp4(),
    lambda: pins.test_single_expert_is_plain_swiglu_mlp(),
    lambda: pins.test_dispatch_invariants_and_brute_force(),
    lambda: pins.test_int4_affine_decode_all_bytes(),
    lambda: pins.test_int4_scale_and_bias_apply_per_64_group(),
    lambda: pins.test_worked_example_int4(),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(o, attr, fn)
    failures = 0
    for pin in PIN_TESTS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"mutation {name} was not caught by any pin"


def test_unmutated_oracle_passes_all_pins():
    for pin in PIN_TESTS:
        pin()
