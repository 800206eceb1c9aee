"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks the oracle against a closed form, an exhaustive table, a
brute-force enumeration or an invariant that the layer definition fixes, so a
plausible slip in the oracle (a dropped term, a swapped operand, a wrong sign,
index or nibble order) fails at least one of them. test_oracle_mutations
plants such slips into the oracle and checks that these pins catch them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as o
from tests.layer_helpers import ArrayLayer, ModifiedLayer, Spec, bf16, random_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
S1 = 1.0 / (1.0 + math.exp(-1.0))        # silu(1)
S2 = 2.0 / (1.0 + math.exp(-2.0))        # silu(2)


def _expr(s):
    return float(eval(s, {"__builtins__": {}}, {"s1": S1, "s2": S2}))  # closed forms only


# ---------------------------------------------------------------- formats

def test_bf16_decode_known_patterns():
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4000, 0x3F00, 0x4049, 0x7F7F, 0x0080],
                    dtype=np.uint16)
    want = [0.0, -0.0, 1.0, -1.0, 2.0, 0.5, 3.140625, 3.3895313892515355e38, 2.0 ** -126]
    got = o.bf16_bits_to_f64(bits)
    assert got.tolist() == want


def test_bf16_rounding_ties_to_even():
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30, -2.0 - 2 ** -7,
                  0.1, 123.456])
    got = o.round_f64_to_bf16_bits(v)
    assert got[0] == 0x3F80
    assert got[1] == 0x3F80          # halfway, mantissa 0 is even -> down
    assert got[2] == 0x3F82          # halfway between ...81 and ...82 -> even
    assert got[3] == 0x3F81          # just above halfway -> up
    assert got[4] == 0xC000          # -2 - 2^-7 is halfway between -2 and -2-2^-6 -> even
    # general values: the result is the nearest bf16 (check against both neighbours)
    for val, b in zip(v[5:], got[5:]):
        r = o.bf16_bits_to_f64(np.array([b], dtype=np.uint16))[0]
        up = o.bf16_bits_to_f64(np.array([b + 1], dtype=np.uint16))[0]
        dn = o.bf16_bits_to_f64(np.array([b - 1], dtype=np.uint16))[0]
        assert abs(val - r) <= abs(val - up) and abs(val - r) <= abs(val - dn)


def test_e2m1_table_exhaustive():
    table = json.load(open(os.path.join(GOLDEN, "e2m1_table.json")))["values"]
    got = o.e2m1_value(np.arange(16))
    assert got.tolist() == table
    assert np.signbit(got[8])  # code 8 is -0


def test_mxfp4_decode_all_bytes_and_scales():
    """Every byte value in every position of a 32-element block, for several scales:
    element 2i is the low nibble, 2i+1 the high nibble; value = e2m1 * 2^(s-127)."""
    table = np.array(json.load(open(os.path.join(GOLDEN, "e2m1_table.json")))["values"])
    scales = [0, 1, 119, 120, 121, 122, 123, 127, 128, 200, 254]
    codes = np.arange(256, dtype=np.uint8).reshape(16, 16)   # 16 rows x 32 elements
    for s in scales:
        sc = np.full((16, 1), s, dtype=np.uint8)
        got = o.mxfp4_to_f64(codes, sc)
        for r in range(16):
            for byte_i in range(16):
                b = int(codes[r, byte_i])
                assert got[r, 2 * byte_i] == table[b & 15] * 2.0 ** (s - 127)
                assert got[r, 2 * byte_i + 1] == table[b >> 4] * 2.0 ** (s - 127)
    assert np.isnan(o.e8m0_value(np.array([255])))[0]


def test_mxfp4_scale_applies_per_32_block():
    codes = np.full((1, 32), 0x22, dtype=np.uint8)        # 64 elements of value 1.0
    sc = np.array([[127, 130]], dtype=np.uint8)
    got = o.mxfp4_to_f64(codes, sc)
    assert (got[0, :32] == 1.0).all() and (got[0, 32:] == 8.0).all()


def test_int4_affine_decode_all_bytes():
    """Every byte in every position of a 64-element group: element 2i is the low
    nibble q0, 2i+1 the high nibble q1, value = q * scale + bias (scale 0.5 = bf16
    0x3F00, bias -4 = bf16 0xC080): byte 0x3A -> 10 * 0.5 - 4 = 1.0 and 3 * 0.5 - 4 = -2.5."""
    codes = np.arange(256, dtype=np.uint8).reshape(8, 32)      # 8 rows x 64 elements
    sc = np.full((8, 1), 0x3F00, dtype=np.uint16)
    bi = np.full((8, 1), 0xC080, dtype=np.uint16)
    got = o.int4_affine_to_f64(codes, sc, bi)
    for r in range(8):
        for byte_i in range(32):
            b = int(codes[r, byte_i])
            assert got[r, 2 * byte_i] == (b & 15) * 0.5 - 4.0
            assert got[r, 2 * byte_i + 1] == (b >> 4) * 0.5 - 4.0
    assert got[0x3A // 32, 2 * (0x3A % 32)] == 1.0 and got[0x3A // 32, 2 * (0x3A % 32) + 1] == -2.5


def test_int4_scale_and_bias_apply_per_64_group():
    codes = np.full((1, 96), 0x11, dtype=np.uint8)             # 192 elements with q = 1
    sc = np.array([[0x3F80, 0x4000, 0x4080]], dtype=np.uint16)  # 1, 2, 4
    bi = np.array([[0x0000, 0x4120, 0x42C8]], dtype=np.uint16)  # 0, 10, 100
    got = o.int4_affine_to_f64(codes, sc, bi)
    assert (got[0, :64] == 1.0).all() and (got[0, 64:128] == 12.0).all() and (got[0, 128:] == 104.0).all()


# ---------------------------------------------------------------- router

def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-row[e], e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(6, 1), (6, 2), (7, 3), (8, 8), (16, 2)])
def test_topk_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    for trial in range(50):
        logits = rng.integers(-3, 4, size=(5, E)).astype(np.float64)  # many exact ties
        idx = o.select_topk(logits, k)
        for t in range(5):
            assert idx[t].tolist() == _brute_topk(logits[t].tolist(), k)
            # brute force over subsets: the chosen set is a maximum-sum k-subset
            best = max(sum(logits[t, list(c)]) for c in itertools.combinations(range(E), k))
            assert logits[t, idx[t]].sum() == best


def test_routing_weights_closed_form():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(20, 16)) * 3
    idx = o.select_topk(logits, 4)
    w = o.routing_weights(logits, idx)
    sel = np.take_along_axis(logits, idx, -1)
    closed = np.exp(sel) / np.exp(sel).sum(-1, keepdims=True)   # softmax over the k selected
    np.testing.assert_allclose(w, closed, rtol=1e-13, atol=0)
    assert (w > 0).all()
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (np.diff(w, axis=-1) <= 0).all()                    # descending with the logits


def test_router_logits_orientation():
    """W_r is [H, E]: logits[t, e] = sum_h x[t, h] W_r[h, e] (non-square to catch a transpose)."""
    x = np.array([[1.0, 2.0, 3.0]])
    wr = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, -1.0]])
    got = o.router_logits(x, wr, router_bias=np.array([0.5, 0.0]), logit_bias=np.array([[0.0, 10.0]]))
    assert got.tolist() == [[1 + 3 + 0.5, 2 - 3 + 10.0]]


# ---------------------------------------------------------------- worked examples

def _golden_layer(ex):
    spec = Spec(H=ex["H"], E=ex["E"], k=ex["k"], I=ex["I"], Is=ex["Is"])
    experts = [{n: bf16(np.array(m[n])) for n in ("gate", "up", "down")} for m in ex["experts"]]
    shared = {n: bf16(np.array(ex["shared"][n])) for n in ("gate", "up", "down")}
    return ArrayLayer(spec, np.array(ex["router"]), experts, shared)


@pytest.mark.parametrize("name", ["k1_two_experts", "k2_softmax_weights"])
def test_worked_examples_bf16(name):
    ex = {e["name"]: e for e in json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["examples"]}[name]
    layer = _golden_layer(ex)
    r = o.moe_forward(layer, bf16(np.array(ex["x"])))
    assert r["idx"].tolist() == ex["idx"]
    np.testing.assert_allclose(r["w"], [[_expr(s) for s in row] for row in ex["w"]], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(r["out"], [[_expr(s) for s in row] for row in ex["out"]], rtol=1e-14, atol=1e-15)


def test_worked_example_mxfp4():
    ex = {e["name"]: e for e in json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["examples"]}["mxfp4_single_expert"]
    H, I = ex["H"], ex["I"]
    spec = Spec(H=H, E=1, k=1, I=I, Is=1, fmt="mxfp4")

    def mat(rows, K, entries):
        c = np.zeros((rows, K // 2), np.uint8)
        s = np.full((rows, K // 32), 127, np.uint8)
        for (r, byte, scale) in entries:
            c[r, 0] = byte
            s[r, 0] = scale
        return c, s

    gc, gs = mat(I, H, [(0, ex["gate_byte0_row0"], ex["gate_scale_row0"])])
    uc, us = mat(I, H, [(0, ex["up_byte0_row0"], ex["up_scale_row0"])])
    dc, ds = mat(H, I, [(0, ex["down_byte0_row0"], ex["down_scale_row0"]),
                        (1, ex["down_byte0_row1"], ex["down_scale_row1"])])
    expert = {"gate_codes": gc, "gate_scales": gs, "up_codes": uc, "up_scales": us,
              "down_codes": dc, "down_scales": ds}
    zero = {"gate": bf16(np.zeros((1, H))), "up": bf16(np.zeros((1, H))), "down": bf16(np.zeros((H, 1)))}
    layer = ArrayLayer(spec, np.zeros((H, 1)), [expert], zero)
    x = np.zeros((1, H))
    for i, v in ex["x_nonzero"].items():
        x[0, int(i)] = v
    r = o.moe_forward(layer, bf16(x))
    want = np.zeros((1, H))
    for i, s in ex["out_nonzero"].items():
        want[0, int(i)] = _expr(s)
    np.testing.assert_allclose(r["out"], want, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- reductions and invariants

def test_single_expert_is_plain_swiglu_mlp():
    """E = 1, k = 1: the layer is a SwiGLU MLP plus the shared MLP (w = 1)."""
    layer = random_layer(H=24, E=1, k=1, I=10, Is=6, seed=5)
    x = bf16(np.random.default_rng(0).normal(size=(7, 24)))
    r = o.moe_forward(layer, x)
    X = o.bf16_bits_to_f64(x)
    raw = layer.expert_raw(0)
    g, u, d = (o.bf16_bits_to_f64(raw[n]) for n in ("gate", "up", "down"))
    sh = layer.shared_raw()
    sg, su, sd = (o.bf16_bits_to_f64(sh[n]) for n in ("gate", "up", "down"))
    # independent element-wise restatement: sum_i d[:, i] * silu(g_i . x) * (u_i . x)
    want = np.zeros_like(X)
    for t in range(X.shape[0]):
        for (G, U, D) in ((g, u, d), (sg, su, sd)):
            for i in range(G.shape[0]):
                a = float(np.dot(G[i], X[t]))
                b = float(np.dot(U[i], X[t]))
                want[t] += D[:, i] * (a / (1.0 + math.exp(-a)) * b)
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-14)
    assert (r["w"] == 1.0).all()


def test_k_equals_E_is_dense_softmax_mixture():
    layer = random_layer(H=16, E=5, k=5, I=8, Is=4, seed=6)
    x = bf16(np.random.default_rng(1).normal(size=(6, 16)))
    r = o.moe_forward(layer, x)
    X = o.bf16_bits_to_f64(x)
    logits = X @ layer.router().astype(np.float64)
    p = np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)
    want = np.zeros_like(X)
    for e in range(5):
        want += p[:, e:e + 1] * o.swiglu_expert(X, *o.decode_expert(layer, e))
    want += o.swiglu_expert(X, *o.decode_shared(layer))
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp4", "int4"])
def test_dense_masked_equals_sparse(fmt):
    """Evaluate every expert on every token, weight by w on the selected experts and 0
    elsewhere: equals the sparse path."""
    H, I = (64, 32) if fmt != "int4" else (128, 64)   # int4 groups are 64 wide
    layer = random_layer(H=H, E=7, k=3, I=I, Is=32, seed=7, fmt=fmt)
    x = bf16(np.random.default_rng(2).normal(size=(9, H)))
    r = o.moe_forward(layer, x)
    X = o.bf16_bits_to_f64(x)
    dense = np.stack([o.swiglu_expert(X, *o.decode_expert(layer, e)) for e in range(7)], 1)  # [T,E,H]
    mask = np.zeros((9, 7))
    np.put_along_axis(mask, r["idx"], r["w"], axis=1)
    want = (mask[:, :, None] * dense).sum(1) + o.swiglu_expert(X, *o.decode_shared(layer))
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-13)


def test_token_permutation_equivariance_and_batch_invariance():
    layer = random_layer(H=32, E=8, k=2, I=16, Is=8, seed=8)
    x = bf16(np.random.default_rng(3).normal(size=(10, 32)))
    r = o.moe_forward(layer, x)
    perm = np.random.default_rng(4).permutation(10)
    rp = o.moe_forward(layer, x[perm])
    np.testing.assert_allclose(rp["out"], r["out"][perm], rtol=1e-13, atol=1e-15)
    assert (rp["idx"] == r["idx"][perm]).all()
    for t in (0, 5, 9):
        r1 = o.moe_forward(layer, x[t:t + 1])
        np.testing.assert_allclose(r1["out"][0], r["out"][t], rtol=1e-13, atol=1e-15)


def test_zero_down_projections_isolate_terms():
    layer = random_layer(H=32, E=6, k=2, I=16, Is=8, seed=9)
    x = bf16(np.random.default_rng(5).normal(size=(4, 32)))
    full = o.moe_forward(layer, x)["out"]
    X = o.bf16_bits_to_f64(x)
    shared_only = o.swiglu_expert(X, *o.decode_shared(layer))

    def zero_down(r):
        r["down"] = np.zeros_like(r["down"])
        return r

    no_routed = o.moe_forward(ModifiedLayer(layer, expert_fn=zero_down), x)["out"]
    np.testing.assert_allclose(no_routed, shared_only, rtol=1e-13, atol=1e-15)
    no_shared = o.moe_forward(ModifiedLayer(layer, shared_fn=zero_down), x)["out"]
    np.testing.assert_allclose(no_shared + shared_only, full, rtol=1e-12, atol=1e-14)
    assert np.abs(no_shared).max() > 0.01 * np.abs(full).max()


def test_linear_in_routed_down_projection():
    layer = random_layer(H=32, E=6, k=3, I=16, Is=8, seed=10)
    x = bf16(np.random.default_rng(6).normal(size=(5, 32)))
    X = o.bf16_bits_to_f64(x)
    shared = o.swiglu_expert(X, *o.decode_shared(layer))
    base = o.moe_forward(layer, x)["out"] - shared

    def double_down(r):
        r["down"] = bf16(2.0 * o.bf16_bits_to_f64(r["down"]))  # exact doubling in bf16
        return r

    doubled = o.moe_forward(ModifiedLayer(layer, expert_fn=double_down), x)["out"] - shared
    np.testing.assert_allclose(doubled, 2 * base, rtol=1e-12, atol=1e-14)


def test_gate_and_up_roles_differ():
    """silu is applied to the gate projection, not to the up projection."""
    layer = random_layer(H=32, E=3, k=1, I=16, Is=8, seed=11)
    x = bf16(np.random.default_rng(7).normal(size=(3, 32)))
    a = o.moe_forward(layer, x)["out"]

    def swap(r):
        r["gate"], r["up"] = r["up"], r["gate"]
        return r

    b = o.moe_forward(ModifiedLayer(layer, expert_fn=swap, shared_fn=swap), x)["out"]
    assert np.abs(a - b).max() > 1e-6


def test_force_idx_and_valid_topk():
    layer = random_layer(H=32, E=8, k=2, I=16, Is=8, seed=12)
    x = bf16(np.random.default_rng(8).normal(size=(4, 32)))
    r = o.moe_forward(layer, x)
    rf = o.moe_forward(layer, x, force_idx=r["idx"])
    assert (rf["out"] == r["out"]).all()
    assert o.valid_topk(r["logits"], r["idx"], 0.0).all()
    swapped = r["idx"].copy()
    swapped[:, 1] = np.argsort(r["logits"], axis=-1)[:, 0]  # the smallest logit: invalid
    assert not o.valid_topk(r["logits"], swapped, 1e-9).any()
    gap = o.topk_boundary_gap(r["logits"], 2)
    s = np.sort(r["logits"], -1)[:, ::-1]
    np.testing.assert_array_equal(gap, s[:, 1] - s[:, 2])


# ---------------------------------------------------------------- dispatch

def test_dispatch_invariants_and_brute_force():
    rng = np.random.default_rng(9)
    T, k, E, BM = 37, 3, 10, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    d = o.dispatch(idx, E, BM)
    assert d["hist"].sum() == T * k
    assert (d["offsets"][1:] == np.cumsum(d["hist"])).all() and d["offsets"][0] == 0
    assert sorted(d["perm"].tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            assert d["perm"][d["pos"][t, j]] == t * k + j
    for e in range(E):
        grp = d["perm"][d["offsets"][e]:d["offsets"][e + 1]]
        toks = [a // k for a in grp]
        assert toks == sorted(t for t in range(T) if e in idx[t])   # brute-force grouping
        assert all(idx[a // k, a % k] == e for a in grp)
    covered = []
    for (e, r0) in d["blocks"]:
        covered += list(range(r0, min(r0 + BM, d["offsets"][e + 1])))
    assert covered == list(range(T * k))


def test_synthetic_layer_shapes():
    import moe_inputs as mi
    L = mi.SynthLayer(mi.WORKLOADS["tiny"].layer)
    r = L.expert_raw(3)
    assert r["gate"].shape == (128, 256) and r["down"].shape == (256, 128)
    assert (L.expert_raw(3)["gate"] == r["gate"]).all()                 # deterministic
    st = L.stacked(threads=4)
    assert (st["up"][3] == r["up"]).all()
    Lm = mi.SynthLayer(mi.WORKLOADS["ling_mxfp4_t1"].layer)
    rm = Lm.expert_raw(0)
    assert rm["gate_codes"].shape == (768, 1280) and rm["gate_scales"].shape == (768, 80)
    assert rm["down_codes"].shape == (2560, 384) and rm["down_scales"].shape == (2560, 24)
    assert rm["gate_scales"].min() == 119 and rm["gate_scales"].max() == 123
    zb = mi.SynthLayer(mi.WORKLOADS["qwen_prefill"].layer).router_bias()
    assert zb.shape == (256,) and abs(float(zb.mean())) < 1e-5


def test_worked_example_int4():
    ex = {e["name"]: e for e in json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["examples"]}["int4_single_expert"]
    H, I = ex["H"], ex["I"]
    spec = Spec(H=H, E=1, k=1, I=I, Is=1, fmt="int4")

    def mat(rows, K, entries):
        c = np.zeros((rows, K // 2), np.uint8)
        s = np.zeros((rows, K // 64), np.uint16)
        b = np.zeros((rows, K // 64), np.uint16)
        for r, e in entries:
            c[r, 0], s[r, 0], b[r, 0] = e["byte0"], e["scale_bf16"], e["bias_bf16"]
        return c, s, b

    gc, gs, gb = mat(I, H, [(0, ex["gate_row0"])])
    uc, us, ub = mat(I, H, [(0, ex["up_row0"])])
    dc, ds, db = mat(H, I, [(0, ex["down_row0"]), (1, ex["down_row1"])])
    expert = {"gate_codes": gc, "gate_scales": gs, "gate_biases": gb, "up_codes": uc, "up_scales": us,
              "up_biases": ub, "down_codes": dc, "down_scales": ds, "down_biases": db}
    zero = {"gate": bf16(np.zeros((1, H))), "up": bf16(np.zeros((1, H))), "down": bf16(np.zeros((H, 1)))}
    layer = ArrayLayer(spec, np.zeros((H, 1)), [expert], zero)
    x = np.zeros((1, H))
    for i, v in ex["x_nonzero"].items():
        x[0, int(i)] = v
    r = o.moe_forward(layer, bf16(x))
    want = np.zeros((1, H))
    for i, s in ex["out_nonzero"].items():
        want[0, int(i)] = _expr(s)
    np.testing.assert_allclose(r["out"], want, rtol=1e-14, atol=1e-15)


def test_tile_plan_covers_every_row_once_and_follows_the_load():
    """The tile plan by expert load: every grouped row in exactly one block, blocks
    of at most block_rows rows in expert then row order, one part per half_rows
    rows; equal to the dispatch's block list (256-row blocks of 128-row parts here,
    128-row blocks of one part as the grouped GEMMs use them)."""
    rng = np.random.default_rng(3)
    E, T, k = 40, 700, 4
    idx = np.stack([rng.choice(E, size=k, replace=False, p=np.arange(1, E + 1)[::-1] / (E * (E + 1) / 2))
                    for _ in range(T)])
    d = o.dispatch(idx, E, 256)
    plan = o.tile_plan(d["hist"], 256, 128)
    assert (plan[:, :2] == d["blocks"]).all()
    covered = np.zeros(T * k, dtype=np.int64)
    for e, r0, rows, halves in plan:
        assert 1 <= rows <= 256 and halves == (1 if rows <= 128 else 2)
        assert d["offsets"][e] <= r0 and r0 + rows <= d["offsets"][e + 1]
        covered[r0:r0 + rows] += 1
    assert (covered == 1).all()
    # hand-made histogram: 0, 1, 128, 129, 256, 257 rows
    plan = o.tile_plan(np.array([0, 1, 128, 129, 256, 257]), 256, 128)
    assert plan.tolist() == [[1, 0, 1, 1], [2, 1, 128, 1], [3, 129, 129, 2], [4, 258, 256, 2],
                             [5, 514, 256, 2], [5, 770, 1, 1]]
    d128 = o.dispatch(idx, E, 128)
    plan = o.tile_plan(d128["hist"])
    assert (plan[:, :2] == d128["blocks"]).all() and (plan[:, 3] == 1).all()
