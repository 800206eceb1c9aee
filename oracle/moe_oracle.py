"""fp64 CPU oracle of one sparse mixture-of-experts layer forward pass.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module. The CUDA library never
calls it, and this module shares no code with the CUDA path.

What it computes (a plain restatement of the layer the two pages describe):

* "Optimizing on-device inference for Apple Silicon", section "Qwen creates
  three different workload shapes": a router scores every routed expert and
  picks 8 of them per token; the layer output combines the selected experts.
* same page, section "Reduce intermediate and state traffic": an expert is a
  gate and an up projection joined by a gated activation, followed by a down
  (output) projection; the layer adds the routing-score-weighted expert outputs
  and the shared expert's output.
* "Three ways to speed up MoE inference on DGX Spark", sections "Why decoding
  was slow in the first place" and "Optimization 1": 512 routed experts, 8
  selected plus one always-on shared expert; routed expert weights in MXFP4.

Readings where the pages are silent, taken here as the plainest reading the
rest of the pages supports: router scores are softmax probabilities
renormalised over the selected k
(equal to a softmax over the k selected logits); the gated activation is
SwiGLU, silu(gate) * up with silu(z) = z / (1 + exp(-z)); the shared expert
has no gate of its own; exact logit ties go to the lower expert index;
MXFP4 is the OCP MX layout: e2m1 codes, two per byte with the even element in
the low nibble, one e8m0 scale byte per 32 consecutive elements along the
contraction dimension, value = e2m1(code) * 2^(scale - 127).

Every input is converted exactly to fp64 (bf16 -> fp64 and fp32 -> fp64 are
exact; MXFP4 decodes exactly) and nothing is rounded until the final optional
bf16 rounding. Library matrix products are used as the dot-product step.

Parity status: no page prints a worked example of layer outputs, so no value
of this oracle is pinned to the pages themselves. It is pinned by closed forms
and invariants in the CPU test suite (dense-masked == sparse, k = E reduces to
a dense softmax mixture, E = 1 reduces to a plain SwiGLU MLP, permutation and
batch invariance, exhaustive MXFP4 decode table, brute-force top-k).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# Storage-format decoding
# ----------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64, exactly (bf16 is the top half of fp32)."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e2m1_value(code: np.ndarray) -> np.ndarray:
    """Value of 4-bit e2m1 codes: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.

    Exponent field 0 is subnormal: value = m * 0.5. Otherwise value =
    2^(e-1) * (1 + m/2). Codes 0 and 8 are +0 and -0.
    """
    c = np.asarray(code).astype(np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, (e - 1).astype(np.int64)))
    return sign * mag


def e8m0_value(scale: np.ndarray) -> np.ndarray:
    """e8m0 scale bytes -> 2^(s - 127); the byte 0xFF encodes NaN."""
    s = np.asarray(scale).astype(np.int64)
    v = np.ldexp(1.0, s - 127)
    return np.where(s == 255, np.nan, v)


def mxfp4_to_f64(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode an MXFP4 matrix: codes [..., K/2] (two e2m1 per byte, even element in the
    low nibble) and scales [..., K/32] (one e8m0 byte per 32 elements) -> fp64 [..., K]."""
    codes = np.asarray(codes)
    lo = codes & 0x0F
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
    vals = e2m1_value(nib)
    sc = np.repeat(e8m0_value(scales), 32, axis=-1)
    return vals * sc


def int4_affine_to_f64(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """Decode a groupwise affine int4 matrix ("Optimizing on-device inference for
    Apple Silicon", section "Decode weights during matrix multiplication": 4-bit
    weights in groups of 64 with a bf16 scale and a bf16 bias per group): codes
    [..., K/2] (two unsigned 4-bit q per byte, even element in the low nibble),
    scales and biases [..., K/64] as bf16 bits -> q * scale + bias in fp64 [..., K]."""
    codes = np.asarray(codes)
    lo = codes & 0x0F
    hi = codes >> 4
    q = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,)).astype(np.float64)
    s = np.repeat(bf16_bits_to_f64(scales), 64, axis=-1)
    b = np.repeat(bf16_bits_to_f64(biases), 64, axis=-1)
    return q * s + b


def round_f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even) in one step; return uint16 bits.

    Only the normal bf16 range is handled (the layer's outputs are far inside it).
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                     # v = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(m * 256.0), e - 8)  # 8 significant bits, rint = ties-to-even
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------
# Router
# ----------------------------------------------------------------------------


def router_logits(x: np.ndarray, w_router: np.ndarray, router_bias=None, logit_bias=None):
    """logits[t, e] = sum_h x[t, h] * W_r[h, e] (+ per-expert bias[e]) (+ per-token bias[t, e])."""
    logits = x @ w_router
    if router_bias is not None:
        logits = logits + np.asarray(router_bias, dtype=np.float64)[None, :]
    if logit_bias is not None:
        logits = logits + np.asarray(logit_bias, dtype=np.float64)
    return logits


def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first."""
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=-1, keepdims=True)


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, in descending order of logit;
    exact ties go to the lower expert index (a stable sort of -logits)."""
    order = np.argsort(-logits, axis=-1, kind="stable")
    return order[:, :k].astype(np.int64)


def routing_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t, j] = p[t, idx[t, j]] / sum_j' p[t, idx[t, j']] with p = softmax over all experts."""
    p = softmax(logits)
    sel = np.take_along_axis(p, idx, axis=-1)
    return sel / sel.sum(axis=-1, keepdims=True)


# ----------------------------------------------------------------------------
# Experts
# ----------------------------------------------------------------------------


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(X: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray):
    """One expert on token rows X [n, H]: h = silu(X W_gate^T) * (X W_up^T); y = h W_down^T.

    W_gate, W_up are [I, H] (row = intermediate feature), W_down is [H, I]."""
    g = X @ w_gate.T
    u = X @ w_up.T
    h = silu(g) * u
    return h @ w_down.T


# ----------------------------------------------------------------------------
# Decoding a layer's weights (duck-typed accessor, see moe_inputs.SynthLayer)
# ----------------------------------------------------------------------------


def decode_expert(layer, e: int):
    """Routed expert e as fp64 (W_gate [I,H], W_up [I,H], W_down [H,I])."""
    raw = layer.expert_raw(e)
    if layer.spec.fmt == "bf16":
        return (bf16_bits_to_f64(raw["gate"]), bf16_bits_to_f64(raw["up"]),
                bf16_bits_to_f64(raw["down"]))
    if layer.spec.fmt == "mxfp4":
        return (mxfp4_to_f64(raw["gate_codes"], raw["gate_scales"]),
                mxfp4_to_f64(raw["up_codes"], raw["up_scales"]),
                mxfp4_to_f64(raw["down_codes"], raw["down_scales"]))
    if layer.spec.fmt == "int4":
        return tuple(int4_affine_to_f64(raw[f"{m}_codes"], raw[f"{m}_scales"], raw[f"{m}_biases"])
                     for m in ("gate", "up", "down"))
    raise ValueError(layer.spec.fmt)


def decode_shared(layer):
    raw = layer.shared_raw()
    return (bf16_bits_to_f64(raw["gate"]), bf16_bits_to_f64(raw["up"]),
            bf16_bits_to_f64(raw["down"]))


# ----------------------------------------------------------------------------
# The layer
# ----------------------------------------------------------------------------


def moe_forward(layer, x_bits: np.ndarray, logit_bias=None, force_idx=None,
                shared: bool = True) -> dict:
    """Forward pass of the layer on bf16 token rows x_bits [T, H] (uint16 bits).

    Steps, in the order the layer defines them:
      1. x -> fp64; logits = x W_r (+ biases)
      2. idx = top-k of the logits (descending, ties to the lower index)
      3. w = softmax probabilities of the selected experts, renormalised
      4. y_j = SwiGLU expert idx_j applied to x
      5. out = sum_j w_j y_j (+ shared expert applied to x)
    force_idx replaces step 2 (used to evaluate a near-tie alternative selection).
    Returns dict(out fp64 [T,H], idx [T,k], w [T,k], logits [T,E]).
    """
    spec = layer.spec
    x = bf16_bits_to_f64(x_bits)
    T = x.shape[0]
    logits = router_logits(x, layer.router().astype(np.float64), layer.router_bias(), logit_bias)
    idx = select_topk(logits, spec.k) if force_idx is None else np.asarray(force_idx, dtype=np.int64)
    w = routing_weights(logits, idx)

    out = np.zeros((T, spec.H), dtype=np.float64)
    # Each expert is evaluated on the rows of the tokens that selected it; the
    # per-token sum over j is then taken in j order.
    y = np.zeros((T, spec.k, spec.H), dtype=np.float64)
    for e in np.unique(idx):
        rows_t, rows_j = np.nonzero(idx == e)
        wg, wu, wd = decode_expert(layer, int(e))
        y[rows_t, rows_j] = swiglu_expert(x[rows_t], wg, wu, wd)
    for j in range(spec.k):
        out += w[:, j:j + 1] * y[:, j]
    if shared and spec.Is > 0:
        sg, su, sd = decode_shared(layer)
        out += swiglu_expert(x, sg, su, sd)
    return {"out": out, "idx": idx, "w": w, "logits": logits}


def topk_boundary_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: gap between the k-th and (k+1)-th largest logit (inf when k == E)."""
    s = -np.sort(-logits, axis=-1)
    if k >= logits.shape[-1]:
        return np.full(logits.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def valid_topk(logits: np.ndarray, idx: np.ndarray, slack: float) -> np.ndarray:
    """Per token: True when idx holds k distinct experts and every selected logit is at
    least every unselected logit minus `slack` (a valid top-k up to near-ties)."""
    T, E = logits.shape
    ok = np.empty(T, dtype=bool)
    for t in range(T):
        sel = np.asarray(idx[t], dtype=np.int64)
        if len(set(sel.tolist())) != len(sel) or sel.min() < 0 or sel.max() >= E:
            ok[t] = False
            continue
        mask = np.zeros(E, dtype=bool)
        mask[sel] = True
        if mask.all():
            ok[t] = True
            continue
        ok[t] = logits[t, mask].min() >= logits[t, ~mask].max() - slack
    return ok


# ----------------------------------------------------------------------------
# Dispatch (grouping token rows by expert), as "Keep expert routing on the GPU"
# describes it: histogram of assignments per expert, prefix scan into offsets,
# scatter of rows into contiguous per-expert groups, list of row blocks.
# ----------------------------------------------------------------------------


def tile_plan(hist: np.ndarray, block_rows: int = 128, half_rows: int = 128) -> np.ndarray:
    """Tiles by expert load ("Optimizing on-device inference for Apple Silicon",
    section "Match tile size to expert load"): each expert's grouped rows are cut
    into blocks of block_rows rows (the last block of an expert holds the rest),
    and a block is computed as as many half_rows-row parts as it holds rows for.
    The grouped GEMMs use block_rows = half_rows = 128: one 128-row tile per block,
    so tiles follow each expert's own row count.

    Returns int64 [n, 4]: (expert, first grouped row, rows in the block, halves),
    in increasing expert order, then increasing first row.
    """
    hist = np.asarray(hist, dtype=np.int64)
    plan = []
    row = 0
    for e, n in enumerate(hist):
        for r0 in range(0, int(n), block_rows):
            rows = min(block_rows, int(n) - r0)
            plan.append((e, row + r0, rows, -(-rows // half_rows)))
        row += int(n)
    return np.array(plan, dtype=np.int64).reshape(-1, 4)


def dispatch(idx: np.ndarray, E: int, block_rows: int) -> dict:
    """Group the (token, slot) assignments by expert.

    hist[e]    number of assignments to expert e
    offsets    exclusive prefix sum of hist, length E + 1
    perm[r]    assignment t*k + j stored at grouped row r; within one expert the
               rows follow increasing token index
    pos[t, j]  grouped row of assignment (t, j) (inverse of perm)
    blocks     (expert, first grouped row) of every block_rows-row block
    """
    T, k = idx.shape
    hist = np.zeros(E, dtype=np.int64)
    for e in idx.reshape(-1):
        hist[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(hist)
    fill = offsets[:-1].copy()
    perm = np.empty(T * k, dtype=np.int64)
    pos = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            perm[fill[e]] = t * k + j
            pos[t, j] = fill[e]
            fill[e] += 1
    blocks = []
    for e in range(E):
        for r0 in range(offsets[e], offsets[e + 1], block_rows):
            blocks.append((e, r0))
    return {"hist": hist, "offsets": offsets, "perm": perm, "pos": pos,
            "blocks": np.array(blocks, dtype=np.int64).reshape(-1, 2)}
