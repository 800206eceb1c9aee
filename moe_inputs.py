"""Seeded synthetic inputs for the sparse mixture-of-experts layer.

This module is the only code shared by the fp64 CPU oracle and the CUDA path.
It draws random numbers and stores them in the layer's storage formats
(bf16 bit patterns, fp32, MXFP4 code bytes and e8m0 scale bytes). It holds
none of the layer's arithmetic: no decoding, no routing, no expert math.

Workloads (the layer shapes come from the two pages' models: Qwen3.6-35B-A3B in
"Optimizing on-device inference for Apple Silicon", section "Qwen creates
three different workload shapes" -- 256 routed experts, 8 selected; and
Ling-3.0-Flash in "Three ways to speed up MoE inference on DGX Spark",
section "Why decoding was slow" -- 512 routed experts, 8 selected, one shared
expert, hidden 2560, moe_intermediate_size 768):

  tiny          H=256,  E=16,  k=2, I=Is=128, T=8, bf16 experts
  qwen_decode   H=2048, E=256, k=8, I=Is=512, T=1 (64 independent tokens)
  qwen_verify   same layer, T=4 windows, per-(token, expert) N(0, 2) logit bias
  ling_mxfp4    H=2560, E=512, k=8, I=Is=768, MXFP4 routed experts, T=1 and 4
  qwen_prefill  same layer as qwen_decode, T=4096, Zipf(1.1) per-expert bias

Random streams. Every array has its own numpy PCG64 stream keyed by
(seed, purpose, index), so any expert can be drawn alone (the oracle draws only
the experts a token touches) and the full layer can be drawn in parallel.
Normals are drawn in float32, scaled in float32 and rounded to bf16 with
round-to-nearest-even.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

# Stream purposes (second element of every seed key).
_P_ROUTER, _P_EXPERT, _P_SHARED, _P_TOKENS, _P_LOGIT_BIAS, _P_ROUTER_BIAS, _P_LMHEAD = range(7)

WEIGHT_STD = np.float32(0.02)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bit patterns.

    Only finite inputs are generated here, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


@dataclass(frozen=True)
class LayerSpec:
    H: int
    E: int
    k: int
    I: int
    Is: int
    fmt: str = "bf16"          # routed-expert storage: "bf16" or "mxfp4"
    seed: int = 0
    router_bias: str = "none"  # "none" or "zipf"
    zipf_s: float = 1.1


@dataclass(frozen=True)
class Workload:
    name: str
    layer: LayerSpec
    T: int                       # tokens per layer call
    calls: int = 1               # independent calls (token windows) in one step
    logit_bias_sigma: float = 0.0
    description: str = ""


QWEN_LAYER = LayerSpec(H=2048, E=256, k=8, I=512, Is=512, fmt="bf16", seed=0)

WORKLOADS = {
    "tiny": Workload(
        "tiny", LayerSpec(H=256, E=16, k=2, I=128, Is=128, fmt="bf16", seed=0), T=8,
        description="tiny MoE layer H=256 E=16 top-2 I=128 + shared, T=8"),
    "qwen_decode": Workload(
        "qwen_decode", QWEN_LAYER, T=1, calls=64,
        description="Qwen-shaped decode H=2048 E=256 top-8 I=512 + shared, T=1, 64 tokens"),
    "qwen_verify": Workload(
        "qwen_verify", QWEN_LAYER, T=4, calls=16, logit_bias_sigma=2.0,
        description="Qwen-shaped verify window T=4 with N(0,2) per-token logit bias"),
    "ling_mxfp4_t1": Workload(
        "ling_mxfp4_t1", LayerSpec(H=2560, E=512, k=8, I=768, Is=768, fmt="mxfp4", seed=0),
        T=1, calls=64,
        description="Ling-shaped MXFP4 decode H=2560 E=512 top-8 I=768 + shared, T=1"),
    "ling_mxfp4_t4": Workload(
        "ling_mxfp4_t4", LayerSpec(H=2560, E=512, k=8, I=768, Is=768, fmt="mxfp4", seed=0),
        T=4, calls=16,
        description="Ling-shaped MXFP4 decode H=2560 E=512 top-8 I=768 + shared, T=4"),
    "ling_mxfp4_prefill": Workload(
        "ling_mxfp4_prefill", LayerSpec(H=2560, E=512, k=8, I=768, Is=768, fmt="mxfp4", seed=0),
        T=4096, calls=1,
        description="Ling-shaped MXFP4 prefill chunk H=2560 E=512 top-8 I=768 + shared, T=4096"),
    "qwen_int4_decode": Workload(
        "qwen_int4_decode", LayerSpec(H=2048, E=256, k=8, I=512, Is=512, fmt="int4", seed=0), T=1, calls=64,
        description="Qwen-shaped decode with groupwise affine int4 routed experts (group 64, bf16 scale + bias)"),
    "qwen_int4_prefill": Workload(
        "qwen_int4_prefill", LayerSpec(H=2048, E=256, k=8, I=512, Is=512, fmt="int4", seed=0,
                                       router_bias="zipf"), T=4096, calls=1,
        description="Qwen-shaped prefill T=4096 with int4 routed experts, Zipf(1.1) per-expert router bias"),
    "qwen_prefill": Workload(
        "qwen_prefill", LayerSpec(H=2048, E=256, k=8, I=512, Is=512, fmt="bf16", seed=0,
                                  router_bias="zipf"), T=4096, calls=1,
        description="Qwen-shaped prefill T=4096, Zipf(1.1) per-expert router bias"),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def _normal_bf16(rng: np.random.Generator, shape, std=WEIGHT_STD) -> np.ndarray:
    z = rng.standard_normal(shape, dtype=np.float32)
    z *= np.float32(std)
    return f32_to_bf16_bits(z)


def _mxfp4_matrix(rng: np.random.Generator, rows: int, K: int):
    """Codes uniform over the 16 e2m1 codes (a uniform byte holds two uniform,
    independent nibbles); one e8m0 scale byte per 32 elements along K with
    exponent uniform in [-8, -4] (byte = 127 + exponent)."""
    codes = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = (127 + rng.integers(-8, -3, size=(rows, K // 32))).astype(np.uint8)
    return codes, scales


def _int4_matrix(rng: np.random.Generator, rows: int, K: int):
    """Groupwise affine int4 (group 64 along K): codes uniform over 0..15 (a uniform
    byte holds two independent uniform nibbles); per group a bf16 scale
    s = 0.02 * (4 / 15) * u, u uniform in [0.5, 1.5), and a bf16 bias
    b = -7.5 * s * (1 + 0.1 z), z ~ N(0, 1), so q * s + b spans about +-0.04 around 0,
    the spread of the bf16 layers' N(0, 0.02) weights."""
    codes = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    u = rng.uniform(0.5, 1.5, size=(rows, K // 64)).astype(np.float32)
    z = rng.standard_normal((rows, K // 64), dtype=np.float32)
    s = f32_to_bf16_bits(np.float32(0.02 * 4 / 15) * u)
    s_f = (s.astype(np.uint32) << np.uint32(16)).view(np.float32)
    b = f32_to_bf16_bits(np.float32(-7.5) * s_f * (np.float32(1) + np.float32(0.1) * z))
    return codes, s, b


class SynthLayer:
    """Lazily drawn weights of one synthetic MoE layer, in storage format.

    expert_raw(e) returns a dict:
      bf16:  gate [I,H] u16, up [I,H] u16, down [H,I] u16   (bf16 bit patterns)
      mxfp4: gate_codes [I,H/2] u8, gate_scales [I,H/32] u8, same for up,
             down_codes [H,I/2] u8, down_scales [H,I/32] u8
      int4:  gate_codes [I,H/2] u8, gate_scales and gate_biases [I,H/64] (bf16 bits),
             same for up, down_codes [H,I/2] u8, down_scales / down_biases [H,I/64]
    shared_raw() returns gate [Is,H], up [Is,H], down [H,Is] as bf16 bits.
    router() returns W_r [H,E] float32; router_bias() returns [E] float32 or None.
    """

    def __init__(self, spec: LayerSpec):
        self.spec = spec
        self._router = None
        self._shared = None

    # -- single pieces -------------------------------------------------------
    def router(self) -> np.ndarray:
        if self._router is None:
            s = self.spec
            r = _rng(s.seed, _P_ROUTER).standard_normal((s.H, s.E), dtype=np.float32)
            r *= WEIGHT_STD
            self._router = r
        return self._router

    def router_bias(self):
        s = self.spec
        if s.router_bias == "none":
            return None
        if s.router_bias == "zipf":
            # Fixed per-expert bias that skews expert load: expert perm[r-1] gets
            # ln p_r - mean(ln p) with p_r proportional to r^-s (Zipf over rank).
            rng = _rng(s.seed, _P_ROUTER_BIAS)
            perm = rng.permutation(s.E)
            r = np.arange(1, s.E + 1, dtype=np.float64)
            logp = -s.zipf_s * np.log(r)
            logp -= np.log(np.exp(logp).sum())
            b = np.empty(s.E, dtype=np.float64)
            b[perm] = logp - logp.mean()
            return b.astype(np.float32)
        raise ValueError(f"unknown router bias {s.router_bias!r}")

    def expert_raw(self, e: int) -> dict:
        s = self.spec
        rng = _rng(s.seed, _P_EXPERT, e)
        if s.fmt == "bf16":
            return {
                "gate": _normal_bf16(rng, (s.I, s.H)),
                "up": _normal_bf16(rng, (s.I, s.H)),
                "down": _normal_bf16(rng, (s.H, s.I)),
            }
        if s.fmt == "mxfp4":
            gc, gs = _mxfp4_matrix(rng, s.I, s.H)
            uc, us = _mxfp4_matrix(rng, s.I, s.H)
            dc, ds = _mxfp4_matrix(rng, s.H, s.I)
            return {"gate_codes": gc, "gate_scales": gs, "up_codes": uc, "up_scales": us,
                    "down_codes": dc, "down_scales": ds}
        if s.fmt == "int4":
            out = {}
            for m, (rows, K) in (("gate", (s.I, s.H)), ("up", (s.I, s.H)), ("down", (s.H, s.I))):
                c, sc, b = _int4_matrix(rng, rows, K)
                out[f"{m}_codes"], out[f"{m}_scales"], out[f"{m}_biases"] = c, sc, b
            return out
        raise ValueError(f"unknown weight format {s.fmt!r}")

    def shared_raw(self) -> dict:
        if self._shared is None:
            s = self.spec
            rng = _rng(s.seed, _P_SHARED)
            self._shared = {
                "gate": _normal_bf16(rng, (s.Is, s.H)),
                "up": _normal_bf16(rng, (s.Is, s.H)),
                "down": _normal_bf16(rng, (s.H, s.Is)),
            }
        return self._shared

    # -- whole layer -----------------------------------------------------------
    def stacked(self, threads: int | None = None) -> dict:
        """All routed experts stacked along a leading E axis (drawn in parallel)."""
        s = self.spec
        threads = threads or min(32, os.cpu_count() or 1)
        first = self.expert_raw(0)
        out = {name: np.empty((s.E,) + a.shape, dtype=a.dtype) for name, a in first.items()}
        for name, a in first.items():
            out[name][0] = a

        def fill(e):
            for name, a in self.expert_raw(e).items():
                out[name][e] = a

        with _cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(1, s.E)))
        return out


def tokens(spec: LayerSpec, n: int, stream: int = 0) -> np.ndarray:
    """n token rows x ~ N(0,1) rounded to bf16; returns uint16 bits [n, H]."""
    rng = _rng(spec.seed, _P_TOKENS, stream)
    return _normal_bf16(rng, (n, spec.H), std=1.0)


def logit_bias(spec: LayerSpec, T: int, sigma: float, stream: int = 0) -> np.ndarray:
    """Per-(token, expert) additive router-logit bias ~ N(0, sigma), float32 [T, E]."""
    rng = _rng(spec.seed, _P_LOGIT_BIAS, stream)
    return (rng.standard_normal((T, spec.E), dtype=np.float32) * np.float32(sigma)).astype(np.float32)


def workload_tokens(w: Workload, call: int) -> np.ndarray:
    """The bf16 token rows [T, H] of one call of a workload."""
    return tokens(w.layer, w.T, stream=hash_stream(w.name, call))


def workload_logit_bias(w: Workload, call: int):
    if w.logit_bias_sigma == 0.0:
        return None
    return logit_bias(w.layer, w.T, w.logit_bias_sigma, stream=hash_stream(w.name, call))


def hash_stream(name: str, call: int) -> int:
    """A stable integer stream id for (workload name, call index)."""
    h = 0
    for ch in name.encode():
        h = (h * 131 + ch) % (1 << 31)
    return h * 100003 + call


def custom_layer(H, E, k, I, Is, fmt="bf16", seed=0, router_bias="none") -> SynthLayer:
    return SynthLayer(LayerSpec(H=H, E=E, k=k, I=I, Is=Is, fmt=fmt, seed=seed,
                                router_bias=router_bias))


# ---------------------------------------------------------------------------
# Output projection (LM head) of the Ling-shaped model: "Three ways to speed up
# MoE inference on DGX Spark", section "Optimization 2": the head projects the
# hidden size 2,560 onto a vocabulary of 157,184 tokens and is stored in bf16.
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class LmHeadSpec:
    V: int = 157_184
    H: int = 2560
    seed: int = 0


LMHEAD = LmHeadSpec()
_LMHEAD_BLOCK = 4096  # rows per random stream


def lmhead_rows(spec: LmHeadSpec, r0: int, r1: int) -> np.ndarray:
    """bf16 bits of rows [r0, r1) of W [V, H] ~ N(0, 0.02); one stream per 4096-row block."""
    out = np.empty((r1 - r0, spec.H), dtype=np.uint16)
    b = r0 // _LMHEAD_BLOCK
    while b * _LMHEAD_BLOCK < r1:
        lo, hi = b * _LMHEAD_BLOCK, min((b + 1) * _LMHEAD_BLOCK, spec.V)
        blk = _normal_bf16(_rng(spec.seed, _P_LMHEAD, b), (hi - lo, spec.H))
        a, z = max(lo, r0), min(hi, r1)
        out[a - r0:z - r0] = blk[a - lo:z - lo]
        b += 1
    return out


def lmhead_weights(spec: LmHeadSpec, threads: int | None = None) -> np.ndarray:
    """All of W [V, H] as bf16 bits (blocks drawn in parallel)."""
    out = np.empty((spec.V, spec.H), dtype=np.uint16)
    nb = (spec.V + _LMHEAD_BLOCK - 1) // _LMHEAD_BLOCK

    def fill(b):
        lo, hi = b * _LMHEAD_BLOCK, min((b + 1) * _LMHEAD_BLOCK, spec.V)
        out[lo:hi] = _normal_bf16(_rng(spec.seed, _P_LMHEAD, b), (hi - lo, spec.H))

    with _cf.ThreadPoolExecutor(threads or min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(nb)))
    return out


def lmhead_tokens(spec: LmHeadSpec, n: int, stream: int = 0) -> np.ndarray:
    """n hidden-state rows x ~ N(0, 1) as bf16 bits [n, H]."""
    return _normal_bf16(_rng(spec.seed, _P_TOKENS, 7_000_000 + stream), (n, spec.H), std=1.0)

