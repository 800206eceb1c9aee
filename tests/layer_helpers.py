"""Small explicit-array layers for oracle pins (test-only helpers)."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import moe_inputs


@dataclass(frozen=True)
class Spec:
    H: int
    E: int
    k: int
    I: int
    Is: int
    fmt: str = "bf16"


def bf16(a) -> np.ndarray:
    """Round float values to bf16 bits (RNE); used to build exact small weights."""
    return moe_inputs.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


class ArrayLayer:
    """A layer given by explicit arrays (bf16 bits for experts, fp32 router)."""

    def __init__(self, spec, router, experts, shared, router_bias=None):
        self.spec = spec
        self._router = np.asarray(router, dtype=np.float32)
        self._experts = experts
        self._shared = shared
        self._bias = router_bias

    def router(self):
        return self._router

    def router_bias(self):
        return self._bias

    def expert_raw(self, e):
        return self._experts[e]

    def shared_raw(self):
        return self._shared


class ModifiedLayer:
    """Wraps a layer and transforms some raw arrays (e.g. zeroes a projection)."""

    def __init__(self, base, expert_fn=None, shared_fn=None):
        self.spec = base.spec
        self._base = base
        self._efn = expert_fn
        self._sfn = shared_fn

    def router(self):
        return self._base.router()

    def router_bias(self):
        return self._base.router_bias()

    def expert_raw(self, e):
        r = dict(self._base.expert_raw(e))
        return self._efn(r) if self._efn else r

    def shared_raw(self):
        r = dict(self._base.shared_raw())
        return self._sfn(r) if self._sfn else r


def random_layer(H=32, E=6, k=2, I=16, Is=8, seed=1, fmt="bf16", router_bias="none"):
    return moe_inputs.custom_layer(H, E, k, I, Is, fmt=fmt, seed=seed, router_bias=router_bias)
