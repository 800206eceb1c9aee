"""A small owner object around the C ABI for callers holding weights as arrays.

MoeLayer uploads host arrays (numpy, storage formats of include/moe_layer.h)
to device memory with torch, calls moe_layer_create (which repacks them into
memory the layer owns), drops the uploaded copies and exposes forward calls on
torch CUDA tensors. All layer arithmetic runs in libmoe.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _native as N


def _dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


class MoeLayer:
    """Owns one moe_layer_t.

    weights: dict with
      router fp32 [H,E]; router_bias fp32 [E] or None;
      bf16 format:  gate [E,I,H] u16, up [E,I,H] u16, down [E,H,I] u16 (bf16 bits)
      mxfp4 format: gate_codes [E,I,H/2] u8, gate_scales [E,I,H/32] u8, up_codes, up_scales,
                    down_codes [E,H,I/2] u8, down_scales [E,H,I/32] u8
      int4 format:  gate_codes [E,I,H/2] u8, gate_scales / gate_biases [E,I,H/64] (bf16 bits),
                    the same for up, down_codes [E,H,I/2] u8, down_scales / down_biases [E,H,I/64]
      shared_gate [Is,H], shared_up [Is,H], shared_down [H,Is] (bf16 bits)
    """

    def __init__(self, H, E, k, I, Is, weights: dict, fmt: str = "bf16", max_tokens: int = 8,
                 flags: int = 0, device="cuda"):
        self.H, self.E, self.k, self.I, self.Is = H, E, k, I, Is
        self.fmt = fmt
        self.max_tokens = max_tokens
        self.device = torch.device(device)
        code = {"bf16": N.MOE_WEIGHTS_BF16, "mxfp4": N.MOE_WEIGHTS_MXFP4, "int4": N.MOE_WEIGHTS_INT4}[fmt]
        cfg = N.moe_layer_config_t(H, E, k, I, Is, max_tokens, code, flags)
        keep = {}

        def up(name):
            if name not in weights or weights[name] is None:
                return None
            t = _dev(weights[name], self.device)
            keep[name] = t
            return t.data_ptr()

        w = N.moe_layer_weights_t()
        w.router_dev = up("router")
        w.router_bias_dev = up("router_bias")
        if fmt in ("mxfp4", "int4"):
            w.gate_dev, w.up_dev, w.down_dev = up("gate_codes"), up("up_codes"), up("down_codes")
            w.gate_scales_dev, w.up_scales_dev = up("gate_scales"), up("up_scales")
            w.down_scales_dev = up("down_scales")
            if fmt == "int4":
                w.gate_biases_dev, w.up_biases_dev = up("gate_biases"), up("up_biases")
                w.down_biases_dev = up("down_biases")
        else:
            w.gate_dev, w.up_dev, w.down_dev = up("gate"), up("up"), up("down")
        w.shared_gate_dev, w.shared_up_dev = up("shared_gate"), up("shared_up")
        w.shared_down_dev = up("shared_down")
        torch.cuda.synchronize(self.device)
        self.handle = N.moe_layer_create(cfg, w)
        del keep
        torch.cuda.empty_cache()

    # ------------------------------------------------------------------ calls
    def forward(self, x: torch.Tensor, out: torch.Tensor = None, logit_bias: torch.Tensor = None,
                stream: torch.cuda.Stream = None) -> torch.Tensor:
        """x: bf16/int16 CUDA tensor [T, H]; returns out (same dtype) [T, H]."""
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        lb = logit_bias.data_ptr() if logit_bias is not None else None
        st = N.moe_layer_forward_ex(self.handle, x.data_ptr(), out.data_ptr(), T, lb, s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_forward_ex")
        return out

    def forward_chunked(self, x: torch.Tensor, chunk: int = 0, out: torch.Tensor = None,
                        logit_bias: torch.Tensor = None, stream: torch.cuda.Stream = None) -> torch.Tensor:
        """Any number of rows, pushed through the grouped path `chunk` rows at a time
        (0 = max_tokens); bit-identical for every chunk size."""
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        lb = logit_bias.data_ptr() if logit_bias is not None else None
        st = N.moe_layer_forward_chunked(self.handle, x.data_ptr(), out.data_ptr(), T, chunk, lb, s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_forward_chunked")
        return out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, logit_bias_host=None,
                     stream: torch.cuda.Stream = None):
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        lb = logit_bias_host.data_ptr() if logit_bias_host is not None else None
        st = N.moe_layer_forward_host(self.handle, x_host.data_ptr(), out_host.data_ptr(), x_host.shape[0], lb, s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_forward_host")
        return out_host

    def routing(self, T: int, stream=None):
        idx = torch.empty((T, self.k), dtype=torch.int32, device=self.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=self.device)
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        st = N.moe_layer_get_routing(self.handle, idx.data_ptr(), w.data_ptr(), s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_get_routing")
        return idx, w

    def dispatch(self, T: int, stream=None):
        E = self.E
        hist = torch.empty(E, dtype=torch.int32, device=self.device)
        offs = torch.empty(E + 1, dtype=torch.int32, device=self.device)
        perm = torch.empty(T * self.k, dtype=torch.int32, device=self.device)
        pos = torch.empty(T * self.k, dtype=torch.int32, device=self.device)
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        st = N.moe_layer_get_dispatch(self.handle, hist.data_ptr(), offs.data_ptr(), perm.data_ptr(),
                                      pos.data_ptr(), s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_get_dispatch")
        return hist, offs, perm, pos

    def block_map(self, T: int, stream=None):
        """(blocks int32 [n, 2] of (expert, first grouped row), n) of the last grouped forward."""
        rows = N.MOE_GROUPED_BLOCK_ROWS
        cap = (self.max_tokens * self.k + rows - 1) // rows + self.E + 1
        blocks = torch.full((cap, 2), -1, dtype=torch.int32, device=self.device)
        n = torch.zeros(1, dtype=torch.int32, device=self.device)
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        st = N.moe_layer_get_block_map(self.handle, blocks.data_ptr(), cap, n.data_ptr(), s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_get_block_map")
        nb = int(n.item())
        return blocks[:nb], nb

    def memory(self):
        """(weight bytes, workspace bytes) the layer holds on the device."""
        st, wb, ws = N.moe_layer_get_memory(self.handle)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_layer_get_memory")
        return wb, ws

    def stats(self, stream=None) -> N.moe_stats_t:
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        return N.moe_layer_get_stats(self.handle, s)

    def sync_status(self, stream=None) -> int:
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        return N.moe_layer_sync_status(self.handle, s)

    def describe(self) -> str:
        return N.moe_layer_describe(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            N.moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def weights_from_raw(router, router_bias, experts_stacked: dict, shared_raw: dict) -> dict:
    """Assemble the MoeLayer weights dict from stacked routed-expert arrays and shared arrays."""
    w = {"router": router, "router_bias": router_bias}
    w.update(experts_stacked)
    w["shared_gate"] = shared_raw["gate"]
    w["shared_up"] = shared_raw["up"]
    w["shared_down"] = shared_raw["down"]
    return w
