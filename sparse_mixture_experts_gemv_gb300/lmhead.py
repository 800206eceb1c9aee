"""Owner of an online-FP8 LM head (moe_lmhead_* in the C ABI): uploads bf16 W with
torch, lets the library quantize it, and runs the GEMV. Argument marshalling only."""
from __future__ import annotations

import numpy as np
import torch

from . import _native as N


class LmHead:
    def __init__(self, w_bits: np.ndarray, device="cuda"):
        """w_bits: bf16 bit patterns [vocab, hidden] (uint16 numpy array)."""
        self.V, self.H = w_bits.shape
        self.device = torch.device(device)
        w = torch.from_numpy(np.ascontiguousarray(w_bits).view(np.int16)).to(self.device)
        torch.cuda.synchronize(self.device)
        st, h = N.moe_lmhead_create(self.H, self.V, w.data_ptr())
        del w
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_lmhead_create")
        self.handle = h

    def forward(self, x: torch.Tensor, out: torch.Tensor = None, stream: torch.cuda.Stream = None) -> torch.Tensor:
        """x: bf16/int16 CUDA tensor [T, hidden]; returns fp32 logits [T, vocab]."""
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.V), dtype=torch.float32, device=self.device)
        s = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        st = N.moe_lmhead_forward(self.handle, x.data_ptr(), out.data_ptr(), T, s)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_lmhead_forward")
        return out

    def weights(self):
        codes = torch.empty((self.V, self.H), dtype=torch.uint8, device=self.device)
        scales = torch.empty(self.V, dtype=torch.float32, device=self.device)
        st = N.moe_lmhead_get_weights(self.handle, codes.data_ptr(), scales.data_ptr(),
                                      torch.cuda.current_stream(self.device).cuda_stream)
        if st != N.MOE_OK:
            raise N.MoeError(st, "moe_lmhead_get_weights")
        return codes, scales

    def close(self):
        if getattr(self, "handle", None):
            N.moe_lmhead_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
