"""ctypes binding of libmoe.so (the C ABI declared in include/moe_layer.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
The functions keep the C names; pointers are passed as Python ints (for
example torch.Tensor.data_ptr()), streams as the integer value of a
cudaStream_t (torch.cuda.Stream.cuda_stream).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_OOM = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_WEIGHTS_BF16 = 0
MOE_WEIGHTS_MXFP4 = 1
MOE_WEIGHTS_INT4 = 2

MOE_FLAG_FORCE_GROUPED = 0x1
MOE_FLAG_ONE_WEIGHT_COPY = 0x2
MOE_FLAG_TEST_FORCE_WAIT_TIMEOUT = 0x100
MOE_DECODE_MAX_T = 8
MOE_GROUPED_BLOCK_ROWS = 128

MOE_PATH_NONE = 0
MOE_PATH_DECODE_GEMV = 1
MOE_PATH_GROUPED = 2


class moe_layer_config_t(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("shared_intermediate", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("weight_format", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class moe_layer_weights_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_dev", "router_bias_dev", "gate_dev", "up_dev", "down_dev", "gate_scales_dev",
        "up_scales_dev", "down_scales_dev", "shared_gate_dev", "shared_up_dev", "shared_down_dev",
        "gate_biases_dev", "up_biases_dev", "down_biases_dev")]


class moe_stats_t(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("tokens", ctypes.c_int32), ("distinct_experts", ctypes.c_int32),
                ("max_expert_rows", ctypes.c_int32), ("weight_bytes", ctypes.c_int64),
                ("algorithmic_bytes", ctypes.c_int64), ("flops", ctypes.c_double)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {moe_status_string(status)}"
        if status == MOE_ERR_CUDA:
            msg += f" ({moe_last_cuda_error()})"
        super().__init__(msg)


_lib = None

# name -> (restype, argtypes); mirrors include/moe_layer.h
_SIGNATURES = {
    "moe_layer_create": (ctypes.c_int, [ctypes.POINTER(moe_layer_config_t), ctypes.POINTER(moe_layer_weights_t),
                                        ctypes.POINTER(ctypes.c_void_p)]),
    "moe_layer_destroy": (None, [ctypes.c_void_p]),
    "moe_layer_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_void_p]),
    "moe_layer_forward_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_forward_chunked": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_forward_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_get_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(moe_stats_t)]),
    "moe_layer_get_routing": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_get_dispatch": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_void_p] * 4 + [ctypes.c_void_p]),
    "moe_layer_get_block_map": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                               ctypes.c_void_p]),
    "moe_layer_get_memory": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64),
                                            ctypes.POINTER(ctypes.c_int64)]),
    "moe_layer_sync_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_describe": (ctypes.c_char_p, [ctypes.c_void_p]),
    "moe_layer_profile_enable": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "moe_layer_profile_read": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_float), ctypes.c_int32,
                                              ctypes.POINTER(ctypes.c_int32)]),
    "moe_route_topk_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int32] * 4 +
                               [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_lmhead_create": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.POINTER(ctypes.c_void_p)]),
    "moe_lmhead_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                          ctypes.c_void_p]),
    "moe_lmhead_get_weights": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_lmhead_destroy": (None, [ctypes.c_void_p]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not found at {path}: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_names():
    return list(_SIGNATURES)


# ---------------------------------------------------------------- thin wrappers

def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_last_cuda_error() -> str:
    return load().moe_last_cuda_error().decode()


def moe_layer_create(cfg: moe_layer_config_t, w: moe_layer_weights_t) -> int:
    """Returns the layer handle (int); raises MoeError on failure."""
    h = ctypes.c_void_p()
    st = load().moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    if st != MOE_OK:
        raise MoeError(st, "moe_layer_create")
    return h.value


def moe_layer_create_status(cfg: moe_layer_config_t, w: moe_layer_weights_t):
    """Like moe_layer_create but returns (status, handle or None) without raising."""
    h = ctypes.c_void_p()
    st = load().moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    return st, h.value


def moe_layer_destroy(layer: int) -> None:
    load().moe_layer_destroy(layer)


def moe_layer_forward(layer: int, x_dev: int, out_dev: int, T: int, stream: int = 0) -> int:
    return load().moe_layer_forward(layer, x_dev, out_dev, T, stream)


def moe_layer_forward_ex(layer: int, x_dev: int, out_dev: int, T: int, logit_bias_dev, stream: int = 0) -> int:
    return load().moe_layer_forward_ex(layer, x_dev, out_dev, T, logit_bias_dev, stream)


def moe_layer_forward_chunked(layer: int, x_dev: int, out_dev: int, T: int, chunk: int = 0, logit_bias_dev=None,
                              stream: int = 0) -> int:
    return load().moe_layer_forward_chunked(layer, x_dev, out_dev, T, chunk, logit_bias_dev, stream)


def moe_layer_forward_host(layer: int, x_host: int, out_host: int, T: int, logit_bias_host=None,
                           stream: int = 0) -> int:
    return load().moe_layer_forward_host(layer, x_host, out_host, T, logit_bias_host, stream)


def moe_layer_get_stats(layer: int, stream: int = 0) -> moe_stats_t:
    st = moe_stats_t()
    s = load().moe_layer_get_stats(layer, stream, ctypes.byref(st))
    if s != MOE_OK:
        raise MoeError(s, "moe_layer_get_stats")
    return st


def moe_layer_get_routing(layer: int, idx_dev, w_dev, stream: int = 0) -> int:
    return load().moe_layer_get_routing(layer, idx_dev, w_dev, stream)


def moe_layer_get_dispatch(layer: int, hist_dev, offsets_dev, perm_dev, pos_dev, stream: int = 0) -> int:
    return load().moe_layer_get_dispatch(layer, hist_dev, offsets_dev, perm_dev, pos_dev, stream)


def moe_layer_get_block_map(layer: int, blocks_dev, max_blocks: int, num_blocks_dev, stream: int = 0) -> int:
    return load().moe_layer_get_block_map(layer, blocks_dev, max_blocks, num_blocks_dev, stream)


def moe_layer_get_memory(layer: int):
    """(status, weight bytes, workspace bytes) the layer holds on the device."""
    wb, ws = ctypes.c_int64(0), ctypes.c_int64(0)
    st = load().moe_layer_get_memory(layer, ctypes.byref(wb), ctypes.byref(ws))
    return st, wb.value, ws.value


def moe_layer_sync_status(layer: int, stream: int = 0) -> int:
    return load().moe_layer_sync_status(layer, stream)


def moe_layer_profile_enable(layer: int, enable: bool) -> int:
    return load().moe_layer_profile_enable(layer, 1 if enable else 0)


def moe_layer_profile_read(layer: int, max_stages: int = 8):
    """Per-stage milliseconds of the last forward (list of floats); raises on failure."""
    buf = (ctypes.c_float * max_stages)()
    n = ctypes.c_int32()
    st = load().moe_layer_profile_read(layer, buf, max_stages, ctypes.byref(n))
    if st != MOE_OK:
        raise MoeError(st, "moe_layer_profile_read")
    return [buf[i] for i in range(n.value)]


MOE_NOALLOC_MAX_TOKENS = 8
MOE_NOALLOC_MAX_EXPERTS = 512


def moe_route_topk_noalloc(x_dev, router_t_dev, router_bias_dev, logit_bias_dev, T, H, E, k, idx_dev,
                           weights_dev, stream=0) -> int:
    return load().moe_route_topk_noalloc(x_dev, router_t_dev, router_bias_dev, logit_bias_dev, T, H, E, k,
                                         idx_dev, weights_dev, stream)


def moe_layer_describe(layer: int) -> str:
    return load().moe_layer_describe(layer).decode()


MOE_LMHEAD_MAX_T = 4
MOE_LMHEAD_MAX_HIDDEN = 8192


def moe_lmhead_create(hidden: int, vocab: int, w_dev: int):
    """Returns (status, handle or None)."""
    h = ctypes.c_void_p()
    st = load().moe_lmhead_create(hidden, vocab, w_dev, ctypes.byref(h))
    return st, h.value


def moe_lmhead_forward(head: int, x_dev: int, logits_dev: int, T: int, stream: int = 0) -> int:
    return load().moe_lmhead_forward(head, x_dev, logits_dev, T, stream)


def moe_lmhead_get_weights(head: int, codes_dev, scales_dev, stream: int = 0) -> int:
    return load().moe_lmhead_get_weights(head, codes_dev, scales_dev, stream)


def moe_lmhead_destroy(head: int) -> None:
    load().moe_lmhead_destroy(head)

