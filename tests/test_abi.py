"""The C-ABI library builds, loads and exports every function include/moe_layer.h declares (CPU only)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_layer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    from sparse_mixture_experts_gemv_gb300 import build as b
    lib_path = b.build()
    lib = ctypes.CDLL(lib_path)
    names = _declared()
    assert "moe_layer_forward" in names and "moe_layer_create" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    from sparse_mixture_experts_gemv_gb300 import _native as N
    assert sorted(N.exported_names()) == names  # the binding covers the whole header


def test_status_strings_without_gpu():
    from sparse_mixture_experts_gemv_gb300 import _native as N
    assert N.moe_status_string(N.MOE_ERR_TIMEOUT) == "MOE_ERR_TIMEOUT"
    assert N.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_create_rejects_bad_config_before_touching_the_device():
    from sparse_mixture_experts_gemv_gb300 import _native as N
    cfg = N.moe_layer_config_t(256, 16, 17, 128, 128, 8, 0, 0)  # k > E
    st, h = N.moe_layer_create_status(cfg, N.moe_layer_weights_t())
    assert st == N.MOE_ERR_INVALID_ARG and h is None
    cfg = N.moe_layer_config_t(256, 16, 2, 128, 128, 8, 7, 0)  # unknown format
    st, h = N.moe_layer_create_status(cfg, N.moe_layer_weights_t())
    assert st == N.MOE_ERR_INVALID_ARG


def test_header_is_plain_c99(tmp_path):
    """include/moe_layer.h compiles as C99 with warnings as errors (a C caller needs
    no C++ or CUDA headers), and a C program links against libmoe.so."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        import pytest
        pytest.skip("gcc not available")
    src = tmp_path / "use_header.c"
    src.write_text(
        '#include "moe_layer.h"\n'
        "int main(void) {\n"
        "  moe_layer_config_t c = {0};\n"
        "  moe_layer_t* L = 0;\n"
        "  (void)c;\n"
        "  if (moe_layer_create(0, 0, &L) != MOE_ERR_INVALID_ARG) return 1;\n"
        "  return moe_status_string(MOE_OK)[0] == 'M' ? 0 : 2;\n"
        "}\n")
    inc = os.path.join(ROOT, "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, "-fsyntax-only",
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    from sparse_mixture_experts_gemv_gb300 import build as b
    lib = b.build()
    exe = tmp_path / "use_header"
    r = subprocess.run([gcc, "-std=c99", "-I", inc, str(src), "-o", str(exe), lib,
                        "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_new_entry_points_reject_bad_arguments_before_touching_the_device():
    import ctypes
    from sparse_mixture_experts_gemv_gb300 import _native as N
    fake = 0x10000   # never dereferenced: every case below fails validation first
    # chunked forward without a layer
    assert N.moe_layer_forward_chunked(None, fake, fake, 10, 0, None, 0) == N.MOE_ERR_INVALID_ARG
    # LM head: hidden not a multiple of 256, empty vocabulary, missing or misaligned weights
    assert N.moe_lmhead_create(250, 10, fake)[0] == N.MOE_ERR_UNSUPPORTED
    assert N.moe_lmhead_create(256 * 33, 10, fake)[0] == N.MOE_ERR_UNSUPPORTED   # above the hidden limit
    assert N.moe_lmhead_create(256, 0, fake)[0] == N.MOE_ERR_INVALID_ARG
    assert N.moe_lmhead_create(256, 10, 0)[0] == N.MOE_ERR_INVALID_ARG
    assert N.moe_lmhead_create(256, 10, fake + 2)[0] == N.MOE_ERR_INVALID_ARG
    assert N.moe_lmhead_forward(None, fake, fake, 1, 0) == N.MOE_ERR_INVALID_ARG
    assert N.moe_lmhead_get_weights(None, None, None, 0) == N.MOE_ERR_INVALID_ARG
    N.moe_lmhead_destroy(None)
    # int4 layers need scales and biases
    cfg = N.moe_layer_config_t(256, 16, 2, 128, 128, 8, N.MOE_WEIGHTS_INT4, 0)
    w = N.moe_layer_weights_t()
    for f in ("router_dev", "gate_dev", "up_dev", "down_dev", "gate_scales_dev", "up_scales_dev",
              "down_scales_dev", "shared_gate_dev", "shared_up_dev", "shared_down_dev"):
        setattr(w, f, fake)
    st, h = N.moe_layer_create_status(cfg, w)
    assert st == N.MOE_ERR_INVALID_ARG and h is None
    cfg3 = N.moe_layer_config_t(256, 16, 2, 128, 128, 8, 3, 0)   # no format 3
    assert N.moe_layer_create_status(cfg3, w)[0] == N.MOE_ERR_INVALID_ARG
