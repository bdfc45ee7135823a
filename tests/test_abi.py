"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every entry point include/kie.h declares, and validates arguments on the host
before touching the device."""
import ctypes as C
import os
import re

import pytest

from autoregressive_decode_gb300 import kie

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "kie.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kie_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("kie_create", "kie_load_weights", "kie_prefill", "kie_decode_step", "kie_generate_greedy",
              "kie_destroy"):
        assert n in names


@pytest.mark.parametrize("lang,std,cc", [("c", "c11", "gcc"), ("c++", "c++17", "g++")])
def test_header_compiles_standalone(lang, std, cc, tmp_path):
    """include/kie.h is a self-contained C header (plain pointers and sizes, no
    torch or CUDA types): a translation unit that includes only it compiles as
    C11 and C++17 with warnings as errors, and the struct layout the Python
    binding mirrors has the size the binding expects."""
    import shutil
    import subprocess
    if shutil.which(cc) is None:
        pytest.skip(f"{cc} not available")
    ext = "c" if lang == "c" else "cpp"
    src = tmp_path / f"t.{ext}"
    src.write_text('#include "kie.h"\n#include <stdio.h>\n'
                   'int main(void) { printf("%zu\\n", sizeof(kie_config)); return 0; }\n')
    exe = tmp_path / "t"
    subprocess.check_call([cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)]).decode().strip()
    assert int(out) == C.sizeof(kie.kie_config)


def test_library_exports_every_declared_symbol():
    lib = kie.load()
    for name in declared_entry_points():
        assert hasattr(lib, name), name
    assert set(declared_entry_points()) <= set(kie.EXPORTS)


def test_invalid_configs_rejected_on_host():
    lib = kie.load()
    h = C.c_void_p()
    bad = [
        kie.make_config(0, 256, 4, 64, 1024, 4096, 64),        # no layers
        kie.make_config(2, 256, 4, 96, 1024, 4096, 64),        # head_dim 96
        kie.make_config(2, 250, 4, 64, 1024, 4096, 64),        # d not a multiple of 8
        kie.make_config(2, 256, 4, 64, 1000, 4096, 64, ffn_wdtype="int4_g128"),  # F % 128
    ]
    for cfg in bad:
        assert lib.kie_create(C.byref(cfg), None, 0, None, C.byref(h)) == kie.KIE_ERR_INVALID_ARG
        assert h.value is None
        assert lib.kie_last_error(None)
        assert lib.kie_workspace_bytes(C.byref(cfg)) == 0


def test_null_arguments():
    lib = kie.load()
    assert lib.kie_create(None, None, 0, None, None) == kie.KIE_ERR_INVALID_ARG
    assert lib.kie_prefill(None, None, 0, None) == kie.KIE_ERR_INVALID_ARG
    assert lib.kie_generate_greedy(None, 0, 1, None, None) == kie.KIE_ERR_INVALID_ARG
    assert lib.kie_sync(None) == kie.KIE_ERR_INVALID_ARG
    assert lib.kie_get_pos(None) == -1
    lib.kie_destroy(None)  # NULL-safe
    assert lib.kie_quantize_kv_u8(None, 1, 8, None, None, None) == kie.KIE_ERR_INVALID_ARG
    assert lib.kie_quantize_int4_g128(None, 1, 100, None, None) == kie.KIE_ERR_INVALID_ARG


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="only meaningful on a host without a GPU")
def test_create_without_gpu_fails_cleanly():
    lib = kie.load()
    cfg = kie.make_config(2, 256, 4, 64, 1024, 4096, 64)
    h = C.c_void_p()
    st = lib.kie_create(C.byref(cfg), None, 0, None, C.byref(h))
    assert st in (kie.KIE_ERR_CUDA, kie.KIE_ERR_LAUNCH)
    assert h.value is None
