"""include/mla.h is a C header: a C11 translation unit built with
-Wall -Wextra -Werror -pedantic includes it and links against libmla.so
(no CUDA call is made), and the layouts it sees agree with the ctypes
binding: every field offset and the size of mla_config and mla_weights, and
every constant the binding mirrors (CPU only)."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mla_latent_kv_82_b300")

CONFIG = ["d_model", "n_heads", "d_nope", "d_v", "d_latent", "d_rope", "page_size",
          "max_position", "softmax_scale", "rope_base", "dtype", "d_cq", "kv_dtype"]
WEIGHTS = ["w_dkv", "w_kr", "w_uk", "w_uv", "w_o", "w_dq", "w_uq", "w_qr"]
CONSTANTS = ["MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_UNSUPPORTED", "MLA_ERR_CUDA",
             "MLA_ERR_WORKSPACE", "MLA_ERR_TIMEOUT", "MLA_ERR_DEVICE_INDEX", "MLA_BF16",
             "MLA_FP32", "MLA_KV_NATIVE", "MLA_KV_FP8", "MLA_FP8_ROW_BYTES", "MLA_FORM_AUTO",
             "MLA_FORM_EXPLICIT", "MLA_FORM_ABSORBED"]


def _program():
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "mla.h"', "int main(void) {"]
    lines.append('  printf("config_size %zu\\n", sizeof(mla_config));')
    for f in CONFIG:
        lines.append(f'  printf("config.{f} %zu\\n", offsetof(mla_config, {f}));')
    lines.append('  printf("weights_size %zu\\n", sizeof(mla_weights));')
    for f in WEIGHTS:
        lines.append(f'  printf("weights.{f} %zu\\n", offsetof(mla_weights, {f}));')
    for c in CONSTANTS:
        lines.append(f'  printf("{c} %d\\n", (int){c});')
    # calls through the C linkage that return before any CUDA call
    lines += ["  mla_ctx* ctx = NULL;",
              '  printf("create_null %d\\n", (int)mla_create(NULL, NULL, 0, &ctx));',
              '  printf("ctx_after %d\\n", ctx == NULL);',
              '  printf("timeout_string %s\\n", mla_status_string(MLA_ERR_TIMEOUT));',
              "  return 0;", "}"]
    return "\n".join(lines) + "\n"


@pytest.fixture(scope="module")
def seen(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("needs gcc")
    lib = os.path.join(PKG, "libmla.so")
    if not os.path.exists(lib):
        pytest.skip("libmla.so not built")
    d = tmp_path_factory.mktemp("header_c")
    src, exe = d / "abi.c", d / "abi"
    src.write_text(_program())
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", PKG, "-lmla", f"-Wl,-rpath,{PKG}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return dict(line.split(" ", 1) for line in out.strip().splitlines())


def test_struct_layouts_match_the_binding(seen):
    import mla_latent_kv_82_b300 as m
    assert int(seen["config_size"]) == ctypes.sizeof(m.mla_config)
    assert [f for f, _ in m.mla_config._fields_] == CONFIG
    for f in CONFIG:
        assert int(seen[f"config.{f}"]) == getattr(m.mla_config, f).offset, f
    assert int(seen["weights_size"]) == ctypes.sizeof(m.mla_weights)
    assert [f for f, _ in m.mla_weights._fields_] == WEIGHTS
    for f in WEIGHTS:
        assert int(seen[f"weights.{f}"]) == getattr(m.mla_weights, f).offset, f


def test_constants_match_the_binding(seen):
    import mla_latent_kv_82_b300 as m
    for c in CONSTANTS:
        assert int(seen[c]) == getattr(m, c), c


def test_c_linkage_calls(seen):
    import mla_latent_kv_82_b300 as m
    assert int(seen["create_null"]) == m.MLA_ERR_INVALID_ARG
    assert seen["ctx_after"] == "1"
    assert seen["timeout_string"] == "MLA_ERR_TIMEOUT"
