"""The C ABI loads, exports every declared symbol and validates arguments
before touching the GPU (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    import mla_latent_kv_82_b300 as m
    names = _declared()
    assert "mla_decode" in names and "mla_compress_append" in names
    for n in names:
        assert hasattr(m.lib(), n), n
    assert sorted(m.EXPORTED) == names


def test_status_strings():
    import mla_latent_kv_82_b300 as m
    assert m.status_string(m.MLA_OK) == "MLA_OK"
    assert m.status_string(m.MLA_ERR_TIMEOUT) == "MLA_ERR_TIMEOUT"
    assert m.status_string(99) == "MLA_ERR_UNKNOWN"


def _cfg(m, **kw):
    base = dict(d_model=5120, n_heads=128, d_nope=128, d_v=128, d_latent=512, d_rope=64,
                page_size=64, max_position=4096, softmax_scale=192 ** -0.5, rope_base=10000.0,
                dtype=m.MLA_BF16)
    base.update(kw)
    return m.mla_config(**base)


def test_create_validates_before_any_cuda_call():
    import mla_latent_kv_82_b300 as m
    w = m.mla_weights(16, 16, 16, 16, 16)       # never dereferenced
    assert m.mla_create(_cfg(m, n_heads=64), w, 0)[0] == m.MLA_ERR_UNSUPPORTED
    assert m.mla_create(_cfg(m, d_latent=256), w, 0)[0] == m.MLA_ERR_UNSUPPORTED
    assert m.mla_create(_cfg(m, d_model=5000), w, 0)[0] == m.MLA_ERR_UNSUPPORTED
    assert m.mla_create(_cfg(m, d_model=5120 + 64), w, 0)[0] == m.MLA_ERR_UNSUPPORTED
    assert m.mla_create(_cfg(m, d_rope=7), w, 0)[0] == m.MLA_ERR_INVALID_ARG
    assert m.mla_create(_cfg(m, softmax_scale=0.0), w, 0)[0] == m.MLA_ERR_INVALID_ARG
    assert m.mla_create(_cfg(m, dtype=7), w, 0)[0] == m.MLA_ERR_INVALID_ARG
    assert m.mla_create(_cfg(m, dtype=m.MLA_FP32, n_heads=129), w, 0)[0] == m.MLA_ERR_UNSUPPORTED
    w_null = m.mla_weights(16, 0, 16, 16, 16)
    assert m.mla_create(_cfg(m), w_null, 0)[0] == m.MLA_ERR_INVALID_ARG
    w_odd = m.mla_weights(16, 18, 16, 16, 16)   # bf16 weights must be 16-byte aligned
    assert m.mla_create(_cfg(m), w_odd, 0)[0] == m.MLA_ERR_INVALID_ARG
    assert m.mla_create(_cfg(m), w, -1)[0] == m.MLA_ERR_INVALID_ARG


def test_calls_reject_null_context():
    import mla_latent_kv_82_b300 as m
    assert m.mla_decode(None, 16, 16, 1, 16, 1, 16, 1, 1, 16, 256, 1 << 20, None) == \
        m.MLA_ERR_INVALID_ARG
    assert m.mla_compress_append(None, 16, 1, 1, 16, 16, 1, 16, 1, None) == m.MLA_ERR_INVALID_ARG
    assert m.mla_decode_workspace_size(None, 1, 1, 1) == 0
    assert m.mla_check_status(None, None) == m.MLA_ERR_INVALID_ARG
    assert m.mla_destroy(None) == m.MLA_ERR_INVALID_ARG
    assert m.mla_launch_count(None) == -1
    assert m.mla_selftest_bounded_wait(None, 10, None) == m.MLA_ERR_INVALID_ARG
    assert m.mla_decode_workspace_offsets(None, 1, 1, 1)[0] == m.MLA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib.util
    import shutil
    pkg = os.path.join(ROOT, "mla_latent_kv_82_b300")
    dst = tmp_path / "mla_latent_kv_82_b300"
    dst.mkdir()
    shutil.copy(os.path.join(pkg, "__init__.py"), dst / "__init__.py")
    spec = importlib.util.spec_from_file_location("mla_copy", dst / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)
