"""Python binding of libmla.so, the B300 MLA decode library.

Argument marshalling only: every computation runs in the library's CUDA
kernels.  The functions below carry the names of the C entry points in
``include/mla.h`` and take raw device pointers (ints) and sizes; ``MLA`` is a
small convenience wrapper that takes torch tensors and passes their
pointers.  Importing this package loads ``libmla.so`` and raises if it is
missing: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_CUDA = 3
MLA_ERR_WORKSPACE = 4
MLA_ERR_TIMEOUT = 5
MLA_ERR_DEVICE_INDEX = 6
MLA_BF16 = 0
MLA_FP32 = 1
MLA_KV_NATIVE = 0
MLA_KV_FP8 = 1
MLA_FP8_ROW_BYTES = 656
MLA_FORM_AUTO = 0
MLA_FORM_EXPLICIT = 1
MLA_FORM_ABSORBED = 2

EXPORTED = (
    "mla_create", "mla_destroy", "mla_compress_append", "mla_decode_workspace_size",
    "mla_decode", "mla_decode_workspace_offsets", "mla_check_status", "mla_launch_count",
    "mla_selftest_bounded_wait", "mla_status_string", "mla_profile_enable", "mla_profile_read",
    "mla_decode_static_workspace", "mla_append_decode", "mla_layer_step",
    "mla_multi_layer_step", "mla_prefill_workspace_size", "mla_prefill", "mla_prefill_form",
)


class mla_config(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int), ("d_nope", ctypes.c_int),
        ("d_v", ctypes.c_int), ("d_latent", ctypes.c_int), ("d_rope", ctypes.c_int),
        ("page_size", ctypes.c_int), ("max_position", ctypes.c_int),
        ("softmax_scale", ctypes.c_float), ("rope_base", ctypes.c_float),
        ("dtype", ctypes.c_int), ("d_cq", ctypes.c_int), ("kv_dtype", ctypes.c_int),
    ]


class mla_weights(ctypes.Structure):
    _fields_ = [("w_dkv", ctypes.c_void_p), ("w_kr", ctypes.c_void_p),
                ("w_uk", ctypes.c_void_p), ("w_uv", ctypes.c_void_p),
                ("w_o", ctypes.c_void_p), ("w_dq", ctypes.c_void_p),
                ("w_uq", ctypes.c_void_p), ("w_qr", ctypes.c_void_p)]


class MLAError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python mla_latent_kv_82_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "mla_create": ([ctypes.POINTER(mla_config), ctypes.POINTER(mla_weights), i32,
                        ctypes.POINTER(vp)], i32),
        "mla_destroy": ([vp], i32),
        "mla_compress_append": ([vp, vp, i32, i32, vp, vp, i32, vp, i32, vp], i32),
        "mla_decode_workspace_size": ([vp, i32, i32, i32], sz),
        "mla_decode": ([vp, vp, vp, i32, vp, i32, vp, i32, i32, vp, vp, sz, vp], i32),
        "mla_decode_workspace_offsets": ([vp, i32, i32, i32, ctypes.POINTER(sz),
                                          ctypes.POINTER(sz)], i32),
        "mla_check_status": ([vp, vp], i32),
        "mla_launch_count": ([vp], ctypes.c_int64),
        "mla_selftest_bounded_wait": ([vp, i32, vp], i32),
        "mla_status_string": ([i32], ctypes.c_char_p),
        "mla_profile_enable": ([vp, i32], i32),
        "mla_decode_static_workspace": ([vp, vp, vp, i32, vp, i32, vp, i32, i32, vp, vp], i32),
        "mla_append_decode": ([vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, vp, vp, sz, vp],
                              i32),
        "mla_prefill_workspace_size": ([vp, i32, i32, i32], sz),
        "mla_prefill_form": ([vp, i32, i32, i32], i32),
        "mla_prefill": ([vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, vp, vp, sz, vp], i32),
        "mla_layer_step": ([vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, vp, vp, sz, vp], i32),
        "mla_multi_layer_step": ([ctypes.POINTER(vp), i32, vp, vp, ctypes.POINTER(vp), i32, vp,
                                  i32, vp, i32, i32, vp, vp, sz, vp], i32),
        "mla_profile_read": ([vp, ctypes.POINTER(ctypes.c_float),
                              ctypes.POINTER(ctypes.c_char_p), i32], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


# ---- same-name wrappers over the C ABI --------------------------------------
def status_string(code: int) -> str:
    return _lib.mla_status_string(code).decode()


mla_status_string = status_string


def mla_create(cfg: mla_config, weights: mla_weights, device: int) -> tuple[int, int]:
    """Returns (status, ctx handle)."""
    h = ctypes.c_void_p()
    st = _lib.mla_create(ctypes.byref(cfg), ctypes.byref(weights), device, ctypes.byref(h))
    return st, h.value


def mla_destroy(ctx) -> int:
    return _lib.mla_destroy(ctx)


def mla_compress_append(ctx, h, batch, T, positions, block_table, max_pages, cache, num_pages,
                        stream) -> int:
    return _lib.mla_compress_append(ctx, h, batch, T, positions, block_table, max_pages, cache,
                                    num_pages, stream)


def mla_decode_workspace_size(ctx, batch, T, max_pages) -> int:
    return _lib.mla_decode_workspace_size(ctx, batch, T, max_pages)


def mla_decode(ctx, q, cache, num_pages, block_table, max_pages, seq_lens, batch, T, out,
               workspace, workspace_bytes, stream) -> int:
    return _lib.mla_decode(ctx, q, cache, num_pages, block_table, max_pages, seq_lens, batch, T,
                           out, workspace, workspace_bytes, stream)


def mla_append_decode(ctx, h, positions, q, cache, num_pages, block_table, max_pages, seq_lens,
                      batch, T, out, workspace, workspace_bytes, stream) -> int:
    return _lib.mla_append_decode(ctx, h, positions, q, cache, num_pages, block_table, max_pages,
                                  seq_lens, batch, T, out, workspace, workspace_bytes, stream)


def mla_prefill_workspace_size(ctx, batch, T, max_pages) -> int:
    return _lib.mla_prefill_workspace_size(ctx, batch, T, max_pages)


def mla_prefill_form(ctx, batch, T, max_pages) -> int:
    return _lib.mla_prefill_form(ctx, batch, T, max_pages)


def mla_prefill(ctx, h, positions, q, cache, num_pages, block_table, max_pages, seq_lens, batch,
                T, form, out, workspace, workspace_bytes, stream) -> int:
    return _lib.mla_prefill(ctx, h, positions, q, cache, num_pages, block_table, max_pages,
                            seq_lens, batch, T, form, out, workspace, workspace_bytes, stream)


def mla_layer_step(ctx, h, positions, cache, num_pages, block_table, max_pages, seq_lens, batch,
                   T, out, workspace, workspace_bytes, stream) -> int:
    return _lib.mla_layer_step(ctx, h, positions, cache, num_pages, block_table, max_pages,
                               seq_lens, batch, T, out, workspace, workspace_bytes, stream)


def mla_multi_layer_step(ctxs, h, positions, caches, num_pages, block_table, max_pages, seq_lens,
                         batch, T, u_scratch, workspace, workspace_bytes, stream) -> int:
    """ctxs and caches: sequences of context handles and pool pointers, one per layer."""
    n = len(ctxs)
    c_arr = (ctypes.c_void_p * n)(*ctxs)
    k_arr = (ctypes.c_void_p * n)(*caches)
    return _lib.mla_multi_layer_step(c_arr, n, h, positions, k_arr, num_pages, block_table,
                                     max_pages, seq_lens, batch, T, u_scratch, workspace,
                                     workspace_bytes, stream)


def mla_decode_static_workspace(ctx, q, cache, num_pages, block_table, max_pages, seq_lens,
                                batch, T, out, stream) -> int:
    """mla_decode with the library's static scratch instead of a workspace
    argument (for callers that cannot allocate device memory at decode time)."""
    return _lib.mla_decode_static_workspace(ctx, q, cache, num_pages, block_table, max_pages,
                                            seq_lens, batch, T, out, stream)


def mla_decode_workspace_offsets(ctx, batch, T, max_pages) -> tuple[int, int, int]:
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    st = _lib.mla_decode_workspace_offsets(ctx, batch, T, max_pages, ctypes.byref(a),
                                           ctypes.byref(b))
    return st, a.value, b.value


def mla_check_status(ctx, stream) -> int:
    return _lib.mla_check_status(ctx, stream)


def mla_launch_count(ctx) -> int:
    return _lib.mla_launch_count(ctx)


def mla_selftest_bounded_wait(ctx, spin_limit, stream) -> int:
    return _lib.mla_selftest_bounded_wait(ctx, spin_limit, stream)


def mla_profile_enable(ctx, enable: int) -> int:
    return _lib.mla_profile_enable(ctx, enable)


def mla_profile_read(ctx, max_kernels: int = 64) -> list[tuple[str, float]]:
    """[(kernel name, ms)] of the kernels enqueued since the last read."""
    ms = (ctypes.c_float * max_kernels)()
    names = (ctypes.c_char_p * max_kernels)()
    n = _lib.mla_profile_read(ctx, ms, names, max_kernels)
    if n < 0:
        raise MLAError(MLA_ERR_CUDA, "mla_profile_read")
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


# ---- torch convenience wrapper ---------------------------------------------
class MLA:
    """Owns a context over torch-held weights; passes tensor pointers through."""

    def __init__(self, dims, weights: dict, dtype: str, max_position: int, device: int = 0,
                 softmax_scale: float | None = None, kv: str = "native"):
        import torch  # noqa: F401  (tensors only provide pointers and streams)
        self.dims = dims
        self.weights = {k: v.contiguous() for k, v in weights.items()}
        self.dtype = dtype
        cfg = mla_config(dims.d_model, dims.n_heads, dims.d_nope, dims.d_v, dims.d_latent,
                         dims.d_rope, dims.page_size, max_position,
                         softmax_scale if softmax_scale is not None else dims.softmax_scale,
                         dims.rope_base, MLA_BF16 if dtype == "bf16" else MLA_FP32,
                         getattr(dims, "d_cq", 0),
                         MLA_KV_FP8 if kv == "fp8" else MLA_KV_NATIVE)
        self.kv = kv
        names = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o", "w_dq", "w_uq", "w_qr")
        w = mla_weights(*(self.weights[k].data_ptr() if k in self.weights else None
                          for k in names))
        st, self.ctx = mla_create(cfg, w, device)
        if st != MLA_OK:
            raise MLAError(st, "mla_create")
        self.device = device

    @staticmethod
    def _stream(stream):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return s.cuda_stream

    def compress_append(self, h, positions, block_table, cache, batch: int, T: int,
                        stream=None):
        st = mla_compress_append(self.ctx, h.data_ptr(), batch, T, positions.data_ptr(),
                                 block_table.data_ptr(), block_table.shape[-1],
                                 cache.data_ptr(),
                                 cache.shape[0] // self.dims.page_size, self._stream(stream))
        if st != MLA_OK:
            raise MLAError(st, "mla_compress_append")

    def workspace_size(self, batch: int, T: int, max_pages: int) -> int:
        return mla_decode_workspace_size(self.ctx, batch, T, max_pages)

    def decode(self, q, cache, block_table, seq_lens, out, workspace, stream=None):
        batch, T = q.shape[0], q.shape[1]
        st = mla_decode(self.ctx, q.data_ptr(), cache.data_ptr(),
                        cache.shape[0] // self.dims.page_size, block_table.data_ptr(),
                        block_table.shape[-1], seq_lens.data_ptr(), batch, T, out.data_ptr(),
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        self._stream(stream))
        if st != MLA_OK:
            raise MLAError(st, "mla_decode")

    def append_decode(self, h, positions, q, cache, block_table, seq_lens, out, workspace,
                      stream=None):
        batch, T = q.shape[0], q.shape[1]
        st = mla_append_decode(self.ctx, h.data_ptr(), positions.data_ptr(), q.data_ptr(),
                               cache.data_ptr(), cache.shape[0] // self.dims.page_size,
                               block_table.data_ptr(), block_table.shape[-1],
                               seq_lens.data_ptr(), batch, T, out.data_ptr(),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               self._stream(stream))
        if st != MLA_OK:
            raise MLAError(st, "mla_append_decode")

    def prefill_workspace_size(self, batch: int, T: int, max_pages: int) -> int:
        return mla_prefill_workspace_size(self.ctx, batch, T, max_pages)

    def prefill_form(self, batch: int, T: int, max_pages: int) -> int:
        return mla_prefill_form(self.ctx, batch, T, max_pages)

    def prefill(self, h, positions, q, cache, block_table, seq_lens, out, workspace,
                form=MLA_FORM_AUTO, stream=None):
        batch, T = q.shape[0], q.shape[1]
        st = mla_prefill(self.ctx, h.data_ptr(), positions.data_ptr(), q.data_ptr(),
                         cache.data_ptr(), cache.shape[0] // self.dims.page_size,
                         block_table.data_ptr(), block_table.shape[-1], seq_lens.data_ptr(),
                         batch, T, form, out.data_ptr(), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), self._stream(stream))
        if st != MLA_OK:
            raise MLAError(st, "mla_prefill")

    def layer_step(self, h, positions, cache, block_table, seq_lens, out, workspace,
                   stream=None):
        batch, T = out.shape[0], out.shape[1]
        st = mla_layer_step(self.ctx, h.data_ptr(), positions.data_ptr(), cache.data_ptr(),
                            cache.shape[0] // self.dims.page_size, block_table.data_ptr(),
                            block_table.shape[-1], seq_lens.data_ptr(), batch, T, out.data_ptr(),
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            self._stream(stream))
        if st != MLA_OK:
            raise MLAError(st, "mla_layer_step")

    def check_status(self, stream=None) -> int:
        return mla_check_status(self.ctx, self._stream(stream))

    def launch_count(self) -> int:
        return mla_launch_count(self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            mla_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
