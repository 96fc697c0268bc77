"""mla_decode_static_workspace: decode for callers that cannot allocate.

Some callers cannot allocate device memory when they decode (a memory
budget fixed up front, an allocator out of reach of the issuing thread, a
plugin handed only its buffers).  The static-workspace entry point serves
them from a scratch array the library reserves once.  This test checks,
through the C ABI, that two calls in a row give the output of the regular
mla_decode byte for byte (both run the same kernels on the same inputs),
starting from scratch that an earlier, larger call left dirty, and that a
shape needing more scratch than the array holds is refused before anything
is enqueued.

This file is collected last so that a failure here stops a `-x` run only
after every other test has run; it also passes on its own.
"""
import pytest
import torch

from gpu_cases import small_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


def _static_decode(st, out):
    import mla_latent_kv_82_b300 as m
    return m.mla_decode_static_workspace(
        st.mla.ctx, st.q.data_ptr(), st.cache.data_ptr(), st.num_pages, st.bt.data_ptr(),
        st.bt.shape[1], st.seq_lens.data_ptr(), st.wl.B, st.wl.T, out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _dirty_scratch():
    """A larger static-workspace call first, so the scratch holds non-zero
    leftovers (plan arrays, partials, query images) when the checked calls run."""
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState

    big = DeviceState(small_bf16([900, 1500, 64, 700, 333, 1000, 5, 1200], 2))
    assert big.ws_bytes <= (32 << 20)
    big.append_new()
    out = torch.empty_like(big.out)
    assert _static_decode(big, out) == m.MLA_OK
    torch.cuda.synchronize()
    assert big.mla.check_status() == 0
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("T,lens", [(1, [300, 77, 1]), (2, [130, 5])])
def test_static_workspace_matches_workspace_decode(T, lens):
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState

    _dirty_scratch()
    st = DeviceState(small_bf16(lens, T))
    st.step()                                  # append + decode (workspace argument)
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    ref = st.out.clone()
    for _ in range(2):                         # two calls in a row share the scratch
        out = torch.full_like(st.out, float("nan"))
        rc = _static_decode(st, out)
        assert rc == m.MLA_OK, m.status_string(rc)
        torch.cuda.synchronize()
        assert st.mla.check_status() == 0
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))


def test_static_workspace_refuses_oversized_shapes():
    """batch 256 with one page each: the query images alone exceed the
    array; every buffer of the call is really allocated at that size."""
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState

    st = DeviceState(small_bf16([10], 1), prefill=False)
    d = st.wl.dims
    batch, T, max_pages = 256, 1, 1
    assert m.mla_decode_workspace_size(st.mla.ctx, batch, T, max_pages) > (32 << 20)
    q = torch.zeros((batch, T, d.n_heads, d.d_nope + d.d_rope), dtype=torch.bfloat16,
                    device=st.dev)
    bt = torch.zeros((batch, max_pages), dtype=torch.int32, device=st.dev)
    seq_lens = torch.ones((batch,), dtype=torch.int32, device=st.dev)
    out = torch.zeros((batch, T, d.d_model), dtype=torch.bfloat16, device=st.dev)
    torch.cuda.synchronize()
    before = st.mla.launch_count()
    rc = m.mla_decode_static_workspace(
        st.mla.ctx, q.data_ptr(), st.cache.data_ptr(), st.num_pages, bt.data_ptr(), max_pages,
        seq_lens.data_ptr(), batch, T, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == m.MLA_ERR_WORKSPACE
    assert st.mla.launch_count() == before
    assert st.mla.check_status() == 0
    assert not out.any()
