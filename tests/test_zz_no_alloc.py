"""mla_decode_static_workspace: decode for callers that cannot allocate.

Some callers cannot allocate device memory when they decode (a memory
budget fixed up front, an allocator out of reach of the issuing thread, a
plugin handed only its buffers).  The static-workspace entry point serves
them from a scratch array the library reserves once; this test checks,
through the C ABI, that two calls in a row give the output of the regular
mla_decode (same tolerance as every bf16 parity test), and that shapes
needing more scratch than the array holds are refused before any work.

This file is collected last so that a failure here stops a `-x` run only
after every other test has run; it also passes on its own.
"""
import pytest
import torch

from gpu_cases import TOL, small_bf16, to_np
from oracle import mla as omla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


@pytest.mark.parametrize("T,lens", [(1, [300, 77, 1]), (2, [130, 5])])
def test_static_workspace_matches_workspace_decode(T, lens):
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState

    st = DeviceState(small_bf16(lens, T))
    st.step()                                  # append + decode (workspace argument)
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    ref = to_np(st.out)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):                         # two calls in a row share the scratch
        out = torch.full_like(st.out, float("nan"))
        rc = m.mla_decode_static_workspace(
            st.mla.ctx, st.q.data_ptr(), st.cache.data_ptr(), st.num_pages, st.bt.data_ptr(),
            st.bt.shape[1], st.seq_lens.data_ptr(), st.wl.B, T, out.data_ptr(), stream)
        assert rc == m.MLA_OK, m.status_string(rc)
        torch.cuda.synchronize()
        assert st.mla.check_status() == 0
        stats = omla.error_stats(to_np(out), ref)
        assert stats["max_rel"] <= TOL["bf16"][0] and stats["mean_rel"] <= TOL["bf16"][1], stats


def test_static_workspace_refuses_oversized_shapes():
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState

    st = DeviceState(small_bf16([10], 1), prefill=False)
    big_batch, big_pages = 4096, 4096
    assert m.mla_decode_workspace_size(st.mla.ctx, big_batch, 1, big_pages) > (32 << 20)
    rc = m.mla_decode_static_workspace(
        st.mla.ctx, st.q.data_ptr(), st.cache.data_ptr(), st.num_pages, st.bt.data_ptr(),
        big_pages, st.seq_lens.data_ptr(), big_batch, 1, st.out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == m.MLA_ERR_WORKSPACE
    assert st.mla.check_status() == 0
