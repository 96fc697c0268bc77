"""mla_layer_step (the decode step from the hidden states alone) vs the oracle.

The oracle makes each new token's query from its hidden state through the
query path (c^Q = W^DQ h, q^C = W^UQ c^Q, q^R = W^QR h) and then decodes it
in the explicit form (or the absorbed form on all heads at full size, with
two heads per sampled sequence also in the explicit form); the CUDA path
runs the query projections, the append and the decode through the C ABI.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import case as ocase
from oracle import mla as omla
from synth import workloads as W

from gpu_cases import check, pool_rows_of, small_bf16, tiny_f32, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
QNAMES = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o", "w_dq", "w_uq", "w_qr")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


def _run(wl):
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl, query_path=True)
    st.layer_step()
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    return st


def _oracle_q(wl, b, w64):
    """Queries of sequence b's T new tokens from their hidden states."""
    L = wl.lens[b]
    h = wl.h_rows(b, L, L + wl.T, device=DEV).to(torch.float64).cpu().numpy()
    return omla.query_from_hidden(wl.dims, h, w64["w_dq"], w64["w_uq"], w64["w_qr"])


def _compare(st, form, seqs=None, heads_explicit=0):
    wl = st.wl
    w64 = ocase.weights_f64(wl, names=QNAMES, device=DEV)
    o = st.workspace_view("o")
    d = wl.dims
    rng = np.random.default_rng(3)
    for b in (range(wl.B) if seqs is None else seqs):
        rows = ocase.sequence_rows(wl, b, w64, device=DEV)
        check(to_np(pool_rows_of(st, b)), rows, wl.dtype, f"cache rows b={b}")
        q = _oracle_q(wl, b, w64)
        fn = omla.decode_explicit if form == "explicit" else omla.decode_absorbed
        res = fn(d, rows, q, w64, wl.T)
        check(to_np(st.out[b]), res["u"], wl.dtype, f"u b={b}")
        m = slice(b * wl.T, (b + 1) * wl.T)
        check(to_np(o[m]), res["o"].reshape(wl.T, -1), wl.dtype, f"o b={b}")
        if heads_explicit:
            import dataclasses
            one = dataclasses.replace(d, n_heads=1)
            for h in rng.choice(d.n_heads, heads_explicit, replace=False):
                h = int(h)
                w1 = {"w_uk": w64["w_uk"][h * d.d_nope:(h + 1) * d.d_nope],
                      "w_uv": w64["w_uv"][h * d.d_v:(h + 1) * d.d_v],
                      "w_o": w64["w_o"][:, h * d.d_v:(h + 1) * d.d_v]}
                ref = omla.decode_explicit(one, rows, q[:, h:h + 1], w1, wl.T)["o"][:, 0]
                got = to_np(o[m, h * d.d_v:(h + 1) * d.d_v])
                check(got, ref, wl.dtype, f"o explicit b={b} head={h}")


@pytest.mark.parametrize("T,lens", [(1, [0, 63, 200, 1000]), (2, [1, 64, 300]), (1, [77]),
                                    (2, [130]), (1, [9, 200]), (3, [5, 130]), (8, [4, 70])])
def test_layer_step_small_bf16(T, lens):
    _compare(_run(small_bf16(lens, T)), "explicit")


def test_layer_step_widest_model():
    """The query path at d_model = 16384 (W^DQ and W^QR read 32 KB rows)."""
    wl = W.Workload("v2-d16384-qp", dataclasses.replace(W.V2, d_model=16384), "bf16",
                    [5, 66], 1, True)
    _compare(_run(wl), "explicit")


@pytest.mark.parametrize("T,lens", [(1, [63]), (2, [0, 30, 100])])
def test_layer_step_tiny_f32(T, lens):
    _compare(_run(tiny_f32(lens, T)), "explicit")


def test_layer_step_needs_query_weights():
    """A context made without the query path refuses the layer step."""
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(small_bf16([10], 1), prefill=False)
    with pytest.raises(m.MLAError) as e:
        st.layer_step()
    assert e.value.code == m.MLA_ERR_UNSUPPORTED
    assert st.mla.check_status() == 0


def test_layer_step_full_size_sampled():
    """The full layer step at DeepSeek-V2 widths (batch 128, 16384 cached
    tokens, two query tokens) from the hidden states alone."""
    wl = W.config("b128-l16k-t2")
    st = _run(wl)
    _compare(st, "absorbed", seqs=[0, 45, 90, 127], heads_explicit=2)
    assert torch.isfinite(st.out.float()).all()
