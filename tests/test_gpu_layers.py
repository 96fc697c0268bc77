"""mla_multi_layer_step (a decode step through a stack of layers) vs the oracle.

Each layer has its own seeded weights and its own cache, prefilled from its
own seeded hidden states; the new tokens' layer-0 hidden states go through
the stack with h_{j+1} = h_j + u_j.  The oracle (decode_layers, explicit
form) runs the same stack in float64 from the same inputs; the final hidden
states, the last layer's output and every layer's cache rows (whose new
rows depend on that layer's input) are compared, each within the stated
bf16 / fp32 bounds times the number of layers whose rounding reaches it.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import case as ocase
from oracle import mla as omla
from synth import workloads as W

from gpu_cases import SMALL_V2, TOL, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
QNAMES = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o", "w_dq", "w_uq", "w_qr")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


def _oracle(wl, b, form="explicit"):
    d = wl.dims
    L = wl.lens[b]
    layers = []
    for j in range(wl.layers):
        w = {n: wl.weight(n, device=DEV, layer=j).to(torch.float64).cpu().numpy() for n in QNAMES}
        h = wl.h_rows(b, 0, L, device=DEV, layer=j).to(torch.float64).cpu().numpy()
        rows = omla.latent_rows(h, w["w_dkv"], w["w_kr"], np.arange(L), d.rope_base)
        layers.append({"w": w, "prefix_rows": rows})
    h_new = wl.h_rows(b, L, L + wl.T, device=DEV).to(torch.float64).cpu().numpy()
    return layers, h_new, omla.decode_layers(d, layers, h_new, wl.T, form=form)


def _pool_rows(st, j, b):
    wl = st.wl
    P = wl.dims.page_size
    pos = torch.arange(wl.seq_lens[b], device=st.dev)
    return st.caches[j][st.bt[b, pos // P].long() * P + pos % P]


def _check_depth(got, ref, wl, depth, what):
    s = omla.error_stats(to_np(got), ref)
    mx, mean = TOL[wl.dtype]
    k = max(1, depth)
    assert s["max_rel"] <= mx * k and s["mean_rel"] <= mean * k, f"{what}: {s}"
    return s


def _run_and_compare(wl, form="explicit", seqs=None):
    from mla_latent_kv_82_b300.workload import StackState
    st = StackState(wl)
    st.step()
    torch.cuda.synchronize()
    assert st.check_status() == 0
    d = wl.dims
    for b in (range(wl.B) if seqs is None else seqs):
        layers, h_new, ref = _oracle(wl, b, form)
        m = slice(b * wl.T, (b + 1) * wl.T)
        # A quantity that depends on the outputs of j layers carries the
        # rounding of each of them (each layer's output is the next layer's
        # input): to first order the per-layer bounds add, so it is held to
        # the stated single-layer bounds times max(1, j).
        _check_depth(st.h[m], ref["h"], wl, wl.layers, f"h_L b={b}")
        _check_depth(st.u[m], ref["u"][-1], wl, wl.layers, f"u of the last layer b={b}")
        # layer j's cache: its prefix rows, then the rows of its own input h_j
        h = h_new
        for j, layer in enumerate(layers):
            S = wl.seq_lens[b]
            new = omla.latent_rows(h, layer["w"]["w_dkv"], layer["w"]["w_kr"],
                                   np.arange(S - wl.T, S), d.rope_base)
            rows = np.concatenate([layer["prefix_rows"], new])
            _check_depth(_pool_rows(st, j, b), rows, wl, j, f"cache of layer {j} b={b}")
            h = h + ref["u"][j]
    return st


@pytest.mark.parametrize("T,lens", [(1, [0, 70, 300]), (2, [1, 130])])
def test_layer_stack_small_bf16(T, lens):
    wl = W.Workload(f"v2-small-stack-T{T}", SMALL_V2, "bf16", lens, T, True, layers=3)
    _run_and_compare(wl)


def test_layer_stack_tiny_f32():
    wl = W.Workload("tiny-stack", dataclasses.replace(W.TINY, page_size=16), "f32",
                    [0, 20, 47], 1, True, layers=2)
    _run_and_compare(wl)


def test_layer_stack_v2_widths():
    """Two layers at DeepSeek-V2 widths on the batch-1, 4096-token cache."""
    wl = dataclasses.replace(W.config("b1-l4096-x60"), layers=2)
    _run_and_compare(wl, form="absorbed")


def test_layer_stack_rejects_a_context_without_query_path():
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(W.Workload("p", SMALL_V2, "bf16", [10], 1, False), prefill=False)
    u = torch.empty_like(st.out)
    h = torch.zeros((1, SMALL_V2.d_model), dtype=torch.bfloat16, device=DEV)
    rc = m.mla_multi_layer_step([st.mla.ctx], h.data_ptr(), st.pos_new.data_ptr(),
                                [st.cache.data_ptr()], st.num_pages, st.bt.data_ptr(),
                                st.bt.shape[1], st.seq_lens.data_ptr(), 1, 1, u.data_ptr(),
                                st.ws.data_ptr(), st.ws_bytes,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == m.MLA_ERR_UNSUPPORTED
    assert st.mla.check_status() == 0
