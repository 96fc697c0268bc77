"""The FP8 latent cache (MLA_KV_FP8) vs the oracle, through the C ABI.

The oracle quantises its own fp64 rows (oracle.fp8.quantize_rows) and runs
the unchanged explicit decode over the dequantised rows.  Checked:

* the pool bytes: E4M3 codes, the row scale and the stored k^R / s against
  the oracle's; the decision is taken in fp32 on both sides, from values
  that may differ in their last bit (fp32 accumulation order), so a row's
  scale may differ by one bf16 step of its maximum and a code by one step;
  everything else is exact, and untouched rows keep their bytes;
* u against the oracle's decode over the dequantised cache, within the FP8
  bounds: the kernels round each head's absorbed query to E4M3 (relative
  error up to 2^-4 per element, about 2^-4/sqrt(3) rms), which moves each
  logit by a few hundredths of the logits' spread; u is held to
  max|err| <= 0.1 max|ref| and sum|err| / sum|ref| <= 0.03;
* the format's own cost: u over the FP8 cache against the exact decode.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import case as ocase
from oracle import fp8
from oracle import mla as omla
from synth import workloads as W

from gpu_cases import small_bf16, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL_FP8 = (0.1, 0.03)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


def _run(wl, sentinel=None):
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl, kv="fp8", sentinel=sentinel)
    st.step()
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    return st


def _pool_bytes(st, b):
    wl = st.wl
    P = wl.dims.page_size
    pos = torch.arange(wl.seq_lens[b], device=st.dev)
    return st.cache[st.bt[b, pos // P].long() * P + pos % P].cpu().numpy()


def _split(raw):
    codes = raw[:, :512]
    kr = torch.from_numpy(np.ascontiguousarray(raw[:, 512:640])).view(torch.bfloat16)
    scale = np.ascontiguousarray(raw[:, 640:644]).view(np.float32)[:, 0]
    return codes, kr.float().numpy(), scale, raw[:, 644:656]


def check_rows(raw, q):
    """GPU pool bytes of a sequence vs the oracle's quantised rows."""
    codes, kr, scale, pad = _split(raw)
    assert not pad.any()
    same = scale == q["scale"]
    # a differing scale comes from a maximum one bf16 step away
    assert np.all(np.abs(scale[~same] / q["scale"][~same] - 1) <= 2.0 ** -7)
    assert (~same).mean() <= 0.02, (~same).sum()
    if same.any():
        v_gpu = fp8.e4m3_decode(codes[same])
        v_ora = fp8.e4m3_decode(q["codes"][same])
        diff = v_gpu != v_ora
        assert diff.mean() <= 1e-3, diff.sum()
        # a differing code is the neighbour of the oracle's
        mag = np.maximum(np.abs(v_ora), 2.0 ** -6)
        step = np.exp2(np.floor(np.log2(mag))) / 8.0
        assert np.all(np.abs(v_gpu - v_ora)[diff] <= step[diff] * 1.0001)
        k_ok = np.abs(kr[same] - q["kr"][same]) <= 2.0 ** -7 * np.abs(q["kr"][same]) + 1e-30
        assert k_ok.mean() >= 0.999
    return same


def _compare(st, seqs=None, exact_too=False):
    wl = st.wl
    w64 = ocase.weights_f64(wl, device=DEV)
    q64 = to_np(st.q)
    stats = []
    for b in (range(wl.B) if seqs is None else seqs):
        rows = ocase.sequence_rows(wl, b, w64, device=DEV)
        q = fp8.quantize_rows(rows, wl.dims.d_latent)
        check_rows(_pool_bytes(st, b), q)
        ref = omla.decode_explicit(wl.dims, q["deq"], q64[b], w64, wl.T)
        s = omla.error_stats(to_np(st.out[b]), ref["u"])
        assert s["max_rel"] <= TOL_FP8[0] and s["mean_rel"] <= TOL_FP8[1], f"u b={b}: {s}"
        if exact_too:
            ex = omla.decode_explicit(wl.dims, rows, q64[b], w64, wl.T)
            s["vs_exact"] = omla.error_stats(to_np(st.out[b]), ex["u"])
            assert s["vs_exact"]["mean_rel"] <= 0.06, s
        stats.append(s)
    return stats


@pytest.mark.parametrize("T,lens", [
    (1, [0, 62, 63, 64, 200, 1000]),
    (2, [0, 62, 63, 127, 500]),
    (3, [2, 64, 190]),
    (1, [300]),
    (2, [200]),
    (1, [70, 1]),
    (4, [3, 130, 260]),
    (5, [63]),
    (8, [0, 100]),      # the largest decode T
])
def test_small_fp8(T, lens):
    _compare(_run(small_bf16(lens, T)), exact_too=True)


def test_append_placement_and_untouched_rows():
    """Only the sequences' rows change; every other pool byte keeps the
    sentinel, and written rows have zero padding."""
    wl = small_bf16([5, 70, 129], 2)
    st = _run(wl, sentinel=0xA5)
    P = wl.dims.page_size
    written = np.zeros(st.cache.shape[0], dtype=bool)
    for b, S in enumerate(wl.seq_lens):
        pos = np.arange(S)
        written[st.bt[b, pos // P].long().cpu().numpy() * P + pos % P] = True
    pool = st.cache.cpu().numpy()
    assert np.all(pool[~written] == 0xA5)
    assert not pool[written][:, 644:].any()
    _compare(st)


def test_separate_append_then_decode_equals_one_call():
    """mla_compress_append then mla_decode gives the same bytes as
    mla_append_decode: the same kernels on the same inputs."""
    from mla_latent_kv_82_b300.workload import DeviceState
    wl = small_bf16([40, 200], 2)
    a = DeviceState(wl, kv="fp8")
    a.step()
    b = DeviceState(wl, kv="fp8")
    b.step_separate()
    torch.cuda.synchronize()
    assert a.mla.check_status() == 0 and b.mla.check_status() == 0
    assert torch.equal(a.cache, b.cache)
    assert torch.equal(a.out.view(torch.uint16), b.out.view(torch.uint16))


@pytest.mark.parametrize("name,seqs", [("b64-paged", [0, 21, 40, 63]), ("b4-l128k", [0, 3]),
                                       ("b128-l16k-t2", [0, 77, 127])])
def test_full_size_sampled(name, seqs):
    """Full-size workloads on the FP8 cache (prefill through chunked appends
    of 4096-token passes), sampled sequences against the oracle."""
    st = _run(W.config(name))
    stats = _compare(st, seqs=seqs)
    assert len(stats) == len(seqs)
    assert torch.isfinite(st.out.float()).all()


def test_prefill_chunk_on_fp8_cache():
    """mla_prefill on an FP8 cache: the automatic choice is the absorbed
    form (the explicit form reads bf16 rows and is refused)."""
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState
    wl = small_bf16([0, 90], 200)
    st = DeviceState(wl, kv="fp8")
    assert st.mla.prefill_form(wl.B, wl.T, st.bt.shape[1]) == m.MLA_FORM_ABSORBED
    st.prefill_chunk(m.MLA_FORM_AUTO)
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    _compare(st)
    with pytest.raises(m.MLAError) as e:
        st.prefill_chunk(m.MLA_FORM_EXPLICIT)
    assert e.value.code == m.MLA_ERR_UNSUPPORTED


def test_fp8_needs_a_bf16_context():
    import dataclasses
    import mla_latent_kv_82_b300 as m
    d = dataclasses.replace(W.TINY, page_size=16)
    wl = W.Workload("tiny", d, "f32", [3], 1, False)
    w = {n: wl.weight(n, device=DEV) for n in ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o")}
    with pytest.raises(m.MLAError) as e:
        m.MLA(dataclasses.replace(d, d_cq=0), w, "f32", max_position=8, kv="fp8")
    assert e.value.code == m.MLA_ERR_UNSUPPORTED


QNAMES = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o", "w_dq", "w_uq", "w_qr")


def test_layer_step_on_fp8_cache():
    """mla_layer_step (queries from the hidden states) over an FP8 pool: the
    oracle makes the queries with query_from_hidden and decodes over its own
    quantised rows."""
    from mla_latent_kv_82_b300.workload import DeviceState
    wl = W.Workload("v2-small-qp-fp8", dataclasses.replace(W.V2, d_model=512), "bf16",
                    [0, 70, 300], 2, True)
    st = DeviceState(wl, query_path=True, kv="fp8")
    st.layer_step()
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    w64 = ocase.weights_f64(wl, names=QNAMES, device=DEV)
    for b in range(wl.B):
        rows = ocase.sequence_rows(wl, b, w64, device=DEV)
        q = fp8.quantize_rows(rows, wl.dims.d_latent)
        check_rows(_pool_bytes(st, b), q)
        L = wl.lens[b]
        h = wl.h_rows(b, L, L + wl.T, device=DEV).to(torch.float64).cpu().numpy()
        qq = omla.query_from_hidden(wl.dims, h, w64["w_dq"], w64["w_uq"], w64["w_qr"])
        ref = omla.decode_explicit(wl.dims, q["deq"], qq, w64, wl.T)
        s = omla.error_stats(to_np(st.out[b]), ref["u"])
        assert s["max_rel"] <= TOL_FP8[0] and s["mean_rel"] <= TOL_FP8[1], f"u b={b}: {s}"


def test_layer_stack_on_fp8_cache():
    """mla_multi_layer_step through three layers with FP8 pools: the oracle
    runs the stack (h_{j+1} = h_j + u_j) with every layer's rows, cached and
    new, quantised as the pools hold them.  Each layer's rounding reaches the
    next layer's input, so to first order the per-layer bounds add: the final
    h is held to the FP8 bounds times the number of layers."""
    from mla_latent_kv_82_b300.workload import StackState
    wl = W.Workload("v2-small-stack-fp8", dataclasses.replace(W.V2, d_model=512), "bf16",
                    [5, 130], 1, True, layers=3)
    st = StackState(wl, kv="fp8")
    st.step()
    torch.cuda.synchronize()
    assert st.check_status() == 0
    d = wl.dims
    for b in range(wl.B):
        L, S = wl.lens[b], wl.seq_lens[b]
        h = wl.h_rows(b, L, L + wl.T, device=DEV).to(torch.float64).cpu().numpy()
        for j in range(wl.layers):
            w = {n: wl.weight(n, device=DEV, layer=j).to(torch.float64).cpu().numpy()
                 for n in QNAMES}
            hp = wl.h_rows(b, 0, L, device=DEV, layer=j).to(torch.float64).cpu().numpy()
            rows = np.concatenate([
                omla.latent_rows(hp, w["w_dkv"], w["w_kr"], np.arange(L), d.rope_base),
                omla.latent_rows(h, w["w_dkv"], w["w_kr"], np.arange(L, S), d.rope_base)])
            deq = fp8.quantize_rows(rows, d.d_latent)["deq"]
            q = omla.query_from_hidden(d, h, w["w_dq"], w["w_uq"], w["w_qr"])
            u = omla.decode_explicit(d, deq, q, w, wl.T)["u"]
            h = h + u
        m = slice(b * wl.T, (b + 1) * wl.T)
        s = omla.error_stats(to_np(st.h[m]), h)
        k = wl.layers
        assert s["max_rel"] <= TOL_FP8[0] * k and s["mean_rel"] <= TOL_FP8[1] * k, f"h b={b}: {s}"
