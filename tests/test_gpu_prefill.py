"""mla_prefill (a chunk of T new tokens per sequence) vs the oracle.

The chunk's tokens are appended and attended to with the causal mask inside
the chunk; the oracle is the explicit decode of the same T tokens
(decode_explicit: query t at position S - T + t sees positions 0..S-T+t).
Both forms of the library (explicit: K^C, V up-projected per head; absorbed:
the decode kernels) and the automatic choice are compared on small cases
with every token, and at DeepSeek-V2 widths on sampled tokens computed by the
oracle one at a time.
"""
import pytest
import torch

from oracle import case as ocase
from oracle import mla as omla
from synth import workloads as W

from gpu_cases import check, pool_rows_of, small_bf16, tiny_f32, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
FORMS = {"auto": 0, "explicit": 1, "absorbed": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


def _run(wl, form):
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl)
    st.prefill_chunk(FORMS[form])
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    return st


def _compare_all(st):
    wl = st.wl
    w64 = ocase.weights_f64(wl, device=DEV)
    q64 = to_np(st.q)
    for b in range(wl.B):
        rows = ocase.sequence_rows(wl, b, w64, device=DEV)
        ref = omla.decode_explicit(wl.dims, rows, q64[b], w64, wl.T)
        check(to_np(pool_rows_of(st, b)), rows, wl.dtype, f"cache rows b={b}")
        check(to_np(st.out[b]), ref["u"], wl.dtype, f"u b={b}")


@pytest.mark.parametrize("form", ["explicit", "absorbed", "auto"])
@pytest.mark.parametrize("T,lens", [
    (200, [0, 70, 300]),   # two query tiles, ragged key tiles, an empty prefix
    (130, [1]),            # one token past a query tile
    (64, [0, 65]),         # a chunk of one page
    (257, [63]),           # odd T (single-token attention clusters when absorbed)
])
def test_small_bf16(form, T, lens):
    _compare_all(_run(small_bf16(lens, T), form))


def test_tiny_f32_absorbed_and_explicit_rejected():
    import mla_latent_kv_82_b300 as m
    wl = tiny_f32([0, 20, 47], 40)
    st = _run(wl, "auto")
    _compare_all(st)
    with pytest.raises(m.MLAError) as e:
        st.prefill_chunk(FORMS["explicit"])
    assert e.value.code == m.MLA_ERR_UNSUPPORTED


def test_argument_errors():
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState
    wl = small_bf16([10, 100], 70)
    st = DeviceState(wl)
    need = st.mla.prefill_workspace_size(wl.B, wl.T, st.bt.shape[1])
    assert need >= st.mla.workspace_size(wl.B, wl.T, st.bt.shape[1])
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    args = [st.mla.ctx, st.h_new.data_ptr(), st.pos_new.data_ptr(), st.q.data_ptr(),
            st.cache.data_ptr(), st.num_pages, st.bt.data_ptr(), st.bt.shape[1],
            st.seq_lens.data_ptr(), wl.B, wl.T, 1, st.out.data_ptr()]
    assert m.mla_prefill(*args, small.data_ptr(), need - 256, stream) == m.MLA_ERR_WORKSPACE
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    bad_form = list(args)
    bad_form[11] = 3
    assert m.mla_prefill(*bad_form, ws.data_ptr(), need, stream) == m.MLA_ERR_INVALID_ARG
    too_long = list(args)
    too_long[10] = 4097
    assert m.mla_prefill(*too_long, ws.data_ptr(), need, stream) == m.MLA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0


def _sampled(st, picks):
    """u of sampled (sequence, token) pairs, each from the oracle alone: the
    rows up to the token's own position and its one query."""
    wl = st.wl
    w64 = ocase.weights_f64(wl, device=DEV)
    q64 = to_np(st.q)
    for b, ts in picks.items():
        rows = ocase.sequence_rows(wl, b, w64, device=DEV)
        S = wl.seq_lens[b]
        for t in ts:
            p = S - wl.T + t
            ref = omla.decode_explicit(wl.dims, rows[:p + 1], q64[b, t:t + 1], w64, 1)
            check(to_np(st.out[b, t:t + 1]), ref["u"], wl.dtype, f"u b={b} t={t}")


@pytest.mark.parametrize("form", ["explicit", "auto"])
def test_v2_widths_chunk_of_1024(form):
    """DeepSeek-V2 widths: a 1024-token chunk after prefixes of 0 and 2000
    (the automatic choice takes the explicit form here)."""
    wl = W.Workload("v2-chunk-1024", W.V2, "bf16", [0, 2000], 1024, True)
    st = _run(wl, form)
    _sampled(st, {0: [0, 1, 127, 128, 700, 1023], 1: [0, 255, 511, 1022, 1023]})
    assert torch.isfinite(st.out.float()).all()


def test_v2_widths_forms_agree():
    """The two forms on the same 384-token chunk: each against sampled oracle
    tokens, and the two outputs against each other."""
    wl = W.Workload("v2-chunk-384", W.V2, "bf16", [500], 384, True)
    outs = {}
    for form in ("explicit", "absorbed"):
        st = _run(wl, form)
        _sampled(st, {0: [0, 100, 383]})
        outs[form] = to_np(st.out)
        del st
        torch.cuda.empty_cache()
    s = omla.error_stats(outs["explicit"], outs["absorbed"])
    assert s["max_rel"] <= 2e-2 and s["mean_rel"] <= 5e-3, s


def test_automatic_form_choice():
    """mla_prefill_form names the form MLA_FORM_AUTO runs: the explicit form
    for prompts on an empty cache, the absorbed form for decode-sized chunks
    and for short chunks after a long prefix; an automatic call launches the
    kernels of the form it names."""
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState
    E, A = m.MLA_FORM_EXPLICIT, m.MLA_FORM_ABSORBED
    st = DeviceState(small_bf16([0], 128))
    f = st.mla.prefill_form
    assert f(1, 128, 2) == E          # a 128-token prompt
    assert f(4, 4096, 64) == E        # four 4096-token prompts
    assert f(1, 1, 64) == A           # one token
    assert f(128, 2, 257) == A        # batched decode on 16K caches
    assert f(1, 256, 200) == A        # 256 tokens after a 12544-token prefix
    assert f(1, 1024, 208) == E       # 1024 tokens after 12288
    assert f(64, 128, 8192) == A      # past the explicit form's row bound
    assert f(1, 0, 2) == -1
    counts = {}
    for form in (m.MLA_FORM_AUTO, E, A):
        n0 = st.mla.launch_count()
        st.prefill_chunk(form)
        counts[form] = st.mla.launch_count() - n0
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    assert counts[m.MLA_FORM_AUTO] == counts[E] != counts[A]
    f32 = DeviceState(tiny_f32([0], 40))
    assert f32.mla.prefill_form(1, 40, 1) == A
