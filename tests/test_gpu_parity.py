"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small cases span several 64-token tiles with ragged tails, single-slot
sequences and T=2 with the causal mask across a page boundary; the five
named workloads run at full size with every sequence (tiny-fp32, b1-l4096)
or a seeded sample of sequences (b64-paged, b128-l16k-t2, b4-l128k) compared
with the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import case as ocase
from synth import workloads as W

from gpu_cases import TOL, check, oracle_sequence, pool_rows_of, small_bf16, tiny_f32, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mla_latent_kv_82_b300  # noqa: F401  (raises if libmla.so is missing)


def _run(wl, sentinel=None, block_table=None):
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl, sentinel=sentinel, block_table=block_table)
    st.step()
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    return st


def _compare_all(st, form="explicit", seqs=None, keep_rows=None):
    wl = st.wl
    w64 = ocase.weights_f64(wl, device=DEV)
    q64 = to_np(st.q)
    o_lat = st.workspace_view("o_lat")
    o = st.workspace_view("o")
    stats = []
    for b in (range(wl.B) if seqs is None else seqs):
        rows, res = oracle_sequence(wl, b, w64, q64, form, DEV)
        if keep_rows is not None:
            keep_rows[b] = rows
        check(to_np(pool_rows_of(st, b)), rows, wl.dtype, f"cache rows b={b}")
        stats.append(check(to_np(st.out[b]), res["u"], wl.dtype, f"u b={b}"))
        m = slice(b * wl.T, (b + 1) * wl.T)
        check(to_np(o[m]), res["o"].reshape(wl.T, -1), wl.dtype, f"o b={b}")
        if form == "absorbed":
            check(to_np(o_lat[m]), res["o_lat"], wl.dtype, f"o_lat b={b}")
    return stats


# --------------------------------------------------------------------------- small
@pytest.mark.parametrize("T,lens", [
    (1, [0, 62, 63, 64, 200, 1000]),
    (2, [0, 62, 63, 127, 500]),
    (1, [300]),          # one token: the projections run as GEMVs
    (2, [200]),          # two tokens: GEMVs, and the paired attention
    (1, [70, 1]),        # two tokens from two sequences
    (3, [2, 64, 190]),   # odd T > 1: single-CTA kernel, three tokens per split
    (4, [3, 130, 260]),  # T = 4: two CTA pairs per split
    (5, [0, 70, 200]),   # odd T: five single-token clusters per split
    (6, [1, 64]),
    (7, [62, 129]),
    (8, [0, 63, 300]),   # the largest decode T: four token pairs per split
])
def test_small_bf16_explicit(T, lens):
    st = _run(small_bf16(lens, T))
    _compare_all(st, "explicit")


@pytest.mark.parametrize("T", [1, 2, 3])
def test_widest_model(T):
    """d_model = 16384, the widest model the bf16 path takes (W_O 512 MB):
    for one or two tokens the CUDA-core append kernel cannot hold its share
    of [W^DKV; W^KR] rows in shared memory at this width, so the append and
    absorbed query run on the tensor-core GEMM instead; W_O streams 32 KB
    rows."""
    wl = W.Workload(f"v2-d16384-T{T}", dataclasses.replace(W.V2, d_model=16384), "bf16",
                    [3, 70], T, True)
    _compare_all(_run(wl), "explicit")


def test_small_bf16_latent_output():
    st = _run(small_bf16([5, 300, 129], 1))
    _compare_all(st, "absorbed")


@pytest.mark.parametrize("T,lens,page", [
    (1, [63], 64), (1, [0, 15, 16, 17, 100], 16), (2, [0, 14, 15, 33], 16), (1, [40, 3], 1),
    (3, [0, 20, 47], 16), (8, [0, 9, 40], 16)])
def test_tiny_f32(T, lens, page):
    st = _run(tiny_f32(lens, T, page))
    _compare_all(st, "explicit")


def test_tiny_fp32_workload():
    st = _run(W.config("tiny-fp32"))
    s = _compare_all(st, "explicit")
    assert s[0]["max_rel"] <= TOL["f32"][0]


# --------------------------------------------------------------------------- exact
def test_append_placement_is_exact_and_untouched_rows_keep_sentinel():
    wl = small_bf16([3, 64, 130], 2)
    sentinel = -1234.0
    st = _run(wl, sentinel=sentinel)
    P = wl.dims.page_size
    written = torch.zeros(st.cache.shape[0], dtype=torch.bool, device=st.dev)
    for b, S in enumerate(wl.seq_lens):
        pos = torch.arange(S, device=st.dev)
        written[st.bt[b, pos // P].long() * P + pos % P] = True
    assert int(written.sum()) == sum(wl.seq_lens)
    untouched = st.cache[~written]
    assert torch.equal(untouched, torch.full_like(untouched, sentinel))
    assert not (st.cache[written] == sentinel).all(dim=1).any()
    w64 = ocase.weights_f64(wl, device=DEV)
    for b in range(wl.B):
        rows = ocase.sequence_rows(wl, b, w64, device=DEV)
        check(to_np(pool_rows_of(st, b)), rows, "bf16", f"rows b={b}")


@pytest.mark.parametrize("T,lens", [(1, [0, 5, 33, 64, 100]), (2, [1, 31, 62, 200])])
def test_stale_pool_rows_do_not_leak(T, lens):
    """Rows of the pool that no sequence owns hold NaN: outputs stay exact."""
    st = _run(small_bf16(lens, T), sentinel=float("nan"))
    assert torch.isfinite(st.out.float()).all()
    _compare_all(st, "explicit")


def test_shuffled_block_table_is_bitwise_identical():
    wl = small_bf16([70, 200, 5, 130], 1, shuffle=True)
    a = _run(wl)
    wl_id = small_bf16([70, 200, 5, 130], 1, shuffle=False)
    b = _run(wl_id)
    assert torch.equal(a.out, b.out)


def test_repeated_decode_is_deterministic():
    st = _run(small_bf16([300, 40], 2))
    first = st.out.clone()
    st.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, st.out)


# --------------------------------------------------------------------------- errors
def test_bad_page_id_is_reported_not_written():
    wl = small_bf16([10], 1)
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl, sentinel=7.0)
    bad = st.bt.clone()
    bad[0, 0] = st.num_pages + 5           # out of range: must be skipped and reported
    before = st.cache.clone()
    st.mla.compress_append(st.h_new, st.pos_new, bad, st.cache, 1, 1)
    assert st.mla.check_status() == 6      # MLA_ERR_DEVICE_INDEX
    assert torch.equal(before, st.cache)
    assert st.mla.check_status() == 0      # the status word was cleared


@pytest.mark.parametrize("lens,T", [([10], 1), ([10], 2), ([10, 70], 1), ([10, 20, 30], 1)])
def test_bad_position_is_reported_not_written(lens, T):
    """A new token whose position lies beyond max_position is reported and
    its row is written nowhere; the other new tokens' rows are written (one
    or two tokens run the CUDA-core projection kernel, three the GEMM)."""
    wl = small_bf16(lens, T)
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl, sentinel=7.0)
    before = st.cache.clone()
    pos = st.pos_new.clone()
    pos[0] = 10 ** 6
    st.mla.compress_append(st.h_new, pos, st.bt, st.cache, wl.B, wl.T)
    assert st.mla.check_status() == 6      # MLA_ERR_DEVICE_INDEX
    P = wl.dims.page_size
    changed = (st.cache != before).any(dim=1).nonzero().flatten().tolist()
    allowed = set()
    for m in range(1, wl.B * wl.T):
        p_m = int(pos[m])
        allowed.add(int(st.bt[m // wl.T, p_m // P]) * P + p_m % P)
    assert set(changed) <= allowed and len(changed) == len(allowed)
    assert st.mla.check_status() == 0


@pytest.mark.parametrize("make", [
    lambda: tiny_f32([5, 40, 64], 1),
    lambda: small_bf16([0, 63, 200, 1000], 1),
    lambda: small_bf16([62, 127, 500], 2),
    lambda: small_bf16([200], 2),       # two tokens of one sequence (CUDA-core projections)
    lambda: small_bf16([70, 1], 1),     # two sequences of one token
    lambda: W.config("b1-l4096"),
])
def test_append_decode_equals_two_calls(make):
    """mla_append_decode (one call; the append may run in the absorbed-query
    launch) gives the cache rows and outputs of mla_compress_append followed
    by mla_decode, bit for bit."""
    from mla_latent_kv_82_b300.workload import DeviceState
    wl = make()
    one = DeviceState(wl, sentinel=0.0)
    two = DeviceState(wl, sentinel=0.0)
    one.step()
    two.step_separate()
    torch.cuda.synchronize()
    assert one.mla.check_status() == 0 and two.mla.check_status() == 0
    assert torch.equal(one.cache.view(torch.uint8), two.cache.view(torch.uint8))
    assert torch.equal(one.out.view(torch.uint8), two.out.view(torch.uint8))


def test_bad_length_is_reported():
    wl = small_bf16([10], 1)
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl)
    st.append_new()
    st.seq_lens.fill_(10 ** 6)             # beyond max_pages * page_size
    st.decode()
    assert st.mla.check_status() == 6


@pytest.mark.parametrize("call", ["decode", "append_decode"])
def test_more_than_eight_query_tokens_are_refused(call):
    """T = 9 is refused before anything is enqueued; the output keeps its bytes."""
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(small_bf16([10], 1), prefill=False)
    d, T = st.wl.dims, 9
    q = torch.zeros((1, T, d.n_heads, d.d_nope + d.d_rope), dtype=torch.bfloat16, device=st.dev)
    h = torch.zeros((1, T, d.d_model), dtype=torch.bfloat16, device=st.dev)
    pos = torch.arange(T, dtype=torch.int32, device=st.dev)
    seq_lens = torch.full((1,), T, dtype=torch.int32, device=st.dev)
    out = torch.zeros((1, T, d.d_model), dtype=torch.bfloat16, device=st.dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=st.dev)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    before = st.mla.launch_count()
    common = (st.cache.data_ptr(), st.num_pages, st.bt.data_ptr(), st.bt.shape[1],
              seq_lens.data_ptr(), 1, T, out.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    if call == "decode":
        rc = m.mla_decode(st.mla.ctx, q.data_ptr(), *common)
    else:
        rc = m.mla_append_decode(st.mla.ctx, h.data_ptr(), pos.data_ptr(), q.data_ptr(), *common)
    assert rc == m.MLA_ERR_INVALID_ARG
    assert st.mla.launch_count() == before
    torch.cuda.synchronize()
    assert st.mla.check_status() == 0
    assert not out.any()


def test_bounded_wait_gives_up_with_status():
    wl = small_bf16([10], 1)
    from mla_latent_kv_82_b300.workload import DeviceState
    st = DeviceState(wl, prefill=False)
    import mla_latent_kv_82_b300 as m
    assert m.mla_selftest_bounded_wait(st.mla.ctx, 1000,
                                       torch.cuda.current_stream().cuda_stream) == 0
    assert st.mla.check_status() == m.MLA_ERR_TIMEOUT
    # the context is still usable afterwards
    st.step()
    assert st.mla.check_status() == 0


# --------------------------------------------------------------------------- full size
def test_b1_l4096_full():
    st = _run(W.config("b1-l4096"))
    _compare_all(st, "explicit")


FULL_SAMPLES = {
    # seeded samples of sequences (all four of b4-l128k)
    "b64-paged": [0, 7, 21, 33, 40, 52, 58, 63],
    "b128-l16k-t2": [0, 17, 38, 64, 77, 99, 111, 127],
    "b4-l128k": [0, 1, 2, 3],
}


def _explicit_heads(wl, rows, q_b, w64, heads):
    """The explicit (non-absorbed) oracle on single heads: K^C and V of each
    head materialised from the rows, its o returned per head."""
    import dataclasses
    from oracle import mla as omla
    d = wl.dims
    one = dataclasses.replace(d, n_heads=1)
    out = {}
    for h in heads:
        w = {"w_uk": w64["w_uk"][h * d.d_nope:(h + 1) * d.d_nope],
             "w_uv": w64["w_uv"][h * d.d_v:(h + 1) * d.d_v],
             "w_o": w64["w_o"][:, h * d.d_v:(h + 1) * d.d_v]}
        out[h] = omla.decode_explicit(one, rows, q_b[:, h:h + 1], w, wl.T)["o"][:, 0]
    return out


@pytest.mark.parametrize("name", list(FULL_SAMPLES))
def test_full_configs_sampled(name):
    """Full-size workloads in the launch configuration the benchmark times:
    sampled sequences against the absorbed oracle (u, o, o_lat, cache rows)
    and, on two heads of each, the value output o against the explicit form."""
    wl = W.config(name)
    seqs = FULL_SAMPLES[name]
    st = _run(wl)
    rows_of = {}
    stats = _compare_all(st, "absorbed", seqs=seqs, keep_rows=rows_of)
    assert len(stats) == len(seqs)
    w64 = ocase.weights_f64(wl, device=DEV)
    q64 = to_np(st.q)
    o = st.workspace_view("o")
    rng = np.random.default_rng(2)
    d = wl.dims
    for b in seqs:
        rows = rows_of[b]
        heads = [int(x) for x in rng.choice(d.n_heads, 2, replace=False)]
        ref = _explicit_heads(wl, rows, q64[b], w64, heads)
        for h in heads:
            got = to_np(o[b * wl.T:(b + 1) * wl.T, h * d.d_v:(h + 1) * d.d_v])
            check(got, ref[h], wl.dtype, f"o explicit b={b} head={h}")
    # every sequence produced finite output
    assert torch.isfinite(st.out.float()).all()
