"""The seeded input generator against its written definition (CPU only)."""
import math

import numpy as np
import torch

from synth import gen, workloads

MASK = (1 << 64) - 1


def _mix(z):
    z &= MASK
    z = ((z ^ (z >> 30)) * gen.C1) & MASK
    z = ((z ^ (z >> 27)) * gen.C2) & MASK
    return z ^ (z >> 31)


def _ref_normal(seed, tid, i):
    key = _mix((((seed << 32) + tid + 1) * gen.GAMMA) & MASK)
    w1 = _mix(key + (2 * i + 1) * gen.GAMMA)
    w2 = _mix(key + (2 * i + 2) * gen.GAMMA)
    u1 = (w1 >> 11) * 2.0 ** -53 + 2.0 ** -54
    u2 = (w2 >> 11) * 2.0 ** -53 + 2.0 ** -54
    return math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)


def test_splitmix_reference_vector():
    # SplitMix64 seeded with state 0: the published first output
    # (state advanced by GAMMA once, then mixed) is 0xE220A8397B1DCDAF.
    assert _mix(gen.GAMMA) == 0xE220A8397B1DCDAF


def test_torch_matches_scalar_definition():
    idx = [0, 1, 2, 999, 123456, (1 << 32) + 5, (1 << 34) + 77]
    for seed, tid in [(0, 0), (0, 6), (7, 3)]:
        for i in idx:
            got = gen.normal_f64(seed, tid, i, 1)[0].item()
            assert got == _ref_normal(seed, tid, i)


def test_moments_and_independence():
    z = gen.normal_f64(0, 0, 0, 1 << 20)
    assert abs(z.mean().item()) < 5e-3 and abs(z.std().item() - 1) < 5e-3
    z2 = gen.normal_f64(0, 1, 0, 1 << 20)
    assert abs(torch.corrcoef(torch.stack([z, z2]))[0, 1].item()) < 5e-3


def test_bf16_rounding_is_rne_of_fp32():
    x = gen.fill(0, 4, (4096,), 0.05, torch.float32)
    b = gen.fill(0, 4, (4096,), 0.05, torch.bfloat16)
    bits = b.view(torch.int16).to(torch.int32) & 0xFFFF
    assert torch.equal(bits, gen.bf16_bits_from_f32(x))
    # ties go to even
    t = torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], dtype=torch.float32)
    assert gen.bf16_bits_from_f32(t).tolist() == [0x3F80, 0x3F82]


def test_fill_offsets_compose():
    a = gen.fill(0, 0, (10, 8), 1.0, torch.float32)
    b = gen.fill(0, 0, (3, 8), 1.0, torch.float32, start=5 * 8)
    assert torch.equal(a[5:8], b)
    a = gen.fill(0, 0, (1000,), 1.0, torch.float32, chunk=64)
    assert torch.equal(a, gen.fill(0, 0, (1000,), 1.0, torch.float32))


def test_workload_recipes():
    paged = workloads.config("b64-paged")
    assert (paged.B, min(paged.lens), max(paged.lens), sum(paged.lens)) == (64, 1043, 8172, 299418)
    assert paged.num_pages == 4709
    bt = paged.block_table()
    used = bt[bt >= 0]
    assert sorted(used.tolist()) == list(range(paged.num_pages))
    t2 = workloads.config("b128-l16k-t2")
    assert t2.seq_lens[0] == 16386 and t2.T == 2
    b1 = workloads.config("b1-l4096")
    assert (b1.block_table()[0] == np.arange(64)).all()
    assert workloads.config("tiny-fp32").dims.softmax_scale == 1 / math.sqrt(24)
    assert workloads.V2.softmax_scale == 1 / math.sqrt(192)
    # h rows of a sequence are slices of one virtual tensor
    h = paged.h_rows(2, 10, 12)
    assert torch.equal(h[1], paged.h_rows(2, 11, 12)[0])
