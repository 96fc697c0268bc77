"""The fixed data layouts shared by the bf16 kernels (csrc/layouts.cuh).

The query image and the split results are written by one kernel and read
by another with different thread mappings, each through qimg_off or
part_off.  A small host program built from the header prints every offset;
the test checks what both sides rely on: each map is a bijection onto its
buffer, the units that one thread moves (16 bytes = 8 features of q~, the
32-byte sector of 16 features, 32 bytes = 8 fp32 columns of a split result,
the swizzled 16-byte chunks of the RoPE block) are contiguous and aligned,
and a warp's 32 heads are contiguous for one chunk.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

CSRC = os.path.join(os.path.dirname(__file__), "..", "mla_latent_kv_82_b300", "csrc")
HEADS, LAT, ROW = 128, 512, 576
QIMG_BYTES = 9 * 128 * 128

PROGRAM = r"""
#define __host__
#define __device__
#define __forceinline__ inline
#include "layouts.cuh"
#include <cstdio>
int main() {
  using namespace mla;
  for (int h = 0; h < kHeads; ++h)
    for (int f = 0; f < kRow; ++f) printf("%u\n", qimg_off(h, f));
  for (int h = 0; h < kHeads; ++h)
    for (int c = 0; c < kLat; ++c) printf("%zu\n", part_off(3, h, c));
  return 0;
}
"""


@pytest.fixture(scope="module")
def offsets(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("needs g++")
    d = tmp_path_factory.mktemp("layouts")
    src, exe = d / "offsets.cpp", d / "offsets"
    src.write_text(PROGRAM)
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    vals = np.array([int(x) for x in out], dtype=np.int64)
    q = vals[:HEADS * ROW].reshape(HEADS, ROW)
    p = vals[HEADS * ROW:].reshape(HEADS, LAT)
    return q, p


def test_query_image_is_a_bijection(offsets):
    q, _ = offsets
    assert q.min() == 0 and q.max() == QIMG_BYTES - 2
    assert np.all(q % 2 == 0)
    assert len(np.unique(q)) == HEADS * ROW   # every bf16 slot of the image once


def test_query_image_chunks(offsets):
    q, _ = offsets
    lat = q[:, :LAT]
    # 16 features of a head are one aligned 32-byte chunk (whole L2 sectors)
    ch = lat.reshape(HEADS, LAT // 16, 16)
    assert np.all(np.diff(ch, axis=2) == 2)
    assert np.all(ch[:, :, 0] % 32 == 0)
    # for one chunk, heads follow each other: a warp's 32 heads read 1 KB
    assert np.all(np.diff(ch[:, :, 0], axis=0) == 32)
    # the RoPE block: 16-byte chunks of 8 features, 128 bytes per head,
    # swizzled (chunk c of head r at position c ^ (r % 8)) in its own 16 KB
    rope = q[:, LAT:] - 8 * 16384
    assert rope.min() == 0 and rope.max() < 16384
    c16 = rope.reshape(HEADS, 8, 8)
    assert np.all(np.diff(c16, axis=2) == 2)
    r = np.arange(HEADS)
    assert np.all(c16 // 128 == r[:, None, None])   # 128 bytes per head, in order
    for c in range(8):
        pos = (c16[:, c, 0] % 1024 // 16) % 8
        assert np.all(pos == (c ^ (r % 8)))


def test_split_result_is_a_bijection(offsets):
    _, p = offsets
    base = 3 * HEADS * LAT
    loc = p - base
    assert loc.min() == 0 and loc.max() == HEADS * LAT - 1
    assert len(np.unique(loc)) == HEADS * LAT


def test_split_result_chunks(offsets):
    _, p = offsets
    loc = (p - 3 * HEADS * LAT).reshape(HEADS, LAT // 8, 8)
    # 8 columns of a head are one aligned 32-byte chunk
    assert np.all(np.diff(loc, axis=2) == 1)
    assert np.all(loc[:, :, 0] % 8 == 0)
    # 16 heads of a group follow each other for one chunk (512 bytes), and a
    # group of 16 heads is one contiguous 32 KB block
    grp = loc[:, :, 0].reshape(8, 16, LAT // 8)
    assert np.all(np.diff(grp, axis=1) == 8)
    for g in range(8):
        assert grp[g].min() == g * 16 * LAT and grp[g].max() == (g + 1) * 16 * LAT - 8


def test_planted_layout_slip_is_caught(offsets):
    """An offset map with two heads swapped for one chunk still covers the
    buffer, so the chunk checks must catch it."""
    q, _ = offsets
    bad = q.copy()
    bad[[0, 1], 0:16] = bad[[1, 0], 0:16]
    ch = bad[:, :LAT].reshape(HEADS, LAT // 16, 16)
    assert not np.all(np.diff(ch[:, :, 0], axis=0) == 32)
