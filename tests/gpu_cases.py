"""Shared helpers of the GPU parity tests: workloads, oracle runs, checks."""
import dataclasses

import numpy as np
import torch

from oracle import case as ocase
from oracle import mla as omla
from synth import workloads as W

# bf16 tolerance (on u, and as a diagnostic on the cache rows, o_lat and o):
# max|err| <= 2e-2 * max|ref| and sum|err| / sum|ref| <= 5e-3.  fp32: 1e-4 both.
TOL = {"bf16": (2e-2, 5e-3), "f32": (1e-4, 1e-4)}

SMALL_V2 = dataclasses.replace(W.V2, d_model=512)


def small_bf16(lens, T, shuffle=True):
    """V2 head widths on a narrow model: several 64-token tiles, ragged tails."""
    return W.Workload(f"v2-small-T{T}", SMALL_V2, "bf16", list(lens), T, shuffle)


def tiny_f32(lens, T, page=16, shuffle=True):
    return W.Workload(f"tiny-f32-T{T}", dataclasses.replace(W.TINY, page_size=page), "f32",
                      list(lens), T, shuffle)


def check(got, ref, dtype, what):
    s = omla.error_stats(got, ref)
    mx, mean = TOL[dtype]
    assert s["max_rel"] <= mx and s["mean_rel"] <= mean, f"{what}: {s}"
    return s


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().to(torch.float64).cpu().numpy()


def oracle_sequence(wl, b, w64, q64, form, device):
    """Oracle rows and decode of sequence b (hidden states generated on `device`)."""
    rows = ocase.sequence_rows(wl, b, w64, device=device)
    res = ocase.expected_u(wl, b, w64, rows, q64, form=form)
    return rows, res


def pool_rows_of(state, b):
    """The GPU pool's rows of sequence b, positions 0..seq_len-1, in order."""
    wl = state.wl
    P = wl.dims.page_size
    S = wl.seq_lens[b]
    pos = torch.arange(S, device=state.dev)
    slots = state.bt[b, pos // P].long() * P + pos % P
    return state.cache[slots]
