"""Run the oracle on a seeded workload (test infrastructure only).

Inputs come from ``synth`` (the seeded generator shared with the CUDA side);
every expected value here is computed by ``oracle.mla`` alone.  Hidden
states of long sequences may be generated on a CUDA device by ``synth`` (the
same seeded definition) and moved to the host: they are inputs, not results
of the library under test.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mla


def weights_f64(wl, names=("w_dkv", "w_kr", "w_uk", "w_uv", "w_o"), device="cpu") -> dict:
    return {n: wl.weight(n, device=device).to(torch.float64).cpu().numpy() for n in names}


def sequence_rows(wl, b: int, w: dict, device="cpu", chunk: int = 8192) -> np.ndarray:
    """Oracle cache rows of sequence b for positions 0..seq_len-1, float64."""
    S = wl.seq_lens[b]
    out = np.empty((S, wl.dims.row_width))
    for p0 in range(0, S, chunk):
        p1 = min(S, p0 + chunk)
        h = wl.h_rows(b, p0, p1, device=device).to(torch.float64).cpu().numpy()
        out[p0:p1] = mla.latent_rows(h, w["w_dkv"], w["w_kr"], np.arange(p0, p1),
                                     wl.dims.rope_base)
    return out


def expected_u(wl, b: int, w: dict, rows: np.ndarray, q_all: np.ndarray,
               form: str = "absorbed") -> dict:
    """Oracle decode of sequence b's T query tokens."""
    fn = mla.decode_explicit if form == "explicit" else mla.decode_absorbed
    return fn(wl.dims, rows, q_all[b], w, wl.T)
