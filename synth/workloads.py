"""Synthetic workload recipes: shapes, lengths, paging and tensor ids.

Nothing here computes any part of the attention method; it only says which
seeded numbers go where, so that the CUDA library and the oracle see the
same inputs.

Widths follow the DeepSeek-V2 form of Multi-head Latent Attention as the
pages give it (page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，四两拨千斤",
liang.world, 第二章:
d = 5120, n_h = 128, d_h = 128, d_c = 512, d_h^R = 64); the tiny fp32 case
uses n_h = 4, d_c = 32, d_R = 8, d_h = 16, d = 64.

Recipe (every value is seeded):
* tensor ids: h=0, W^DKV=1, W^KR=2, W^UK=3, W^UV=4, W_O=5, q=6, and for the
  query path W^DQ=7, W^UQ=8, W^QR=9; in a stack of layers, layer j's weights
  and cached hidden states use id + 16 j (layer 0 the ids above);
* h and q ~ N(0, 1); every weight ~ N(0, 1/fan_in), fan_in = input width;
* sequence b has ``lens[b]`` cached tokens before the step and ``T`` new
  tokens; h of token p of sequence b is row ``b * row_stride + p`` of a
  virtual [B * row_stride, d] tensor (row_stride = max(lens) + T);
* the step appends the T new tokens at positions lens[b] .. lens[b]+T-1
  and decodes them; query t sits at position lens[b] + t;
* pages of 64 tokens; each sequence owns ceil((lens[b]+T)/page) pages,
  taken in order from ``numpy.random.default_rng(1).permutation(num_pages)``
  when the table is shuffled, else in identity order.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from . import gen

TID_H, TID_WDKV, TID_WKR, TID_WUK, TID_WUV, TID_WO, TID_Q, TID_WDQ, TID_WUQ, TID_WQR = range(10)


@dataclasses.dataclass(frozen=True)
class Dims:
    d_model: int
    n_heads: int
    d_nope: int
    d_v: int
    d_latent: int
    d_rope: int
    page_size: int
    rope_base: float = 10000.0
    d_cq: int = 0          # width of the query latent c^Q (query path); not on the pages

    @property
    def row_width(self) -> int:
        return self.d_latent + self.d_rope

    @property
    def softmax_scale(self) -> float:
        # The pages give no scale; 1/sqrt(d_nope + d_rope) is the stated
        # assumption (1/sqrt(192) at V2 widths).
        return 1.0 / math.sqrt(self.d_nope + self.d_rope)


V2 = Dims(d_model=5120, n_heads=128, d_nope=128, d_v=128, d_latent=512,
          d_rope=64, page_size=64, d_cq=1536)
TINY = Dims(d_model=64, n_heads=4, d_nope=16, d_v=16, d_latent=32,
            d_rope=8, page_size=64, d_cq=48)


@dataclasses.dataclass
class Workload:
    name: str
    dims: Dims
    dtype: str            # "bf16" or "f32"
    lens: list            # cached tokens per sequence before the step
    T: int                # new (query) tokens per sequence
    shuffle_pages: bool
    seed: int = 0
    layers: int = 1       # attention layers of a multi-layer step

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def seq_lens(self) -> list:
        return [L + self.T for L in self.lens]

    @property
    def row_stride(self) -> int:
        return max(self.lens) + self.T

    @property
    def pages_per_seq(self) -> list:
        P = self.dims.page_size
        return [(s + P - 1) // P for s in self.seq_lens]

    @property
    def max_pages(self) -> int:
        return max(self.pages_per_seq)

    @property
    def num_pages(self) -> int:
        return sum(self.pages_per_seq)

    def block_table(self) -> np.ndarray:
        """int32 [B, max_pages]; unused entries are -1."""
        ids = np.arange(self.num_pages, dtype=np.int64)
        if self.shuffle_pages:
            ids = np.random.default_rng(1).permutation(self.num_pages)
        bt = np.full((self.B, self.max_pages), -1, dtype=np.int32)
        k = 0
        for b, n in enumerate(self.pages_per_seq):
            bt[b, :n] = ids[k:k + n]
            k += n
        return bt

    # ---- seeded tensors -------------------------------------------------
    def weight(self, name: str, device="cpu", layer: int = 0) -> torch.Tensor:
        d = self.dims
        spec = {
            "w_dkv": (TID_WDKV, (d.d_latent, d.d_model), d.d_model),
            "w_kr": (TID_WKR, (d.d_rope, d.d_model), d.d_model),
            "w_uk": (TID_WUK, (d.n_heads * d.d_nope, d.d_latent), d.d_latent),
            "w_uv": (TID_WUV, (d.n_heads * d.d_v, d.d_latent), d.d_latent),
            "w_o": (TID_WO, (d.d_model, d.n_heads * d.d_v), d.n_heads * d.d_v),
            "w_dq": (TID_WDQ, (d.d_cq, d.d_model), d.d_model),
            "w_uq": (TID_WUQ, (d.n_heads * d.d_nope, d.d_cq), d.d_cq),
            "w_qr": (TID_WQR, (d.n_heads * d.d_rope, d.d_model), d.d_model),
        }[name]
        tid, shape, fan_in = spec
        return gen.fill(self.seed, tid + 16 * layer, shape, 1.0 / math.sqrt(fan_in),
                        self.torch_dtype, device=device)

    def h_rows(self, b: int, p0: int, p1: int, device="cpu", layer: int = 0) -> torch.Tensor:
        """Hidden states of tokens p0..p1-1 of sequence b, [p1-p0, d] (layer j's
        cached positions use their own seeded states; the new tokens' states of
        layer j > 0 come from the layers below)."""
        d = self.dims.d_model
        start = (b * self.row_stride + p0) * d
        return gen.fill(self.seed, TID_H + 16 * layer, (p1 - p0, d), 1.0, self.torch_dtype,
                        device=device, start=start)

    def q(self, device="cpu") -> torch.Tensor:
        """Queries [B, T, n_h, d_nope + d_rope] (rope part not rotated)."""
        d = self.dims
        return gen.fill(self.seed, TID_Q,
                        (self.B, self.T, d.n_heads, d.d_nope + d.d_rope), 1.0,
                        self.torch_dtype, device=device)


def paged_lens() -> list:
    return [int(x) for x in np.random.default_rng(0).integers(1024, 8193, 64)]


def config(name: str) -> Workload:
    """The five named workloads, by the short keys used in tests and bench."""
    if name == "tiny-fp32":   # tiny fp32 oracle check: 64 cached rows in total
        return Workload("tiny-fp32-L64", TINY, "f32", [63], 1, False)
    if name == "b1-l4096":   # batch 1, contiguous cache of 4096 tokens
        return Workload("v2-b1-L4096-contig", V2, "bf16", [4095], 1, False)
    if name == "b64-paged":   # batch 64, lengths U[1024, 8192], shuffled pages
        return Workload("v2-b64-paged-Lrand", V2, "bf16", paged_lens(), 1, True)
    if name == "b4-l128k":   # batch 4, 128K cached tokens each
        return Workload("v2-b4-L131072", V2, "bf16", [131071] * 4, 1, False)
    if name == "b128-l16k-t2":   # batch 128, L=16384, two query tokens, full step
        return Workload("v2-b128-L16384-T2", V2, "bf16", [16384] * 128, 2, False)
    if name == "b1-l4096-x60":   # the batch-1 step through 60 layers
        return Workload("v2-b1-L4096-x60layers", V2, "bf16", [4095], 1, False, layers=60)
    if name == "b64-paged-x8":   # the batch-64 paged step through 8 layers
        return Workload("v2-b64-paged-Lrand-x8layers", V2, "bf16", paged_lens(), 1, True,
                        layers=8)
    if name == "prefill-b4-t4096":   # four 4096-token prompts, one chunk each
        return Workload("v2-prefill-b4-T4096", V2, "bf16", [0] * 4, 4096, False)
    if name == "chunk-b1-l12k-t4096":   # the last 4096-token chunk of a 16K prompt
        return Workload("v2-chunk-b1-L12288-T4096", V2, "bf16", [12288], 4096, False)
    if name == "prefill-b64-t128":   # 64 short prompts of 128 tokens, shuffled pages
        return Workload("v2-prefill-b64-T128", V2, "bf16", [0] * 64, 128, True)
    raise KeyError(name)


CONFIG_NAMES = ("tiny-fp32", "b1-l4096", "b64-paged", "b4-l128k", "b128-l16k-t2",
                "b1-l4096-x60", "b64-paged-x8")
PREFILL_NAMES = ("prefill-b4-t4096", "chunk-b1-l12k-t4096", "prefill-b64-t128")
