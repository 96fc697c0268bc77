"""Device state for one decode workload: weights, paged pool, prefill, step.

Builds everything a decode step needs on one GPU from a seeded
``synth.workloads.Workload`` and drives the library through ``MLA``:
weights and queries come from the seeded generator (on the device), the
pool is prefilled by chunked ``mla_compress_append`` calls, and ``step()``
is one pass of the hot path: append the T new tokens of every sequence,
then decode them.  With ``query_path`` the context also holds the query
projections and ``layer_step()`` makes the same step from the hidden states
alone (the queries come from the new tokens' hidden states).
"""
from __future__ import annotations

import dataclasses

import torch

from . import MLA

W_NAMES = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o")
Q_NAMES = ("w_dq", "w_uq", "w_qr")


class DeviceState:
    def __init__(self, wl, device: int = 0, prefill: bool = True, chunk: int = 32768,
                 sentinel: float | None = None, block_table=None, query_path: bool = False,
                 kv: str = "native"):
        self.wl = wl
        self.dev = torch.device("cuda", device)
        d = wl.dims
        dt = wl.torch_dtype
        names = W_NAMES + (Q_NAMES if query_path else ())
        self.weights = {n: wl.weight(n, device=self.dev) for n in names}
        ctx_dims = d if query_path else dataclasses.replace(d, d_cq=0)
        self.kv = kv
        self.mla = MLA(ctx_dims, self.weights, wl.dtype, max_position=max(wl.seq_lens),
                       device=device, kv=kv)
        bt = wl.block_table() if block_table is None else block_table
        self.bt = torch.as_tensor(bt, dtype=torch.int32, device=self.dev).contiguous()
        self.num_pages = int(self.bt.max().item()) + 1
        rows = self.num_pages * d.page_size
        if kv == "fp8":
            # FP8 rows of MLA_FP8_ROW_BYTES bytes; the sentinel is a byte value
            self.cache = torch.full((rows, 656), 0 if sentinel is None else int(sentinel),
                                    dtype=torch.uint8, device=self.dev)
        elif sentinel is None:
            self.cache = torch.empty((rows, d.row_width), dtype=dt, device=self.dev)
        else:
            self.cache = torch.full((rows, d.row_width), sentinel, dtype=dt, device=self.dev)
        T = wl.T
        seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=self.dev)
        q = wl.q(device=self.dev).contiguous()
        h_new = torch.cat([wl.h_rows(b, L, L + T, device=self.dev)
                           for b, L in enumerate(wl.lens)]).contiguous()
        pos_new = torch.tensor([L + t for L in wl.lens for t in range(T)],
                               dtype=torch.int32, device=self.dev)
        # The step's inputs live in one buffer (256-byte aligned parts), so
        # that a caller can bring a step's inputs over in one copy.
        parts = [h_new, q, pos_new, seq_lens]
        offs, off = [], 0
        for x in parts:
            offs.append(off)
            off = (off + x.numel() * x.element_size() + 255) // 256 * 256
        self.step_inputs = torch.empty(off, dtype=torch.uint8, device=self.dev)
        views = []
        for x, o in zip(parts, offs):
            nb = x.numel() * x.element_size()
            v = self.step_inputs[o:o + nb].view(x.dtype).view(x.shape)
            v.copy_(x)
            views.append(v)
        self.h_new, self.q, self.pos_new, self.seq_lens = views
        self.out = torch.empty((wl.B, T, d.d_model), dtype=dt, device=self.dev)
        self.ws_bytes = self.mla.workspace_size(wl.B, T, self.bt.shape[1])
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
        self.chunk = chunk
        if prefill:
            self.prefill()

    def prefill(self):
        """Append cached tokens 0..lens[b]-1 of every sequence, in chunks."""
        for b, L in enumerate(self.wl.lens):
            for p0 in range(0, L, self.chunk):
                p1 = min(L, p0 + self.chunk)
                h = self.wl.h_rows(b, p0, p1, device=self.dev)
                pos = torch.arange(p0, p1, dtype=torch.int32, device=self.dev)
                self.mla.compress_append(h, pos, self.bt[b:b + 1], self.cache, 1, p1 - p0)

    def append_new(self, stream=None):
        self.mla.compress_append(self.h_new, self.pos_new, self.bt, self.cache, self.wl.B,
                                 self.wl.T, stream=stream)

    def decode(self, stream=None):
        self.mla.decode(self.q, self.cache, self.bt, self.seq_lens, self.out, self.ws,
                        stream=stream)

    def step(self, stream=None):
        """Append the T new tokens of every sequence, then decode them (one
        mla_append_decode call)."""
        self.mla.append_decode(self.h_new, self.pos_new, self.q, self.cache, self.bt,
                               self.seq_lens, self.out, self.ws, stream=stream)

    def layer_step(self, stream=None):
        """The step from the hidden states alone (mla_layer_step): the query
        path makes the queries of the new tokens, then append and decode."""
        self.mla.layer_step(self.h_new, self.pos_new, self.cache, self.bt, self.seq_lens,
                            self.out, self.ws, stream=stream)

    def prefill_chunk(self, form: int = 0, stream=None):
        """The T new tokens of every sequence as one prefill chunk
        (mla_prefill): appended, then attended to with the causal mask, in
        `form` (MLA_FORM_AUTO, _EXPLICIT or _ABSORBED)."""
        need = self.mla.prefill_workspace_size(self.wl.B, self.wl.T, self.bt.shape[1])
        if need > self.ws_bytes:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.dev)
            self.ws_bytes = need
        self.mla.prefill(self.h_new, self.pos_new, self.q, self.cache, self.bt, self.seq_lens,
                         self.out, self.ws, form=form, stream=stream)

    def step_separate(self, stream=None):
        """The same step as two calls: mla_compress_append, then mla_decode."""
        self.append_new(stream)
        self.decode(stream)

    def workspace_view(self, which: str) -> torch.Tensor:
        """o_lat [B*T, n_h, d_c] or o [B*T, n_h*d_v] left in the workspace by decode."""
        from . import mla_decode_workspace_offsets
        d, B, T = self.wl.dims, self.wl.B, self.wl.T
        st, off_lat, off_o = mla_decode_workspace_offsets(self.mla.ctx, B, T, self.bt.shape[1])
        assert st == 0
        es = 2 if self.wl.dtype == "bf16" else 4
        if which == "o_lat":
            n, off, shape = B * T * d.n_heads * d.d_latent, off_lat, (B * T, d.n_heads, d.d_latent)
        else:
            n, off, shape = B * T * d.n_heads * d.d_v, off_o, (B * T, d.n_heads * d.d_v)
        return self.ws[off:off + n * es].view(self.wl.torch_dtype).view(*shape)


class StackState:
    """A stack of wl.layers attention layers on one GPU: per-layer contexts
    (with the query path), weights and cache pools sharing one block table,
    each pool prefilled from that layer's own seeded hidden states.
    ``step()`` runs mla_multi_layer_step on the new tokens' layer-0 hidden
    states (copied into ``h`` first, so every step repeats the same work)."""

    def __init__(self, wl, device: int = 0, chunk: int = 32768, kv: str = "native"):
        from . import MLA
        self.wl = wl
        self.kv = kv
        self.dev = torch.device("cuda", device)
        d, dt, T = wl.dims, wl.torch_dtype, wl.T
        bt = wl.block_table()
        self.bt = torch.as_tensor(bt, dtype=torch.int32, device=self.dev).contiguous()
        self.num_pages = int(self.bt.max().item()) + 1
        rows = self.num_pages * d.page_size
        self.weights, self.mlas, self.caches = [], [], []
        for j in range(wl.layers):
            w = {n: wl.weight(n, device=self.dev, layer=j) for n in W_NAMES + Q_NAMES}
            self.weights.append(w)
            self.mlas.append(MLA(d, w, wl.dtype, max_position=max(wl.seq_lens), device=device,
                                 kv=kv))
            self.caches.append(torch.empty((rows, 656), dtype=torch.uint8, device=self.dev)
                               if kv == "fp8" else
                               torch.empty((rows, d.row_width), dtype=dt, device=self.dev))
        self.seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=self.dev)
        self.pos_new = torch.tensor([L + t for L in wl.lens for t in range(T)],
                                    dtype=torch.int32, device=self.dev)
        self.h0 = torch.cat([wl.h_rows(b, L, L + T, device=self.dev)
                             for b, L in enumerate(wl.lens)]).contiguous()
        self.h = torch.empty_like(self.h0)
        self.u = torch.empty_like(self.h0)
        self.ws_bytes = self.mlas[0].workspace_size(wl.B, T, self.bt.shape[1])
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
        for j in range(wl.layers):
            for b, L in enumerate(wl.lens):
                for p0 in range(0, L, chunk):
                    p1 = min(L, p0 + chunk)
                    h = wl.h_rows(b, p0, p1, device=self.dev, layer=j)
                    pos = torch.arange(p0, p1, dtype=torch.int32, device=self.dev)
                    self.mlas[j].compress_append(h, pos, self.bt[b:b + 1], self.caches[j], 1,
                                                 p1 - p0)

    def step(self, stream=None):
        from . import MLAError, mla_multi_layer_step
        s = stream if stream is not None else torch.cuda.current_stream()
        self.h.copy_(self.h0)
        st = mla_multi_layer_step([m.ctx for m in self.mlas], self.h.data_ptr(),
                                  self.pos_new.data_ptr(), [c.data_ptr() for c in self.caches],
                                  self.num_pages, self.bt.data_ptr(), self.bt.shape[1],
                                  self.seq_lens.data_ptr(), self.wl.B, self.wl.T,
                                  self.u.data_ptr(), self.ws.data_ptr(), self.ws_bytes,
                                  s.cuda_stream)
        if st != 0:
            raise MLAError(st, "mla_multi_layer_step")

    def check_status(self) -> int:
        for m in self.mlas:
            r = m.check_status()
            if r:
                return r
        return 0
