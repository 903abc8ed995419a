"""Typed views of state pages and slot pools (host-side marshalling only).

A page pool is one ``uint8`` CUDA tensor of ``num_pages * page_bytes`` bytes;
the byte layout comes from ``gdn_page_layout`` (see include/gdn.h). These
helpers only slice and reinterpret that memory with PyTorch so that callers
can seed or inspect pages; no part of the method's arithmetic lives here.
"""
from __future__ import annotations

import torch

from . import (GDN_BF16, Dims, gdn_page_layout, gdn_slot_layout)

_TORCH = {0: torch.float32, 1: torch.bfloat16}


def torch_dtype(code: int):
    return _TORCH[int(code)]


class PagePool:
    """``num_pages`` one-page-per-request state pages on ``device``."""

    def __init__(self, dims: Dims, num_pages: int, device="cuda", zero=True):
        self.dims = dims
        self.layout = gdn_page_layout(dims)
        self.num_pages = int(num_pages)
        alloc = torch.zeros if zero else torch.empty
        self.buf = alloc(self.num_pages * self.layout.page_bytes, dtype=torch.uint8, device=device)
        d = dims
        self.C = d.C
        io_size = 2 if d.io_dtype == GDN_BF16 else 4
        self.rec_row = ((self.C + 2 * d.num_v_heads) * io_size + 15) // 16 * 16 // io_size

    def _bytes(self, p, off, nbytes):
        base = int(p) * self.layout.page_bytes + off
        return self.buf[base: base + nbytes]

    def state(self, p):
        """[Hv][Dv][Dk] view (state dtype) of page p's state."""
        d = self.dims
        v = self._bytes(p, self.layout.state_offset, self.layout.state_bytes)
        return v.view(torch_dtype(d.state_dtype)).view(d.num_v_heads, d.head_v_dim, d.head_k_dim)

    def window(self, p):
        """[(W-1)+Kc][C] view (io dtype) of page p's conv window."""
        d = self.dims
        v = self._bytes(p, self.layout.window_offset, self.layout.window_bytes)
        return v.view(torch_dtype(d.io_dtype)).view(d.conv_width - 1 + d.max_candidates, self.C)

    def record(self, p):
        """[2][Kc][rec_row] view (io dtype) of page p's record rows."""
        d = self.dims
        n = 2 * d.max_candidates * self.rec_row * torch_dtype(d.io_dtype).itemsize
        v = self._bytes(p, self.layout.record_offset, n)
        return v.view(torch_dtype(d.io_dtype)).view(2, d.max_candidates, self.rec_row)

    def record_coefficients(self, p):
        """[2][Hv][144] fp32 view of page p's record run coefficients (per slot
        and value head: G/|k| [8], G [8], R/|k| [8][8], M [8][8])."""
        d = self.dims
        n = 2 * d.max_candidates * self.rec_row * torch_dtype(d.io_dtype).itemsize
        v = self._bytes(p, self.layout.record_offset + n, self.layout.record_bytes - n)
        return v.view(torch.float32).view(2, d.num_v_heads, 144)

    def flag(self, p):
        return self._bytes(p, self.layout.flag_offset, 4).view(torch.int32)

    def set_state_math(self, p, S):
        """Seed page p from a state in the math layout [Hv][Dk][Dv]."""
        self.state(p).copy_(torch.as_tensor(S).transpose(-1, -2).to(self.state(p).dtype))

    def state_math(self, p):
        """Page p's state as fp32 in the math layout [Hv][Dk][Dv]."""
        return self.state(p).float().transpose(-1, -2)


class SlotPool:
    """Slot-per-candidate pools: one pool of max_candidates slots per page index."""

    def __init__(self, dims: Dims, num_pages: int, device="cuda"):
        self.dims = dims
        self.layout = gdn_slot_layout(dims)
        self.num_pages = int(num_pages)
        self.buf = torch.zeros(self.num_pages * self.layout.pool_bytes, dtype=torch.uint8,
                               device=device)
        self.C = dims.C

    def _bytes(self, p, i, off, nbytes):
        base = int(p) * self.layout.pool_bytes + int(i) * self.layout.slot_bytes + off
        return self.buf[base: base + nbytes]

    def state(self, p, i):
        d = self.dims
        nbytes = d.num_v_heads * d.head_v_dim * d.head_k_dim * (2 if d.state_dtype == GDN_BF16 else 4)
        v = self._bytes(p, i, self.layout.state_offset, nbytes)
        return v.view(torch_dtype(d.state_dtype)).view(d.num_v_heads, d.head_v_dim, d.head_k_dim)

    def window(self, p, i):
        d = self.dims
        nbytes = (d.conv_width - 1) * self.C * (2 if d.io_dtype == GDN_BF16 else 4)
        v = self._bytes(p, i, self.layout.window_offset, nbytes)
        return v.view(torch_dtype(d.io_dtype)).view(d.conv_width - 1, self.C)
