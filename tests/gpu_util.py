"""Helpers for the GPU parity tests: device copies of seeded inputs and a
small per-layer harness around the C ABI (argument marshalling only)."""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_14_gb300 as gdn
from gated_deltanet_linear_14_gb300.pages import PagePool, SlotPool
import synth


def to_dev(t, dtype=None):
    """A synth.Tensor (bf16 bits or fp32) or a numpy array, on the GPU."""
    if isinstance(t, synth.Tensor):
        if t.dtype == synth.BF16:
            return torch.from_numpy(np.ascontiguousarray(t.store).view(np.int16)).cuda().view(
                torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(t.store)).cuda()
    a = np.ascontiguousarray(t if dtype is None else np.asarray(t, dtype))
    return torch.from_numpy(a).cuda()


def io_code(dt: str) -> int:
    return gdn.GDN_BF16 if dt == synth.BF16 else gdn.GDN_F32


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a device tensor (for bitwise comparisons)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


class Layer:
    """One GDN layer's dims, parameters, page pool and status word."""

    def __init__(self, sh: synth.Shapes, io: str, A_log, dt_bias, conv_w, Kc=0,
                 state=gdn.GDN_F32, out=gdn.GDN_F32, num_pages=1, gate_mode=0, eps=1e-6,
                 slots=False):
        self.sh = sh
        self.io = io
        self.dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, Kc, io_code(io), state, out)
        self.A_log = to_dev(A_log, np.float32)
        self.dt_bias = to_dev(dt_bias, np.float32)
        self.params = gdn.make_params(self.A_log, self.dt_bias, norm_eps=eps, gate_mode=gate_mode)
        self.conv_w = to_dev(conv_w)
        self.pool = PagePool(self.dims, num_pages)
        self.slots = SlotPool(self.dims, num_pages) if slots else None
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    @property
    def out_dtype(self):
        return torch.float32 if self.dims.out_dtype == gdn.GDN_F32 else torch.bfloat16

    @property
    def io_dtype(self):
        return torch.bfloat16 if self.io == synth.BF16 else torch.float32

    def batch(self, row_start, row_len, page=None, flags=0, n_accepted=None, order=None,
              num_rows=None, max_rows=None):
        row_start = np.asarray(row_start, np.int32)
        row_len = np.asarray(row_len, np.int32)
        R = row_start.shape[0]
        page = np.arange(R, dtype=np.int32) if page is None else np.asarray(page, np.int32)
        flags = np.broadcast_to(np.asarray(flags, np.int64), (R,)).astype(np.uint32).view(np.int32)
        arrs = [to_dev(row_start), to_dev(row_len), to_dev(page), to_dev(flags)]
        acc = None if n_accepted is None else to_dev(np.asarray(n_accepted, np.int32))
        ordr = None if order is None else to_dev(np.asarray(order, np.int32))
        end = int((row_start + row_len).max(initial=0))
        num_rows = end if num_rows is None else max(int(num_rows), end)
        max_rows = int(row_len.max(initial=0)) if max_rows is None else max_rows
        B = gdn.make_batch(R, num_rows, max_rows, self.pool.num_pages, *arrs, acc, ordr)
        B._keep = arrs + [acc, ordr]  # the struct owns the device arrays it points to
        return B

    def out(self, T):
        return torch.zeros(T, self.sh.Hv, self.sh.Dv, dtype=self.out_dtype, device="cuda")

    def conv(self, batch, x, y_dtype=None):
        T = batch.num_rows
        yd = self.dims.io_dtype if y_dtype is None else y_dtype
        y = torch.zeros(T, self.sh.C, device="cuda",
                        dtype=torch.float32 if yd == gdn.GDN_F32 else torch.bfloat16)
        gdn.gdn_conv(self.dims, batch, self.params, x, self.conv_w, y, yd, self.pool.buf,
                     self.status)
        return y

    def seq(self, batch, qkv, a, b):
        o = self.out(batch.num_rows)
        gdn.gdn_seq(self.dims, batch, self.params, qkv, a, b, o, self.pool.buf, self.status)
        return o

    def prefill(self, batch, qkv, a, b, chunk_min_rows=0):
        o = self.out(batch.num_rows)
        gdn.gdn_prefill(self.dims, batch, self.params, qkv, a, b, o, self.pool.buf, self.status,
                        chunk_min_rows)
        return o

    def verify(self, batch, qkv, a, b):
        o = self.out(batch.num_rows)
        gdn.gdn_spec_verify(self.dims, batch, self.params, qkv, a, b, o, self.pool.buf,
                            self.status)
        return o

    def spec_slots(self, batch, x, a, b):
        T = batch.num_rows
        y = torch.zeros(T, self.sh.C, dtype=self.io_dtype, device="cuda")
        o = self.out(T)
        gdn.gdn_spec_slots(self.dims, batch, self.params, x, self.conv_w, y, a, b, o,
                           self.slots.buf, self.status)
        return y, o

    def status_code(self) -> int:
        return int(self.status.item())

    def ok(self):
        code = self.status_code()
        assert code == 0, f"device status {gdn.STATUS.get(code, code)}"

    def reset_status(self):
        self.status.zero_()

    def seed(self, pages, S0=None, hist=None):
        """Seed states (math layout [R][Hv][Dk][Dv]) and windows [R][W-1][C]."""
        for i, p in enumerate(pages):
            if S0 is not None:
                self.pool.set_state_math(p, torch.from_numpy(np.asarray(S0[i], np.float32)))
            if hist is not None:
                self.pool.window(p)[: self.sh.W - 1].copy_(hist[i])
