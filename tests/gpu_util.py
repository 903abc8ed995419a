"""Helpers for the GPU parity tests: device copies of seeded inputs and a
small per-layer harness around the C ABI (argument marshalling only)."""
from __future__ import annotations

import json
import os

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


# Element-wise parity constant: every element lies within ELEM_C * tol of the
# RMS of its slice of the reference (one value head of one output row, or one
# head's state). c = 1 holds each (row, head) to the same 1e-4 as the tensor,
# so an error confined to a few heads or columns, which a tensor-wide norm
# averages away, fails. The fp32 paths (token by token, the closed-form
# verify, the fused decode) keep every element within about 1e-5 of it.
ELEM_C = 1.0
# The chunked prefill feeds fp32 operands to the bf16 tensor cores as hi + lo
# pairs, 16 significant bits (2^-17 relative per operand, against 2^-24 in
# fp32): its tensor-wide error stays near 5e-6, but single elements where the
# in-chunk terms cancel reach about 1.5e-4 of their slice's RMS. Its bound is
# c = 4: still an element-wise bar, which an error concentrated in a few
# heads or columns at the tensor-wide 1e-4 breaks.
CHUNK_ELEM_C = 4.0
# Rounding errors scale with the magnitudes of the terms that are summed, not
# with the sum: a slice whose outputs cancel (strong decay, beta near 0) has a
# small RMS but errors of the tensor's scale. A slice whose RMS is under this
# fraction of the tensor RMS is measured against that fraction instead.
SLICE_FLOOR = 0.1


def parity(x, ref, inner=1, floor=None):
    """(tensor-wide relative error, max over elements of |x - ref| divided by
    the RMS of the element's slice, floored). `inner` trailing axes form a
    slice."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0, 0.0
    err = np.abs(x - ref)
    g_rms = float(np.sqrt(np.mean(ref ** 2)))
    axes = tuple(range(ref.ndim - inner, ref.ndim))
    s_rms = np.sqrt(np.mean(ref ** 2, axis=axes, keepdims=True))
    fl = SLICE_FLOOR if floor is None else floor
    scale = np.maximum(s_rms, max(fl * g_rms, 1e-300))
    return rel(x, ref), float(np.max(err / scale))


def assert_close(x, ref, tol=1e-4, inner=1, what="", c=ELEM_C):
    """The fp32 parity bar: relative error <= tol per tensor AND every element
    within c * tol of its slice's RMS. Prints both figures (and appends them
    to $GDN_PARITY_LOG when set)."""
    e_norm, e_elem = parity(x, ref, inner)
    msg = f"{what} rel={e_norm:.3e} max_elem/rms={e_elem:.3e}"
    print(msg)
    log = os.environ.get("GDN_PARITY_LOG")
    if log:
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        with open(log, "a") as f:
            extra = {f"elem_floor_{fl:g}": parity(x, ref, inner, fl)[1] for fl in (1e-3, 1e-2, 1.0)}
            f.write(json.dumps({"test": test, "what": what, "rel": e_norm, "elem": e_elem,
                                **extra}) + "\n")
    assert e_norm <= tol, msg
    assert e_elem <= c * tol, msg
    return e_norm, e_elem


def assert_bf16_stored(x, ref, tol=1e-4, inner=1, what="", c=ELEM_C):
    """A value stored in bf16 (a bf16 state page) is one round-to-nearest of
    an fp32 value y that meets the fp32 bar: |y - ref| <= c tol rms, and
    the rounding moves y by at most half a bf16 step, 2^-8 |y| at most. So
    every element obeys |x - ref| <= 2^-8 (|ref| + e) + e, e = c tol rms
    (rms of the element's slice, floored as in parity())."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    g_rms = float(np.sqrt(np.mean(ref ** 2)))
    axes = tuple(range(ref.ndim - inner, ref.ndim))
    s_rms = np.maximum(np.sqrt(np.mean(ref ** 2, axis=axes, keepdims=True)),
                       max(SLICE_FLOOR * g_rms, 1e-300))
    e = c * tol * s_rms
    bound = 2.0 ** -8 * (np.abs(ref) + e) + e
    worst = float(np.max(np.abs(x - ref) / bound))
    msg = f"{what} rel={rel(x, ref):.3e} max_err/bound={worst:.3e}"
    print(msg)
    assert worst <= 1.0, msg
    return worst


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

    def prefill(self, batch, qkv, a, b, chunk_min_rows=0, workspace=False):
        o = self.out(batch.num_rows)
        ws, ws_bytes = None, 0
        if workspace:
            ws_bytes = gdn.gdn_chunk_prefill_workspace_bytes(self.dims, batch)
            ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
        gdn.gdn_prefill(self.dims, batch, self.params, qkv, a, b, o, self.pool.buf, self.status,
                        chunk_min_rows, workspace=ws, workspace_bytes=ws_bytes)
        return o

    def verify(self, batch, qkv, a, b):
        o = self.out(batch.num_rows)
        gdn.gdn_spec_verify(self.dims, batch, self.params, qkv, a, b, o, self.pool.buf,
                            self.status)
        return o

    def spec_step(self, batch, x, a, b):
        o = self.out(batch.num_rows)
        gdn.gdn_spec_step(self.dims, batch, self.params, x, self.conv_w, a, b, o, self.pool.buf,
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
