"""The usage example the README shows (one fused decode step), kept here as
code: it runs through the C ABI and produces finite, non-zero outputs."""
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
from gated_deltanet_linear_14_gb300.pages import PagePool

pytestmark = pytest.mark.gpu


def test_usage_example_runs():
    R, Hk, Hv, D = 64, 16, 32, 128
    dims = gdn.make_dims(Hk, Hv, D, D, W=4, Kc=8, io=gdn.GDN_BF16, state=gdn.GDN_F32,
                         out=gdn.GDN_BF16)
    pool = PagePool(dims, R)                       # zero-filled pages are valid empty pages
    A_log = torch.rand(Hv, device="cuda") * 2 - 1
    dt_bias = torch.rand(Hv, device="cuda") - 0.5
    params = gdn.make_params(A_log, dt_bias)       # scale 0 selects Dk^-1/2
    conv_w = (torch.rand(dims.C, 4, device="cuda") - 0.5).to(torch.bfloat16)

    # one decode token per request; the row map lives in device memory and
    # must stay alive while the batch is in use
    def i32(v):
        return torch.tensor(list(v), dtype=torch.int32, device="cuda")

    row_start, row_len, page = i32(range(R)), i32([1] * R), i32(range(R))
    flags = i32([gdn.GDN_REQ_FRESH] * R)
    batch = gdn.make_batch(R, R, 1, R, row_start, row_len, page, flags)

    x = torch.randn(R, dims.C, device="cuda").to(torch.bfloat16)
    a = torch.randn(R, Hv, device="cuda").to(torch.bfloat16)
    b = torch.randn(R, Hv, device="cuda").to(torch.bfloat16)
    o = torch.empty(R, Hv, D, device="cuda", dtype=torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_decode(dims, batch, params, x, conv_w, a, b, o, pool.buf, status)
    gdn.raise_on_status(status)

    assert int(status.item()) == 0
    assert bool(o.float().isfinite().all())
    assert float(o.float().abs().max()) > 0.0
