"""Failure detection without a GPU fault: a bounded on-chip wait that runs
out reports GDN_DEV_TIMEOUT through the status word and leaves the context
usable.

gdn_check_bounded_wait runs the path every kernel takes when one of its own
copies or MMAs does not complete: one block waits on an mbarrier that
nothing arrives at and gives up after the given global time. Nothing
faults, traps or hangs; afterwards the same context runs a normal step,
which must still match the oracle.
"""
import time

import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import oracle
import synth
from tests.gpu_util import Layer, assert_close, f64, to_dev

pytestmark = pytest.mark.gpu


def test_wait_runs_out_reports_timeout_and_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    gdn.gdn_check_bounded_wait(50_000_000, status)          # 50 ms
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == gdn.CODES["GDN_DEV_TIMEOUT"]
    assert 0.045 <= waited < 5.0, waited

    # first error wins: a second expiry leaves the word as it is
    gdn.gdn_check_bounded_wait(1_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.CODES["GDN_DEV_TIMEOUT"]

    # the context still runs the path: the tiny case against the oracle
    d = synth.tiny()
    sh = d["shapes"]
    R = len(d["row_len"])
    L = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], state=gdn.GDN_F32,
              out=gdn.GDN_F32, num_pages=R)
    L.seed(range(R), S0=d["S0"])
    B = L.batch(d["row_start"], d["row_len"], flags=[gdn.GDN_REQ_FRESH] * R)
    o = L.seq(B, to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"]))
    L.ok()
    o_ref, _ = oracle.gdn_f64(d["x"].value, d["a"].value, d["b"].value, d["A_log"],
                              d["dt_bias"], d["row_start"], d["row_len"], sh.Hk, sh.Hv, sh.Dk,
                              sh.Dv, S0=None)
    assert_close(f64(o), o_ref, 1e-4, what="o")
