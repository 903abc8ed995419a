"""gdn_decode (fused conv + rule, one token per request): bit-identical to
gdn_conv followed by gdn_seq (outputs, states, conv windows), within 1e-4 of
the fp64 oracle, and refusing what it does not support."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import oracle
import synth
from tests.gpu_util import Layer, assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu


def two_layers(d, R, state, out, Kc=0, gate_mode=0):
    sh = d["shapes"]
    Ls = [Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=Kc, state=state, out=out,
                num_pages=R + 3, gate_mode=gate_mode) for _ in range(2)]
    S0 = d["S0"][:R]
    if state == gdn.GDN_BF16:
        S0 = oracle.round_bf16(S0).astype(np.float32)
    pages = np.random.default_rng(R).permutation(R + 3)[:R].astype(np.int32)  # scattered, distinct
    for L in Ls:
        L.seed(pages, S0=S0, hist=to_dev(d["hist0"])[:R])
    return Ls, pages, S0


@pytest.mark.parametrize("state,out", [(gdn.GDN_F32, gdn.GDN_F32), (gdn.GDN_BF16, gdn.GDN_BF16),
                                       (gdn.GDN_F32, gdn.GDN_BF16)])
def test_decode_bitwise_equals_conv_then_seq(state, out):
    d = synth.decode()
    R = d["R"]
    (L1, L2), pages, _ = two_layers(d, R, state, out)
    fresh = np.array([r % 5 == 0 for r in range(R)])
    flags = np.where(fresh, gdn.GDN_REQ_FRESH, 0)
    x, a, b = to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"])
    B1 = L1.batch(d["row_start"], d["row_len"], page=pages, flags=flags)
    o1 = L1.out(R)
    gdn.gdn_decode(L1.dims, B1, L1.params, x, L1.conv_w, a, b, o1, L1.pool.buf, L1.status)
    L1.ok()
    B2 = L2.batch(d["row_start"], d["row_len"], page=pages, flags=flags)
    y = L2.conv(B2, x)
    o2 = L2.seq(B2, y, a, b)
    L2.ok()
    assert np.array_equal(bits(o1), bits(o2))
    assert torch.equal(L1.pool.buf, L2.pool.buf)          # states, windows, flags


def test_decode_gate_mode_precomputed_bitwise_equals_conv_then_seq():
    """With precomputed gates (a = g <= 0, b = beta in [0, 1]) the fused step
    still equals gdn_conv + gdn_seq bit for bit (gdn_seq's precomputed-gate
    path is pinned to the oracle in test_gpu_seq.py)."""
    d = synth.decode()
    R = d["R"]
    sh = d["shapes"]
    rng = np.random.default_rng(11)
    g = synth.as_io(-np.abs(rng.standard_normal((R, sh.Hv))) * 0.7, synth.BF16)
    beta = synth.as_io(rng.uniform(0, 1, (R, sh.Hv)), synth.BF16)
    (L1, L2), pages, _ = two_layers(d, R, gdn.GDN_F32, gdn.GDN_F32, gate_mode=1)
    fresh = np.array([r % 7 == 0 for r in range(R)])
    flags = np.where(fresh, gdn.GDN_REQ_FRESH, 0)
    x, a, b = to_dev(d["x"]), to_dev(g), to_dev(beta)
    B1 = L1.batch(d["row_start"], d["row_len"], page=pages, flags=flags)
    o1 = L1.out(R)
    gdn.gdn_decode(L1.dims, B1, L1.params, x, L1.conv_w, a, b, o1, L1.pool.buf, L1.status)
    L1.ok()
    B2 = L2.batch(d["row_start"], d["row_len"], page=pages, flags=flags)
    y = L2.conv(B2, x)
    o2 = L2.seq(B2, y, a, b)
    L2.ok()
    assert np.array_equal(bits(o1), bits(o2))
    assert torch.equal(L1.pool.buf, L2.pool.buf)


def test_decode_vs_oracle_and_repeated_steps():
    """Three decode steps in a row against the oracle's conv mirror + fp64 rule."""
    d = synth.decode(R=8)
    sh = d["shapes"]
    R = 8
    L = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], num_pages=R)
    L.seed(range(R), S0=d["S0"], hist=to_dev(d["hist0"]))
    rng = np.random.default_rng(3)
    hist = d["hist0"].value.copy()
    S = d["S0"].astype(np.float64)
    for step in range(3):
        rows = synth.rows(rng, R, sh, synth.BF16)
        B = L.batch(np.arange(R), np.ones(R))
        o = L.out(R)
        gdn.gdn_decode(L.dims, B, L.params, to_dev(rows["x"]), L.conv_w, to_dev(rows["a"]),
                       to_dev(rows["b"]), o, L.pool.buf, L.status)
        L.ok()
        y, hist = oracle.conv_f32(rows["x"].value, hist, d["conv_w"].value, np.arange(R), np.ones(R))
        o_ref, S = oracle.gdn_f64(oracle.round_bf16(y), rows["a"].value, rows["b"].value,
                                  d["A_log"], d["dt_bias"], np.arange(R), np.ones(R), sh.Hk,
                                  sh.Hv, sh.Dk, sh.Dv, S0=S)
        hist = hist.astype(np.float64)
        assert_close(f64(o), o_ref, 1e-4, what=f"o step {step}")
    Sg = np.stack([f64(L.pool.state_math(r)) for r in range(R)])
    assert_close(Sg, S, 1e-4, inner=2, what="S")


@pytest.mark.parametrize("shape", [(4, 8, 64), (2, 2, 32), (1, 4, 128)])
@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_decode_other_head_shapes(shape, state):
    Hk, Hv, D = shape
    sh = synth.Shapes(Hk=Hk, Hv=Hv, Dk=D, Dv=D)
    io = synth.F32 if D == 32 else synth.BF16
    d = synth.decode(R=6, sh=sh, io=io)
    (L1, L2), pages, _ = two_layers(d, 6, state, gdn.GDN_F32)
    x, a, b = to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"])
    B1 = L1.batch(d["row_start"], d["row_len"], page=pages)
    o1 = L1.out(6)
    gdn.gdn_decode(L1.dims, B1, L1.params, x, L1.conv_w, a, b, o1, L1.pool.buf, L1.status)
    L1.ok()
    B2 = L2.batch(d["row_start"], d["row_len"], page=pages)
    o2 = L2.seq(B2, L2.conv(B2, x), a, b)
    L2.ok()
    assert np.array_equal(bits(o1), bits(o2))
    assert torch.equal(L1.pool.buf, L2.pool.buf)


def _page_bytes(L, p):
    lay = L.pool.layout
    return L.pool.buf[p * lay.page_bytes:(p + 1) * lay.page_bytes].clone()


def test_decode_skips_spec_zeroes_empty_fresh_and_refuses_open_records():
    d = synth.decode(R=4)
    (L1, L2), pages, _ = two_layers(d, 4, gdn.GDN_F32, gdn.GDN_F32, Kc=8)
    x, a, b = to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"])
    # request 1 is SPEC (skipped), request 2 is FRESH with no token
    flags = [0, gdn.GDN_REQ_SPEC, gdn.GDN_REQ_FRESH, 0]
    ln = [1, 1, 0, 1]
    spec_page = _page_bytes(L1, pages[1])
    B = L1.batch(d["row_start"], ln, page=pages, flags=flags, num_rows=4)
    o = L1.out(4)
    gdn.gdn_decode(L1.dims, B, L1.params, x, L1.conv_w, a, b, o, L1.pool.buf, L1.status)
    L1.ok()
    assert torch.equal(spec_page, _page_bytes(L1, pages[1]))
    # the two-launch path on the plain requests alone
    keep = [0, 2, 3]
    B2 = L2.batch(np.asarray(d["row_start"])[keep], np.asarray(ln)[keep], page=pages[keep],
                  flags=np.asarray(flags)[keep], num_rows=4)
    o2 = L2.seq(B2, L2.conv(B2, x), a, b)
    L2.ok()
    for r in keep:
        assert torch.equal(_page_bytes(L1, pages[r]), _page_bytes(L2, pages[r])), r
    assert np.array_equal(bits(o[[0, 3]]), bits(o2[[0, 3]]))
    assert float(L1.pool.state(pages[2]).abs().max()) == 0.0
    assert float(L1.pool.window(pages[2])[:3].float().abs().max()) == 0.0
    # an open record on request 3's page: refused, nothing written there
    L1.pool.flag(pages[3]).fill_(8 << 2)
    before = _page_bytes(L1, pages[3])
    B = L1.batch(d["row_start"], [1, 1, 1, 1], page=pages, flags=[0, gdn.GDN_REQ_SPEC, 0, 0])
    o = L1.out(4)
    gdn.gdn_decode(L1.dims, B, L1.params, x, L1.conv_w, a, b, o, L1.pool.buf, L1.status)
    assert L1.status_code() == gdn.CODES["GDN_DEV_RECORD_OPEN"]
    assert torch.equal(before, _page_bytes(L1, pages[3]))
    # more than one token per request: refused on the host (max_rows) ...
    L1.reset_status()
    B = L1.batch([0, 1], [1, 2], page=pages[:2], flags=[0, 0], num_rows=4)
    with pytest.raises(gdn.GdnError) as err:
        gdn.gdn_decode(L1.dims, B, L1.params, x, L1.conv_w, a, b, o, L1.pool.buf, L1.status)
    assert err.value.code == gdn.CODES["GDN_ERR_INVALID_ARG"]
    # ... and on the device when max_rows understates a row count
    B = L1.batch([0, 1], [1, 2], page=pages[:2], flags=[0, 0], num_rows=4, max_rows=1)
    gdn.gdn_decode(L1.dims, B, L1.params, x, L1.conv_w, a, b, o, L1.pool.buf, L1.status)
    assert L1.status_code() == gdn.CODES["GDN_DEV_BAD_ROWS"]


def test_max_request_count_in_one_launch():
    """65535 one-token requests (the most one launch takes; more is refused
    on the host) through gdn_decode and through gdn_conv + gdn_seq: equal bit
    for bit, and sampled requests within 1e-4 of the oracle."""
    R = 65535
    sh = synth.Shapes(Hk=2, Hv=2, Dk=32, Dv=32)
    d = synth.decode(R=R, sh=sh, io=synth.F32)
    (L1, L2), pages, S0 = two_layers(d, R, gdn.GDN_F32, gdn.GDN_F32)
    x, a, b = to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"])
    B1 = L1.batch(d["row_start"], d["row_len"], page=pages)
    o1 = L1.out(R)
    gdn.gdn_decode(L1.dims, B1, L1.params, x, L1.conv_w, a, b, o1, L1.pool.buf, L1.status)
    L1.ok()
    B2 = L2.batch(d["row_start"], d["row_len"], page=pages)
    o2 = L2.seq(B2, L2.conv(B2, x), a, b)
    L2.ok()
    assert np.array_equal(bits(o1), bits(o2))
    assert torch.equal(L1.pool.buf, L2.pool.buf)
    for r in (0, 1, 40000, R - 1):
        y, _ = oracle.conv_f64(d["x"].value[r:r + 1], d["hist0"].value[r:r + 1], d["conv_w"].value,
                               [0], [1])
        o_ref, S_ref = oracle.gdn_f64(y, d["a"].value[r:r + 1], d["b"].value[r:r + 1], d["A_log"],
                                      d["dt_bias"], [0], [1], sh.Hk, sh.Hv, sh.Dk, sh.Dv,
                                      S0=S0[r:r + 1])
        assert_close(f64(o1[r]), o_ref[0], 1e-4, what=f"o request {r}")
        assert_close(f64(L1.pool.state_math(int(pages[r]))), S_ref[0], 1e-4, inner=2,
                     what=f"S request {r}")
