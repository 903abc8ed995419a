"""gdn_chunk_prefill (tensor-core chunked form) against the fp64 token loop.

Bar: relative error <= 1e-4 per tensor with fp32 state and fp32 outputs, on
ragged requests (several chunks, an exact chunk, one token, none), with and
without an initial state, and at the full long-prefill size (4 x 8192 tokens,
16/32 heads) on sampled heads the oracle recomputes exactly.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import oracle
import synth
from tests.gpu_util import CHUNK_ELEM_C, Layer, assert_bf16_stored, assert_close, f64, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-4


def chunk_run(L, B, qkv, a, b, o_dtype=torch.float32):
    o = torch.zeros(B.num_rows, L.sh.Hv, L.sh.Dv, dtype=o_dtype, device="cuda")
    ws_bytes = gdn.gdn_chunk_prefill_workspace_bytes(L.dims, B)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_prefill(L.dims, B, L.params, qkv, a, b, o, L.pool.buf, ws, ws_bytes, L.status)
    return o


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_chunk_ragged_requests_vs_oracle(state):
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    rng = np.random.default_rng(101)
    lengths = [200, 64, 1, 130, 0, 129]
    R = len(lengths)
    order = [3, 0, 5, 1, 4, 2]
    start, ln, T = synth.pack(lengths, order)
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    S0 = synth.state(rng, R, sh, std=0.1)
    fresh = np.array([False, True, False, True, True, False])
    S0[fresh] = 0.0
    if state == gdn.GDN_BF16:
        S0 = oracle.round_bf16(S0).astype(np.float32)
    L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], state=state, num_pages=R)
    L.seed(range(R), S0=S0)
    B = L.batch(start, ln, flags=np.where(fresh, gdn.GDN_REQ_FRESH, 0))
    o = chunk_run(L, B, to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"]))
    L.ok()
    o_ref, S_ref = oracle.gdn_f64(rows["x"].value, rows["a"].value, rows["b"].value, d["A_log"],
                                  d["dt_bias"], start, ln, sh.Hk, sh.Hv, sh.Dk, sh.Dv, S0=S0)
    assert_close(f64(o), o_ref, TOL, what="o", c=CHUNK_ELEM_C)
    S = np.stack([f64(L.pool.state_math(r)) for r in range(R)])
    for r in range(R):
        if ln[r]:
            sl = slice(start[r], start[r] + ln[r])
            assert_close(f64(o[sl]), o_ref[sl], TOL, what=f"o request {r}", c=CHUNK_ELEM_C)
        if state == gdn.GDN_F32:
            assert_close(S[r], S_ref[r], TOL, inner=2, what=f"S request {r}", c=CHUNK_ELEM_C)
        else:   # a bf16 page rounds the stored state once
            assert_bf16_stored(S[r], S_ref[r], TOL, inner=2, what=f"S request {r}",
                               c=CHUNK_ELEM_C)


def test_chunk_agrees_with_token_by_token_kernel_and_skips_spec():
    """Plain requests: chunked and token-by-token GPU results agree; SPEC
    requests in the same batch are left alone by the chunked prefill."""
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    rng = np.random.default_rng(7)
    lengths = [150, 70, 8]
    start, ln, T = synth.pack(lengths)
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    S0 = synth.state(rng, 3, sh, std=0.05)
    qkv, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
    flags = [0, 0, gdn.GDN_REQ_SPEC]
    L1 = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=3)
    L1.seed(range(3), S0=S0)
    before = L1.pool.state(2).clone()
    o1 = chunk_run(L1, L1.batch(start, ln, flags=flags, n_accepted=[0, 0, 0]), qkv, a, b)
    L1.ok()
    L2 = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=3)
    L2.seed(range(3), S0=S0)
    o2 = L2.seq(L2.batch(start, ln, flags=flags, n_accepted=[0, 0, 0]), qkv, a, b)
    L2.ok()
    sl = slice(0, 220)
    assert_close(f64(o1[sl]), f64(o2[sl]), 2 * TOL, what="o chunk vs seq", c=CHUNK_ELEM_C)
    for r in range(2):
        assert_close(f64(L1.pool.state_math(r)), f64(L2.pool.state_math(r)), 2 * TOL, inner=2,
                     what=f"S chunk vs seq {r}", c=CHUNK_ELEM_C)
    assert torch.equal(L1.pool.state(2), before)


def test_chunk_gate_mode_precomputed():
    sh = synth.Shapes(Hk=1, Hv=2, Dk=128, Dv=128)
    rng = np.random.default_rng(8)
    T = 100
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    rows["a"] = synth.as_io(-np.abs(rng.standard_normal((T, sh.Hv))) * 0.5, synth.BF16)
    rows["b"] = synth.as_io(rng.uniform(0, 1, (T, sh.Hv)), synth.BF16)
    L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], gate_mode=1)
    B = L.batch([0], [T], flags=gdn.GDN_REQ_FRESH)
    o = chunk_run(L, B, to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"]))
    L.ok()
    o_ref, S_ref = oracle.gdn_f64(rows["x"].value, rows["a"].value, rows["b"].value, d["A_log"],
                                  d["dt_bias"], [0], [T], 1, 2, 128, 128, gate_mode=1)
    assert_close(f64(o), o_ref, TOL, what="o", c=CHUNK_ELEM_C)
    assert_close(f64(L.pool.state_math(0)), S_ref[0], TOL, inner=2, what="S", c=CHUNK_ELEM_C)


@pytest.mark.parametrize("path", ["chunk", "seq"])
@pytest.mark.parametrize("case", ["strong_decay", "no_decay", "beta_edges"])
def test_gate_extremes_vs_oracle(case, path):
    """Precomputed gates at their extremes on a ragged 150-token sequence,
    chunked and token by token: g down to -40 per token (in-chunk decays far
    below fp32's range), g = 0 (nothing decays), and beta exactly 0 or 1."""
    sh = synth.Shapes(Hk=1, Hv=2, Dk=128, Dv=128)
    rng = np.random.default_rng({"strong_decay": 11, "no_decay": 12, "beta_edges": 13}[case])
    T = 150
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    if case == "strong_decay":
        g = rng.uniform(-40.0, -8.0, (T, sh.Hv))
        beta = rng.uniform(0.0, 1.0, (T, sh.Hv))
    elif case == "no_decay":
        g = np.zeros((T, sh.Hv))
        beta = rng.uniform(0.0, 1.0, (T, sh.Hv))
    else:
        g = rng.uniform(-1.0, 0.0, (T, sh.Hv))
        beta = rng.integers(0, 2, (T, sh.Hv)).astype(np.float64)
    rows["a"] = synth.as_io(g, synth.BF16)
    rows["b"] = synth.as_io(beta, synth.BF16)
    L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], gate_mode=1)
    B = L.batch([0], [T], flags=gdn.GDN_REQ_FRESH)
    x, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
    o = chunk_run(L, B, x, a, b) if path == "chunk" else L.seq(B, x, a, b)
    L.ok()
    assert bool(torch.isfinite(o.float()).all())
    o_ref, S_ref = oracle.gdn_f64(rows["x"].value, rows["a"].value, rows["b"].value, d["A_log"],
                                  d["dt_bias"], [0], [T], 1, 2, 128, 128, gate_mode=1)
    assert_close(f64(o), o_ref, TOL, what=f"o {case} {path}",
                 c=CHUNK_ELEM_C if path == "chunk" else 1.0)
    assert_close(f64(L.pool.state_math(0)), S_ref[0], TOL, inner=2, what=f"S {case} {path}",
                 c=CHUNK_ELEM_C if path == "chunk" else 1.0)


def _head_pair(d, rows, r, kh, start, ln):
    """The oracle's inputs for value heads 2kh, 2kh+1 (q/k head kh) of request r."""
    sh = d["shapes"]
    D = sh.Dk
    sl = slice(start[r], start[r] + ln[r])
    x = rows["x"].value[sl]
    h0 = kh * (sh.Hv // sh.Hk)
    q = x[:, kh * D:(kh + 1) * D]
    k = x[:, sh.Hk * D + kh * D: sh.Hk * D + (kh + 1) * D]
    v = x[:, 2 * sh.Hk * D + h0 * D: 2 * sh.Hk * D + (h0 + 2) * D]
    qkv = np.concatenate([q, k, v], axis=1)
    a = rows["a"].value[sl][:, h0:h0 + 2]
    b = rows["b"].value[sl][:, h0:h0 + 2]
    return qkv, a, b, h0


def test_chunk_long_prefill_full_size_sampled_heads():
    """4 x 8192 tokens at 16/32 heads, launched as the benchmark launches it;
    the oracle recomputes four sampled (request, head-pair) chains whole."""
    d = synth.long()
    sh = d["shapes"]
    start, ln = d["row_start"], d["row_len"]
    L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], num_pages=d["R"])
    B = L.batch(start, ln, flags=gdn.GDN_REQ_FRESH)
    rows = {"x": d["x"], "a": d["a"], "b": d["b"]}
    o = chunk_run(L, B, to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"]))
    L.ok()
    assert torch.isfinite(o).all()
    # the benchmark's bf16 outputs: exactly the fp32 outputs rounded to nearest even
    Lb = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], num_pages=d["R"],
               out=gdn.GDN_BF16)
    Bb = Lb.batch(start, ln, flags=gdn.GDN_REQ_FRESH)
    ob = chunk_run(Lb, Bb, to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"]), o_dtype=torch.bfloat16)
    Lb.ok()
    assert ob.dtype == torch.bfloat16 and torch.equal(ob, o.to(torch.bfloat16))
    assert torch.equal(Lb.pool.buf, L.pool.buf)
    del Lb, Bb, ob
    for r, kh in ((0, 0), (1, 7), (2, 11), (3, 15)):
        qkv, a, b, h0 = _head_pair(d, rows, r, kh, start, ln)
        o_ref, S_ref = oracle.gdn_f64(qkv, a, b, d["A_log"][h0:h0 + 2], d["dt_bias"][h0:h0 + 2],
                                      [0], [ln[r]], 1, 2, sh.Dk, sh.Dv)
        sl = slice(start[r], start[r] + ln[r])
        assert_close(f64(o[sl, h0:h0 + 2]), o_ref, TOL, what=f"o request {r} heads {h0},{h0 + 1}",
                     c=CHUNK_ELEM_C)
        S = f64(L.pool.state_math(r))[h0:h0 + 2]
        assert_close(S, S_ref[0], TOL, inner=2, what=f"S request {r} heads {h0},{h0 + 1}", c=CHUNK_ELEM_C)


@pytest.mark.parametrize("use_ws", [False, True])
def test_prefill_dispatch_matches_each_path(use_ws):
    """gdn_prefill sends requests with >= threshold rows through the chunked
    form (one launch without a workspace, two passes with one) and the rest
    token by token: each request equals, bit for bit, the kernel it was sent
    to, and all are within 1e-4 of the oracle."""
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    rng = np.random.default_rng(55)
    lengths = [20, 63, 64, 200, 1, 0, 130]
    R = len(lengths)
    start, ln, T = synth.pack(lengths, [6, 2, 0, 5, 1, 4, 3])
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    S0 = synth.state(rng, R, sh, std=0.1)
    fresh = np.array([False, True, False, False, False, True, False])
    S0[fresh] = 0.0
    qkv, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
    flags = np.where(fresh, gdn.GDN_REQ_FRESH, 0)
    thr = 64

    def layer():
        L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], num_pages=R)
        L.seed(range(R), S0=S0)
        return L

    Lp = layer()
    Bp = Lp.batch(start, ln, flags=flags)
    op = Lp.out(T)
    ws_bytes = gdn.gdn_chunk_prefill_workspace_bytes(Lp.dims, Bp) if use_ws else 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if use_ws else None
    gdn.gdn_prefill(Lp.dims, Bp, Lp.params, qkv, a, b, op, Lp.pool.buf, Lp.status, thr,
                    workspace=ws, workspace_bytes=ws_bytes)
    Lp.ok()
    Ls = layer()
    os_ = Ls.seq(Ls.batch(start, ln, flags=flags), qkv, a, b)
    Ls.ok()
    Lc = layer()
    oc = chunk_run(Lc, Lc.batch(start, ln, flags=flags), qkv, a, b)
    Lc.ok()
    for r in range(R):
        sl = slice(start[r], start[r] + ln[r])
        ref_o, ref_L = (oc, Lc) if ln[r] >= thr else (os_, Ls)
        assert torch.equal(op[sl], ref_o[sl]), r
        assert torch.equal(Lp.pool.state(r), ref_L.pool.state(r)), r
    o_ref, S_ref = oracle.gdn_f64(rows["x"].value, rows["a"].value, rows["b"].value, d["A_log"],
                                  d["dt_bias"], start, ln, sh.Hk, sh.Hv, sh.Dk, sh.Dv, S0=S0)
    assert_close(f64(op), o_ref, TOL, what="o", c=CHUNK_ELEM_C)
    S = np.stack([f64(Lp.pool.state_math(r)) for r in range(R)])
    assert_close(S, S_ref, TOL, inner=2, what="S", c=CHUNK_ELEM_C)


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_two_pass_form_bit_identical_to_one_launch_form(state):
    """gdn_chunk_prefill with a workspace (chunk-parallel pre-pass, then the
    state chain) and without one (everything on the chain) produce the same
    outputs and final states bit for bit, on ragged requests with and
    without an initial state."""
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    rng = np.random.default_rng(211)
    lengths = [300, 64, 1, 130, 0, 191, 65]
    R = len(lengths)
    start, ln, T = synth.pack(lengths, [4, 2, 6, 0, 5, 1, 3])
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    S0 = synth.state(rng, R, sh, std=0.1)
    fresh = np.array([False, True, False, False, True, True, False])
    if state == gdn.GDN_BF16:
        S0 = oracle.round_bf16(S0).astype(np.float32)
    qkv, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
    outs = []
    for use_ws in (False, True):
        L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], state=state, num_pages=R)
        L.seed(range(R), S0=S0)
        B = L.batch(start, ln, flags=np.where(fresh, gdn.GDN_REQ_FRESH, 0))
        o = torch.zeros(B.num_rows, sh.Hv, sh.Dv, dtype=torch.float32, device="cuda")
        ws_bytes = gdn.gdn_chunk_prefill_workspace_bytes(L.dims, B)
        assert ws_bytes == R * sh.Hv * ((max(lengths) + 63) // 64) * 99328
        ws = torch.full((ws_bytes,), 0xA5, dtype=torch.uint8, device="cuda") if use_ws else None
        gdn.gdn_chunk_prefill(L.dims, B, L.params, qkv, a, b, o, L.pool.buf, ws,
                              ws_bytes if use_ws else 0, L.status)
        L.ok()
        outs.append((o.clone(), torch.stack([L.pool.state(r).clone() for r in range(R)])))
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
    s0, s1 = outs[0][1], outs[1][1]
    assert torch.equal(s0.view(torch.int16) if s0.dtype == torch.bfloat16 else s0.view(torch.int32),
                       s1.view(torch.int16) if s1.dtype == torch.bfloat16 else s1.view(torch.int32))


def test_two_pass_form_rejects_a_short_workspace():
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    rng = np.random.default_rng(5)
    start, ln, T = synth.pack([100, 20])
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], num_pages=2)
    B = L.batch(start, ln, flags=gdn.GDN_REQ_FRESH)
    o = torch.zeros(T, sh.Hv, sh.Dv, dtype=torch.float32, device="cuda")
    need = gdn.gdn_chunk_prefill_workspace_bytes(L.dims, B)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn.GdnError):
        gdn.gdn_chunk_prefill(L.dims, B, L.params, to_dev(rows["x"]), to_dev(rows["a"]),
                              to_dev(rows["b"]), o, L.pool.buf, ws, need - 16, L.status)
