"""Steps captured in a CUDA graph equal the same steps run eagerly, bit for bit.

The r9700-stack v0.2.4 notes ("A defect found and fixed before the tag")
describe a conv-window width taken from a tensor shape that differed between
graph-captured and eager steps. Here everything a step depends on (row map,
step parity, accepted counts, the record width in each page's flag word)
lives in device memory, so one captured step replays correctly for every
later step once its inputs are written in place.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import synth
from tests.gpu_util import Layer, bits, to_dev

pytestmark = pytest.mark.gpu

SPEC, PAR = gdn.GDN_REQ_SPEC, gdn.GDN_REQ_PARITY


def _layer(d, R):
    L = Layer(d["shapes"], d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R)
    L.seed(range(R), S0=d["S0"][:R], hist=to_dev(d["hist0"])[:R])
    return L


@pytest.mark.parametrize("fused", [False, True])
def test_spec_steps_graph_replay_equals_eager(fused):
    """Captured conv + verify (or the fused gdn_spec_step) replayed over 6
    steps: outputs and pages equal the eager conv + verify steps."""
    R, n, steps = 8, 8, 6
    d = synth.spec(R=R, steps=steps)
    start, ln = d["row_start"], d["row_len"]

    # eager
    Le = _layer(d, R)
    outs_e = []
    for s in range(steps):
        rows = d["step_rows"][s]
        flags = np.full(R, SPEC | (PAR if s % 2 else 0))
        B = Le.batch(start, ln, flags=flags, n_accepted=d["accepted"][s])
        y = Le.conv(B, to_dev(rows["x"]))
        outs_e.append(Le.verify(B, y, to_dev(rows["a"]), to_dev(rows["b"])).clone())
        Le.ok()

    # graph: static buffers, step inputs written in place before each replay
    Lg = _layer(d, R)
    T = R * n
    x = to_dev(d["step_rows"][0]["x"]).clone()
    a = to_dev(d["step_rows"][0]["a"]).clone()
    b = to_dev(d["step_rows"][0]["b"]).clone()
    flags_t = torch.zeros(R, dtype=torch.int32, device="cuda")
    acc_t = torch.zeros(R, dtype=torch.int32, device="cuda")
    y = torch.zeros(T, d["shapes"].C, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(T, d["shapes"].Hv, d["shapes"].Dv, dtype=torch.float32, device="cuda")
    rs, rl, pg = (torch.from_numpy(np.asarray(v, np.int32)).cuda() for v in (start, ln, np.arange(R)))
    B = gdn.make_batch(R, T, n, R, rs, rl, pg, flags_t, acc_t)

    def step():
        if fused:
            gdn.gdn_spec_step(Lg.dims, B, Lg.params, x, Lg.conv_w, a, b, o, Lg.pool.buf, Lg.status)
            return
        gdn.gdn_conv(Lg.dims, B, Lg.params, x, Lg.conv_w, y, gdn.GDN_BF16, Lg.pool.buf, Lg.status)
        gdn.gdn_spec_verify(Lg.dims, B, Lg.params, y, a, b, o, Lg.pool.buf, Lg.status)

    def load_inputs(s):
        rows = d["step_rows"][s]
        x.copy_(to_dev(rows["x"]))
        a.copy_(to_dev(rows["a"]))
        b.copy_(to_dev(rows["b"]))
        flags_t.copy_(torch.full((R,), SPEC | (PAR if s % 2 else 0), dtype=torch.int32))
        acc_t.copy_(torch.from_numpy(np.asarray(d["accepted"][s], np.int32)))

    # capture on a side stream (the pages are not touched by the capture)
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            step()
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()

    for s in range(steps):
        load_inputs(s)
        g.replay()
        torch.cuda.synchronize()
        Lg.ok()
        assert np.array_equal(bits(o), bits(outs_e[s])), f"step {s}"
    assert torch.equal(Lg.pool.buf, Le.pool.buf)


def test_decode_graph_replay_equals_eager():
    d = synth.decode(R=16)
    R = 16
    rng = np.random.default_rng(17)
    inputs = [synth.rows(rng, R, d["shapes"], synth.BF16) for _ in range(4)]
    Le = _layer(d, R)
    Lg = _layer(d, R)
    Be = Le.batch(np.arange(R), np.ones(R))
    outs = []
    for rows in inputs:
        o = Le.out(R)
        gdn.gdn_decode(Le.dims, Be, Le.params, to_dev(rows["x"]), Le.conv_w, to_dev(rows["a"]),
                       to_dev(rows["b"]), o, Le.pool.buf, Le.status)
        outs.append(o)
    Le.ok()
    x, a, b = (to_dev(inputs[0][k]).clone() for k in ("x", "a", "b"))
    o = Lg.out(R)
    Bg = Lg.batch(np.arange(R), np.ones(R))
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            gdn.gdn_decode(Lg.dims, Bg, Lg.params, x, Lg.conv_w, a, b, o, Lg.pool.buf, Lg.status)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    for i, rows in enumerate(inputs):
        x.copy_(to_dev(rows["x"]))
        a.copy_(to_dev(rows["a"]))
        b.copy_(to_dev(rows["b"]))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(o), bits(outs[i])), i
    Lg.ok()
    assert torch.equal(Lg.pool.buf, Le.pool.buf)
