"""gdn_conv against the CPU fp32-accumulate conv: bit for bit.

fp32 outputs are compared first (a bf16 store could hide a 1-ulp fp32
difference), then bf16 outputs, then the rolled conv window.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import oracle
import synth
from tests.gpu_util import Layer, bits, to_dev

pytestmark = pytest.mark.gpu


def run_conv(d, lengths, order=None, fresh=None, seed=0, bias=False):
    sh, io = d["shapes"], d["io"]
    rng = np.random.default_rng(seed)
    R = len(lengths)
    start, ln, T = synth.pack(lengths, order)
    x = synth.as_io(rng.standard_normal((T, sh.C)), io)
    hist = synth.as_io(rng.standard_normal((R, sh.W - 1, sh.C)), io)
    fresh = np.zeros(R, bool) if fresh is None else np.asarray(fresh)
    L = Layer(sh, io, d["A_log"], d["dt_bias"], d["conv_w"], num_pages=R)
    cb = None
    if bias:
        cb_np = rng.standard_normal(sh.C).astype(np.float32)
        cb = to_dev(cb_np)
        L.params = gdn.make_params(L.A_log, L.dt_bias, conv_bias=cb)
    L.seed(range(R), hist=to_dev(hist))
    flags = np.where(fresh, gdn.GDN_REQ_FRESH, 0)
    B = L.batch(start, ln, flags=flags)
    xd = to_dev(x)
    y32 = L.conv(B, xd, gdn.GDN_F32)
    L.ok()
    win = torch.stack([L.pool.window(r)[: sh.W - 1].clone() for r in range(R)])
    # the window was rolled by the first call: restore it for the bf16 call
    L.seed(range(R), hist=to_dev(hist))
    yio = L.conv(B, xd)
    L.ok()
    # CPU reference: fp32 mirror with the same history (zero for fresh ones)
    h_ref = hist.value.copy()
    h_ref[fresh] = 0.0
    y_ref, h_out = oracle.conv_f32(x.value, h_ref, d["conv_w"].value, start, ln,
                                   bias=None if cb is None else cb_np)
    return y32, yio, win, y_ref, h_out


@pytest.mark.parametrize("cfg", ["tiny", "decode"])
def test_conv_bitwise_workloads(cfg):
    d = synth.tiny() if cfg == "tiny" else synth.decode()
    R = d["R"]
    lengths = list(np.asarray(d["row_len"]))
    y32, yio, win, y_ref, h_out = run_conv(d, lengths, seed=R)
    assert np.array_equal(bits(y32), y_ref.view(np.int32))
    if d["io"] == synth.BF16:
        assert np.array_equal(bits(yio), synth.bf16_bits(y_ref).view(np.int16))
        assert np.array_equal(bits(win), synth.bf16_bits(h_out).view(np.int16))
    else:
        assert np.array_equal(bits(yio), y_ref.view(np.int32))
        assert np.array_equal(bits(win), h_out.view(np.int32))


def test_conv_ragged_rows_fresh_and_continuing_shuffled():
    d = synth.decode(R=1)
    lengths = [1, 2, 3, 31, 32, 33, 100, 257, 0, 5]
    order = [7, 2, 9, 0, 5, 1, 8, 3, 6, 4]
    fresh = [i % 2 == 0 for i in range(len(lengths))]
    y32, yio, win, y_ref, h_out = run_conv(d, lengths, order=order, fresh=fresh, seed=3)
    assert np.array_equal(bits(y32), y_ref.view(np.int32))
    assert np.array_equal(bits(yio), synth.bf16_bits(y_ref).view(np.int16))
    assert np.array_equal(bits(win), synth.bf16_bits(h_out).view(np.int16))


def test_conv_with_bias_fp32_rows():
    d = synth.tiny()
    y32, yio, win, y_ref, h_out = run_conv(d, [16, 7, 40], bias=True, seed=5)
    assert np.array_equal(bits(y32), y_ref.view(np.int32))
    assert np.array_equal(bits(win), h_out.view(np.int32))


def test_conv_long_request_with_initial_window_is_race_free():
    """One request far longer than a row tile, with an initial window: every
    block but the first reads rows, only the first reads and writes the
    window. Run several times: identical bits and equal to the CPU conv."""
    d = synth.decode(R=1)
    outs = []
    for rep in range(3):
        y32, _, win, y_ref, h_out = run_conv(d, [4099], seed=11)
        outs.append((bits(y32), bits(win)))
        assert np.array_equal(outs[-1][0], y_ref.view(np.int32))
        assert np.array_equal(outs[-1][1], synth.bf16_bits(h_out).view(np.int16))
    assert all(np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1]) for o in outs)


def test_own_exp_silu_against_cuda_expf():
    """SiLU of the conv (own exp, correctly rounded quotient) on the GPU: bit-identical
    to the CPU mirror, within 4 ulp of the exact value (2^-140 absolutely
    where e^x is subnormal), and within 8 ulp of torch's CUDA-exp SiLU on the
    same values (the two methods' bounds added: neither need match the
    other)."""
    sh = synth.Shapes(Hk=1, Hv=1, Dk=32, Dv=32)
    C = sh.C
    # identity taps: w = [0, 0, 0, 1], so y = SiLU(x)
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0
    conv_w = synth.as_io(w, synth.F32)
    xs = np.concatenate([np.linspace(-104, 104, 96 * 300),
                         np.linspace(-1, 1, 96 * 20)]).astype(np.float32).reshape(-1, C)
    T = xs.shape[0]
    x = synth.as_io(xs, synth.F32)
    L = Layer(sh, synth.F32, np.zeros(1), np.zeros(1), conv_w)
    B = L.batch([0], [T])
    y = L.conv(B, to_dev(x), gdn.GDN_F32)
    L.ok()
    got = y.cpu().numpy()
    mirror, _ = oracle.conv_f32(xs, np.zeros((1, 3, C)), w, [0], [T])
    assert np.array_equal(got.view(np.int32), mirror.astype(np.float32).view(np.int32))
    x64 = xs.astype(np.float64)
    exact = x64 * np.exp(np.minimum(x64, 0)) / (1.0 + np.exp(-np.abs(x64)))
    normal = np.abs(xs) <= 87
    tol = 4 * np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64) + 1e-45
    assert np.all(np.abs(got - exact)[normal] <= tol[normal])
    assert np.all(np.abs(got - exact)[~normal] <= 2.0 ** -140)
    xt = torch.from_numpy(xs).cuda()
    ref = (xt / (1.0 + torch.exp(-xt))).cpu().numpy()
    inside = np.abs(xs) <= 80
    tol8 = 8 * np.spacing(np.abs(ref).astype(np.float32)) + 1e-45
    assert np.all(np.abs(got - ref)[inside] <= tol8[inside])
