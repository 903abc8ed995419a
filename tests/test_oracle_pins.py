"""Pins for the CPU oracle: brute force, closed forms and invariants.

None of these re-type the oracle's formula. Each compares the oracle with a
different formulation (``oracle.brute``), a closed form, or a property the
mathematics fixes, and the mutation test at the end shows that planted
mistakes in the oracle fail at least one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import brute
import synth


def rel(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def random_case(seed, T, Hk, Hv, Dk, Dv, s0_std=0.3, gate_mode=0):
    rng = np.random.default_rng(seed)
    C = 2 * Hk * Dk + Hv * Dv
    qkv = rng.standard_normal((T, C))
    a = rng.standard_normal((T, Hv))
    b = rng.standard_normal((T, Hv))
    A_log = rng.uniform(-1, 1, Hv)
    dt_bias = rng.uniform(-0.5, 0.5, Hv)
    S0 = rng.standard_normal((Hv, Dk, Dv)) * s0_std
    if gate_mode == 1:
        a = -np.abs(a) * 0.5        # log decay <= 0
        b = expit(b)                # beta in (0, 1)
    return dict(qkv=qkv, a=a, b=b, A_log=A_log, dt_bias=dt_bias, S0=S0,
                Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, gate_mode=gate_mode)


def run_oracle(c, mutate="none", eps=1e-6):
    T = c["qkv"].shape[0]
    o, S = oracle.gdn_f64(c["qkv"], c["a"], c["b"], c["A_log"], c["dt_bias"], [0], [T],
                          c["Hk"], c["Hv"], c["Dk"], c["Dv"], S0=c["S0"][None], eps=eps,
                          gate_mode=c["gate_mode"], mutate=mutate)
    return o, S[0]


def run_brute(c, eps=1e-6):
    return brute.gdn_transition(c["qkv"], c["a"], c["b"], c["A_log"], c["dt_bias"],
                                c["Hk"], c["Hv"], c["Dk"], c["Dv"], S0=c["S0"], eps=eps,
                                gate_mode=c["gate_mode"])


# ---------------------------------------------------------------- recurrence

@pytest.mark.parametrize("shape", [(2, 2, 32, 32), (2, 4, 8, 8), (1, 2, 8, 16), (2, 4, 16, 8)])
@pytest.mark.parametrize("gate_mode", [0, 1])
def test_recurrence_matches_transition_product_form(shape, gate_mode):
    Hk, Hv, Dk, Dv = shape
    c = random_case(11 + Hv + Dk, T=7, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, gate_mode=gate_mode)
    o, S = run_oracle(c)
    ob, Sb = run_brute(c)
    assert rel(o, ob) < 1e-12
    assert rel(S, Sb) < 1e-12


def test_tiny_workload_matches_transition_form():
    """The tiny workload end to end: fp32 rows, zero state, 16 tokens."""
    d = synth.tiny()
    sh = d["shapes"]
    y, _ = oracle.conv_f64(d["x"].value, d["hist0"].value, d["conv_w"].value,
                           d["row_start"], d["row_len"])
    o, S = oracle.gdn_f64(y, d["a"].value, d["b"].value, d["A_log"], d["dt_bias"],
                          d["row_start"], d["row_len"], sh.Hk, sh.Hv, sh.Dk, sh.Dv)
    ob, Sb = brute.gdn_transition(y, d["a"].value, d["b"].value, d["A_log"],
                                  d["dt_bias"].astype(np.float64), sh.Hk, sh.Hv, sh.Dk, sh.Dv)
    assert rel(o, ob) < 1e-12 and rel(S[0], Sb) < 1e-12


def test_closed_form_single_token_zero_state():
    """T=1, S0=0: o = scale * beta * (k_hat . q_hat) * v."""
    rng = np.random.default_rng(5)
    Hk, Hv, Dk, Dv = 2, 4, 16, 8
    c = random_case(5, T=1, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    c["S0"][:] = 0.0
    o, S = run_oracle(c)
    q = c["qkv"][0, : Hk * Dk].reshape(Hk, Dk)
    k = c["qkv"][0, Hk * Dk: 2 * Hk * Dk].reshape(Hk, Dk)
    v = c["qkv"][0, 2 * Hk * Dk:].reshape(Hv, Dv)
    for h in range(Hv):
        kh = h // (Hv // Hk)
        qh = q[kh] / math.sqrt(q[kh] @ q[kh] + 1e-6)
        kk = k[kh] / math.sqrt(k[kh] @ k[kh] + 1e-6)
        beta = 1.0 / (1.0 + math.exp(-c["b"][0, h]))
        expect = Dk ** -0.5 * beta * (kk @ qh) * v[h]
        assert np.allclose(o[0, h], expect, rtol=1e-13, atol=1e-15)
        assert np.allclose(S[h], beta * np.outer(kk, v[h]), rtol=1e-13, atol=1e-15)
    del rng


def test_no_decay_no_write_leaves_state_bitwise():
    """A_log = -inf gives g = 0 (no decay); b = -inf gives beta = 0 (no write)."""
    c = random_case(7, T=5, Hk=2, Hv=4, Dk=16, Dv=16)
    c["A_log"][:] = -np.inf
    c["b"][:] = -np.inf
    o, S = run_oracle(c)
    assert np.array_equal(S, c["S0"])
    # the read-out is then scale * S0^T q_hat for every token
    q = c["qkv"][:, : 2 * 16].reshape(5, 2, 16)
    for h in range(4):
        qh = q[:, h // 2] / np.sqrt(np.sum(q[:, h // 2] ** 2, axis=1, keepdims=True) + 1e-6)
        assert np.allclose(o[:, h], 16 ** -0.5 * qh @ c["S0"][h], rtol=1e-13, atol=1e-15)


def test_unit_key_full_write_reads_back_value():
    """beta = 1 and |k| = 1 (eps 0): after the step, S^T k returns v exactly."""
    c = random_case(9, T=1, Hk=1, Hv=2, Dk=16, Dv=8)
    k = c["qkv"][0, 16:32]
    c["qkv"][0, 16:32] = k / np.linalg.norm(k)
    c["b"][:] = np.inf
    o, S = run_oracle(c, eps=0.0)
    kk = c["qkv"][0, 16:32]
    for h in range(2):
        v = c["qkv"][0, 32 + 8 * h: 32 + 8 * (h + 1)]
        assert np.allclose(S[h].T @ kk, v, rtol=1e-12, atol=1e-12)


def test_split_and_carry_is_bitwise():
    """Running T rows at once equals running [0,t) then [t,T) with the state carried."""
    c = random_case(13, T=12, Hk=2, Hv=4, Dk=8, Dv=8)
    o_all, S_all = run_oracle(c)
    for t in (1, 5, 11):
        c1 = dict(c, qkv=c["qkv"][:t], a=c["a"][:t], b=c["b"][:t])
        o1, S1 = run_oracle(c1)
        c2 = dict(c, qkv=c["qkv"][t:], a=c["a"][t:], b=c["b"][t:], S0=S1)
        o2, S2 = run_oracle(c2)
        assert np.array_equal(np.concatenate([o1, o2]), o_all)
        assert np.array_equal(S2, S_all)


def test_state_norm_contraction_bound():
    """|S_t|_F <= alpha_t |S_{t-1}|_F + beta_t |v_t| for every token."""
    c = random_case(17, T=10, Hk=2, Hv=2, Dk=8, Dv=8, s0_std=1.0)
    S_prev = c["S0"]
    for t in range(10):
        ct = dict(c, qkv=c["qkv"][t:t + 1], a=c["a"][t:t + 1], b=c["b"][t:t + 1], S0=S_prev)
        _, S_t = run_oracle(ct)
        for h in range(2):
            alpha = math.exp(-math.exp(c["A_log"][h]) * np.logaddexp(0, c["a"][t, h] + c["dt_bias"][h]))
            beta = expit(c["b"][t, h])
            v = c["qkv"][t, 2 * 2 * 8 + 8 * h: 2 * 2 * 8 + 8 * (h + 1)]
            lhs = np.linalg.norm(S_t[h])
            rhs = alpha * np.linalg.norm(S_prev[h]) + beta * np.linalg.norm(v)
            assert lhs <= rhs * (1 + 1e-12)
        S_prev = S_t


def test_gate_modes_agree():
    """Raw a/b with in-oracle softplus/sigmoid equals precomputed g/beta."""
    c = random_case(19, T=6, Hk=2, Hv=4, Dk=8, Dv=8)
    o0, S0 = run_oracle(c)
    g = -np.exp(c["A_log"])[None] * np.logaddexp(0.0, c["a"] + c["dt_bias"][None])
    c1 = dict(c, a=g, b=expit(c["b"]), gate_mode=1)
    o1, S1 = run_oracle(c1)
    assert rel(o1, o0) < 1e-14 and rel(S1, S0) < 1e-14


def test_requests_are_independent_of_packing():
    """A row map of several requests gives each request's lone result."""
    rng = np.random.default_rng(23)
    Hk, Hv, Dk, Dv = 2, 4, 8, 8
    C = 2 * Hk * Dk + Hv * Dv
    lens = [3, 1, 6]
    order = [2, 0, 1]
    start, ln, T = synth.pack(lens, order)
    qkv = rng.standard_normal((T, C))
    a = rng.standard_normal((T, Hv))
    b = rng.standard_normal((T, Hv))
    A_log = rng.uniform(-1, 1, Hv)
    dt = rng.uniform(-0.5, 0.5, Hv)
    S0 = rng.standard_normal((3, Hv, Dk, Dv))
    o, S = oracle.gdn_f64(qkv, a, b, A_log, dt, start, ln, Hk, Hv, Dk, Dv, S0=S0)
    for r in range(3):
        sl = slice(start[r], start[r] + ln[r])
        ob, Sb = brute.gdn_transition(qkv[sl], a[sl], b[sl], A_log, dt, Hk, Hv, Dk, Dv, S0=S0[r])
        assert rel(o[sl], ob) < 1e-12 and rel(S[r], Sb) < 1e-12


# ---------------------------------------------------------------- chunk form

@pytest.mark.parametrize("T,chunk", [(200, 64), (64, 64), (5, 64), (130, 16)])
def test_chunk_form_equals_token_loop(T, chunk):
    c = random_case(29 + T, T=T, Hk=2, Hv=4, Dk=16, Dv=8)
    o, S = run_oracle(c)
    oc, Sc = brute.gdn_chunked(c["qkv"], c["a"], c["b"], c["A_log"], c["dt_bias"], 2, 4, 16, 8,
                               S0=c["S0"], chunk=chunk)
    assert rel(oc, o) < 1e-10 and rel(Sc, S) < 1e-10


# ---------------------------------------------------------------------- conv

def test_conv_f64_matches_direct_sum():
    rng = np.random.default_rng(31)
    C, W = 24, 4
    lens = [5, 1, 2, 9]
    start, ln, T = synth.pack(lens, [1, 3, 0, 2])
    x = rng.standard_normal((T, C))
    hist = rng.standard_normal((4, W - 1, C))
    w = rng.uniform(-0.5, 0.5, (C, W))
    bias = rng.standard_normal(C)
    y, hout = oracle.conv_f64(x, hist, w, start, ln, bias=bias)
    for r in range(4):
        sl = slice(start[r], start[r] + ln[r])
        yb, hb = brute.conv_direct(x[sl], hist[r], w, bias=bias)
        assert np.allclose(y[sl], yb, rtol=1e-13, atol=1e-14)
        assert np.array_equal(hout[r], hb)


def test_conv_f32_within_fp32_bound_of_f64():
    """fp32 mirror vs fp64: |y32 - y64| <= 8 ulp-of-scale, on bf16 inputs."""
    rng = np.random.default_rng(37)
    C, W, T = 512, 4, 40
    x = synth.as_io(rng.standard_normal((T, C)), synth.BF16).value
    hist = synth.as_io(rng.standard_normal((1, W - 1, C)), synth.BF16).value
    w = synth.as_io(rng.uniform(-0.5, 0.5, (C, W)), synth.BF16).value
    y32, h32 = oracle.conv_f32(x, hist, w, [0], [T])
    y64, h64 = oracle.conv_f64(x, hist, w, [0], [T])
    # bound: accumulation and SiLU each a few fp32 roundings of |terms|
    full = np.concatenate([hist[0], x])
    mag = np.stack([np.sum(np.abs(full[t:t + W].T * w), axis=1) for t in range(T)])
    assert np.all(np.abs(y32 - y64) <= 8 * 2.0 ** -24 * (mag + np.abs(y64)) + 1e-30)
    assert np.array_equal(h32, h64.astype(np.float32))


def test_own_exp_within_one_ulp():
    """The conv's own exp, taken only of arguments a <= 0: within 1 ulp of
    e^a wherever e^a is a normal float (0.90 ulp at worst over every float
    argument), within one subnormal spacing below, and 0 from -104 down
    (e^-104 is under half the smallest subnormal)."""
    xs = np.concatenate([np.linspace(-87.3, 0.0, 20001), np.linspace(-1, 0, 2001),
                         [-0.0, -1e-8, -0.5 * math.log(2), -math.log(2), -87.0]])
    for x in xs.astype(np.float32):
        got = oracle.exp_f32(float(x))
        ref = math.exp(float(x))
        ulp = np.spacing(np.float32(ref))
        assert abs(got - ref) <= ulp, (x, got, ref)
    assert oracle.exp_f32(0.0) == 1.0 and oracle.exp_f32(-0.0) == 1.0
    tiny = 2.0 ** -149
    for x in np.linspace(-103.9, -87.4, 2001).astype(np.float32):
        assert abs(oracle.exp_f32(float(x)) - math.exp(float(x))) <= tiny, x
    for x in (-104.0, -150.0, -1e30, -math.inf):
        assert oracle.exp_f32(x) == 0.0


def test_own_silu_within_four_ulp():
    """SiLU(x) = x sigmoid(x) through the own exp and an IEEE quotient:
    within 4 ulp of the exact value where it is a normal float of at least
    2^-124, and within 2^-140 absolutely below that (x < -87, where e^x is
    subnormal)."""
    xs = np.concatenate([np.linspace(-87, 87, 34801), np.linspace(-1, 1, 4001),
                         [0.0, -0.0, 1e-30, -1e-30, 1e-6, -1e-6, 100.0, 1e30]])
    for x in xs.astype(np.float32):
        got = oracle.silu_f32(float(x))
        ref = float(x) / (1.0 + math.exp(-float(x)))
        assert abs(got - ref) <= 4 * np.spacing(np.float32(abs(ref))) + 1e-45, (x, got, ref)
    for x in np.linspace(-104, -87, 3401).astype(np.float32):
        ref = float(x) * math.exp(float(x)) / (1.0 + math.exp(float(x)))
        assert abs(oracle.silu_f32(float(x)) - ref) <= 2.0 ** -140, x
    assert oracle.silu_f32(-200.0) == 0.0   # an underflowed zero, of either sign
    assert oracle.silu_f32(math.inf) == math.inf
    assert math.isnan(oracle.silu_f32(math.nan))


# ----------------------------------------------------------- slot simulation

def _spec_small(seed, R=3, n=4, steps=5, Hk=1, Hv=2, Dk=8, Dv=8, W=4):
    rng = np.random.default_rng(seed)
    C = 2 * Hk * Dk + Hv * Dv
    p = dict(R=R, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, W=W,
             conv_w=rng.uniform(-0.5, 0.5, (C, W)), A_log=rng.uniform(-1, 1, Hv),
             dt_bias=rng.uniform(-0.5, 0.5, Hv),
             S0=rng.standard_normal((R, Hv, Dk, Dv)) * 0.1,
             hist0=rng.standard_normal((R, W - 1, C)))
    xs = [rng.standard_normal((R, n, C)) for _ in range(steps)]
    As = [rng.standard_normal((R, n, Hv)) for _ in range(steps)]
    Bs = [rng.standard_normal((R, n, Hv)) for _ in range(steps)]
    acc = rng.integers(0, n, size=(steps, R))
    acc[0] = 0
    return p, xs, As, Bs, acc


def _plain(p, r, x, a, b):
    """The plain sequence (conv + recurrence) over rows x of request r."""
    T = x.shape[0]
    y, _ = oracle.conv_f64(x, p["hist0"][r][None], p["conv_w"], [0], [T])
    o, S = oracle.gdn_f64(y, a, b, p["A_log"], p["dt_bias"], [0], [T], p["Hk"], p["Hv"],
                          p["Dk"], p["Dv"], S0=p["S0"][r][None])
    return o, S[0]


def test_slot_sim_equals_rerun_of_accepted_history():
    """Step s candidate i equals a fresh run over the accepted history plus
    candidates 0..i of step s (a different formulation: no slots at all)."""
    p, xs, As, Bs, acc = _spec_small(41)
    sim = oracle.SlotSim(p["R"], p["Hk"], p["Hv"], p["Dk"], p["Dv"], p["W"], p["conv_w"],
                         p["A_log"], p["dt_bias"], S0=p["S0"], hist0=p["hist0"])
    hist_rows = [[] for _ in range(p["R"])]  # accepted rows so far: (x, a, b)
    for s in range(len(xs)):
        _, o = sim.step(xs[s], As[s], Bs[s], acc[s])
        for r in range(p["R"]):
            if s > 0:
                keep = acc[s][r] + 1
                hist_rows[r].append((xs[s - 1][r][:keep], As[s - 1][r][:keep], Bs[s - 1][r][:keep]))
            hx = np.concatenate([h[0] for h in hist_rows[r]] + [xs[s][r]])
            ha = np.concatenate([h[1] for h in hist_rows[r]] + [As[s][r]])
            hb = np.concatenate([h[2] for h in hist_rows[r]] + [Bs[s][r]])
            o_ref, _ = _plain(p, r, hx, ha, hb)
            n = xs[s].shape[1]
            assert rel(o[r], o_ref[-n:]) < 1e-12
    # the state resumed from the last accepted slot is the accepted-history state
    last = np.array([1, 3, 2])
    for r in range(p["R"]):
        hx = np.concatenate([h[0] for h in hist_rows[r]] + [xs[-1][r][: last[r] + 1]])
        ha = np.concatenate([h[1] for h in hist_rows[r]] + [As[-1][r][: last[r] + 1]])
        hb = np.concatenate([h[2] for h in hist_rows[r]] + [Bs[-1][r][: last[r] + 1]])
        _, S_ref = _plain(p, r, hx, ha, hb)
        assert rel(sim.state(r, last[r]), S_ref) < 1e-12


def test_slot_sim_accept_all_is_plain_sequence():
    p, xs, As, Bs, _ = _spec_small(43, steps=3)
    n = xs[0].shape[1]
    sim = oracle.SlotSim(p["R"], p["Hk"], p["Hv"], p["Dk"], p["Dv"], p["W"], p["conv_w"],
                         p["A_log"], p["dt_bias"], S0=p["S0"], hist0=p["hist0"])
    outs = []
    for s in range(3):
        _, o = sim.step(xs[s], As[s], Bs[s], np.full(p["R"], 0 if s == 0 else n - 1))
        outs.append(o)
    for r in range(p["R"]):
        o_ref, S_ref = _plain(p, r, np.concatenate([x[r] for x in xs]),
                              np.concatenate([a[r] for a in As]), np.concatenate([b[r] for b in Bs]))
        assert rel(np.concatenate([o[r] for o in outs]), o_ref) < 1e-12
        assert rel(sim.state(r, n - 1), S_ref) < 1e-12


def test_round_bf16_ties_and_values():
    """bf16 keeps 8 significant bits: the spacing at 1.0 is 2^-7."""
    vals = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1.005, 1.003, -3.14159, 0.0])
    out = oracle.round_bf16(vals)
    assert out[0] == 1.0
    assert out[1] == 1.0                  # tie between 1 and 1+2^-7: to even
    assert out[2] == 1 + 2.0 ** -6        # tie between 1+2^-7 and 1+2^-6: to even
    assert out[3] == 1 + 2.0 ** -7        # above half a spacing
    assert out[4] == 1.0                  # below half a spacing
    assert out[5] == -3.140625
    assert out[6] == 0.0
    assert np.array_equal(oracle.round_bf16(out), out)


# ------------------------------------------------------------------ mutants

@pytest.mark.parametrize("mutation", [m for m in oracle.MUTATIONS if m != "none"])
def test_planted_mistakes_fail_a_pin(mutation):
    """Each planted mistake in the oracle fails the product-form pin."""
    c = random_case(47, T=6, Hk=2, Hv=4, Dk=8, Dv=8)
    ob, Sb = run_brute(c)
    o, S = run_oracle(c, mutate=mutation)
    assert max(rel(o, ob), rel(S, Sb)) > 1e-3
    o0, S0 = run_oracle(c)
    assert max(rel(o0, ob), rel(S0, Sb)) < 1e-12
