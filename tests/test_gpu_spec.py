"""Speculative-decode verify with one page per request.

* bit-identical to the slot-per-candidate layout (gdn_spec_slots) under
  random acceptance, over 20 steps, with fp32 and bf16 state pages;
* within 1e-4 of the fp64 slot simulation of the oracle (fp32 state);
* the fused step (gdn_spec_step: conv + verify in one launch) equals
  gdn_conv + gdn_spec_verify bit for bit, pages included, and the slots;
* identical requests in lockstep equal the same request alone;
* commit closes the record and plain rows continue from it;
* a mixed step (prefills + spec requests, one conv launch) through a row map;
* device-side error codes leave the offending page untouched.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import oracle
import synth
from tests.gpu_util import CHUNK_ELEM_C, Layer, assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu

SPEC = gdn.GDN_REQ_SPEC
PAR = gdn.GDN_REQ_PARITY
TOL = 1e-4


def spec_flags(step, R):
    return np.full(R, SPEC | (PAR if step % 2 else 0), np.int64)


def make_layers(d, R, state, slots=True, Kc=8):
    sh = d["shapes"]
    L1 = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=Kc, state=state,
               num_pages=R)
    L2 = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=Kc, state=state,
               num_pages=R, slots=slots) if slots else None
    hist = to_dev(d["hist0"])[:R]
    S0 = d["S0"][:R]
    if state == gdn.GDN_BF16:
        S0 = oracle.round_bf16(S0).astype(np.float32)
    L1.seed(range(R), S0=S0, hist=hist)
    if L2 is not None:
        for r in range(R):
            L2.slots.state(r, 0).copy_(torch.from_numpy(S0[r]).transpose(-1, -2))
            L2.slots.window(r, 0).copy_(hist[r])
    return L1, L2, S0


def one_page_step(L, start, ln, flags, acc, x, a, b):
    B = L.batch(start, ln, flags=flags, n_accepted=acc)
    y = L.conv(B, x)
    o = L.verify(B, y, a, b)
    return y, o


def step_rows(d, s, R, n):
    rows = d["step_rows"][s]
    sl = slice(0, R * n)
    return to_dev(rows["x"])[sl], to_dev(rows["a"])[sl], to_dev(rows["b"])[sl]


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_one_page_bit_identical_to_slot_layout_20_steps(state):
    d = synth.spec()
    R, n, steps = d["R"], d["n"], d["steps"]
    start, ln = d["row_start"], d["row_len"]
    L1, L2, _ = make_layers(d, R, state)
    for s in range(steps):
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s]
        y1, o1 = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        B2 = L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
        y2, o2 = L2.spec_slots(B2, x, a, b)
        L1.ok()
        L2.ok()
        assert np.array_equal(bits(y1), bits(y2)), f"conv rows differ at step {s}"
        assert np.array_equal(bits(o1), bits(o2)), f"outputs differ at step {s}"
    # commit the last step's acceptance and compare the checkpoint with the slot
    acc = d["accepted"][steps]
    zero = np.zeros(R, np.int32)
    B = L1.batch(start, zero, flags=spec_flags(steps, R), n_accepted=acc, num_rows=int(start[-1]) + n)
    L1.conv(B, x)
    L1.verify(B, y1, a, b)
    L1.ok()
    for r in range(R):
        assert np.array_equal(bits(L1.pool.state(r)), bits(L2.slots.state(r, int(acc[r]))))
        assert np.array_equal(bits(L1.pool.window(r)[:3]), bits(L2.slots.window(r, int(acc[r]))))
        assert int(L1.pool.flag(r).item()) & 0xFC == 0     # record closed (width 0)


def test_one_page_matches_oracle_slot_simulation():
    d = synth.spec()
    R_all, n = d["R"], d["n"]
    R, steps = 4, 6
    sh = d["shapes"]
    start, ln = d["row_start"][:R], d["row_len"][:R]
    L1, _, S0 = make_layers(d, R, gdn.GDN_F32, slots=False)
    sim = oracle.SlotSim(R, sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, d["conv_w"].value, d["A_log"],
                         d["dt_bias"], S0=S0, hist0=d["hist0"].value[:R],
                         row_store=oracle.round_bf16)
    for s in range(steps):
        rows = d["step_rows"][s]
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s][:R]
        y, o = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        L1.ok()
        xs = rows["x"].value[: R * n].reshape(R, n, -1)
        As = rows["a"].value[: R * n].reshape(R, n, -1)
        Bs = rows["b"].value[: R * n].reshape(R, n, -1)
        y_ref, o_ref = sim.step(xs, As, Bs, acc)
        # the conv'd rows are bit-exact against the fp32 mirror
        assert np.array_equal(bits(y), synth.bf16_bits(y_ref.reshape(R * n, -1)).view(np.int16))
        assert_close(f64(o), o_ref.reshape(R * n, sh.Hv, sh.Dv), TOL, what=f"o step {s}")
    del R_all


def test_lockstep_identical_requests_equal_request_alone():
    d = synth.spec(R=8, steps=5)
    n, steps = d["n"], d["steps"]
    twin = [1, 3, 4, 6]
    # requests in `twin` are copies of request 1: same rows, state, window, acceptance
    for s in range(steps):
        for k in ("x", "a", "b"):
            t = d["step_rows"][s][k]
            st = t.store.reshape(8, n, -1)
            st[twin] = st[1]
            t.store[:] = st.reshape(t.store.shape)
        d["accepted"][s][twin] = d["accepted"][s][1]
    d["S0"][twin] = d["S0"][1]
    d["hist0"].store[twin] = d["hist0"].store[1]
    d["hist0"].value[twin] = d["hist0"].value[1]
    start, ln = d["row_start"], d["row_len"]
    L, _, _ = make_layers(d, 8, gdn.GDN_F32, slots=False)
    # the same request alone, as request 0 of a batch of one, on page 0
    d1 = dict(d)
    d1["S0"] = d["S0"][1:2]
    h1 = synth.Tensor(d["hist0"].store[1:2], d["hist0"].value[1:2], d["hist0"].dtype)
    d1["hist0"] = h1
    La, _, _ = make_layers(d1, 1, gdn.GDN_F32, slots=False)
    for s in range(steps):
        x, a, b = step_rows(d, s, 8, n)
        _, o = one_page_step(L, start, ln, spec_flags(s, 8), d["accepted"][s], x, a, b)
        _, oa = one_page_step(La, [0], [n], spec_flags(s, 1), d["accepted"][s][1:2],
                              x[n:2 * n], a[n:2 * n], b[n:2 * n])
        L.ok()
        La.ok()
        for r in twin:
            assert np.array_equal(bits(o[r * n:(r + 1) * n]), bits(oa))


def test_commit_then_plain_decode_continues():
    """Commit (zero new candidates) closes the record; plain rows then run
    from the committed state, and plain rows on an open record are refused."""
    d = synth.spec(R=2, steps=2)
    sh, n = d["shapes"], d["n"]
    start, ln = d["row_start"], d["row_len"]
    L, _, S0 = make_layers(d, 2, gdn.GDN_F32, slots=False)
    x, a, b = step_rows(d, 0, 2, n)
    one_page_step(L, start, ln, spec_flags(0, 2), d["accepted"][0], x, a, b)
    L.ok()
    # plain rows while the record is open: refused, page untouched
    before = L.pool.buf.clone()
    rng = np.random.default_rng(5)
    rows = synth.rows(rng, 2, sh, synth.BF16)
    xp, ap, bp = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
    Bp = L.batch([0, 1], [1, 1])
    L.conv(Bp, xp)
    assert L.status_code() == gdn.CODES["GDN_DEV_RECORD_OPEN"]
    L.reset_status()
    L.seq(Bp, xp, ap, bp)
    assert L.status_code() == gdn.CODES["GDN_DEV_RECORD_OPEN"]
    L.reset_status()
    assert torch.equal(before, L.pool.buf)
    # commit with acceptance [2, 5]
    acc = np.array([2, 5], np.int32)
    Bc = L.batch(start, [0, 0], flags=spec_flags(1, 2), n_accepted=acc, num_rows=2 * n)
    L.conv(Bc, x)
    L.verify(Bc, x, a, b)
    L.ok()
    # then one plain decode token through conv + rule
    y = L.conv(Bp, xp)
    o = L.seq(Bp, y, ap, bp)
    L.ok()
    # oracle: accepted history (rows 0..acc of step 0) then the decode row
    for r in range(2):
        xs = np.concatenate([d["step_rows"][0]["x"].value[r * n: r * n + acc[r] + 1],
                             rows["x"].value[r:r + 1]])
        As = np.concatenate([d["step_rows"][0]["a"].value[r * n: r * n + acc[r] + 1],
                             rows["a"].value[r:r + 1]])
        Bs = np.concatenate([d["step_rows"][0]["b"].value[r * n: r * n + acc[r] + 1],
                             rows["b"].value[r:r + 1]])
        yy, _ = oracle.conv_f32(xs, d["hist0"].value[r:r + 1], d["conv_w"].value, [0], [len(xs)])
        yy = oracle.round_bf16(yy)
        o_ref, S_ref = oracle.gdn_f64(yy, As, Bs, d["A_log"], d["dt_bias"], [0], [len(xs)],
                                      sh.Hk, sh.Hv, sh.Dk, sh.Dv, S0=S0[r:r + 1])
        assert_close(f64(o[r]), o_ref[-1], TOL, what=f"o request {r}")
        assert_close(f64(L.pool.state_math(r)), S_ref[0], TOL, inner=2, what=f"S request {r}")


@pytest.mark.parametrize("prefill_entry", ["seq", "prefill", "prefill_ws"])
def test_mixed_prefill_and_spec_step_through_row_map(prefill_entry):
    """gdn_seq, or gdn_prefill (prefills of 64+ rows take the chunked form: one
    launch, or with a workspace two passes), for the plain rows of a step that
    also verifies spec requests, through a row map with a processing order."""
    for shuffled in (False, True):
        d = synth.mixed(shuffled=shuffled)
        sh, n, ns, npf = d["shapes"], d["n"], d["n_spec"], d["n_prefill"]
        R = d["R"]
        L = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R)
        spec = d["is_spec"]
        S0 = d["S0"]
        L.seed(range(R), S0=S0, hist=to_dev(d["hist0"]))
        # one earlier spec step seeds the spec requests' records
        pr = d["prev_rows"]
        st0, ln0, _ = synth.pack([n] * ns)
        one_page_step(L, st0, ln0, spec_flags(0, ns), np.zeros(ns, np.int32), to_dev(pr["x"]),
                      to_dev(pr["a"]), to_dev(pr["b"]))
        L.ok()
        # the mixed step: one conv launch over every row, then rule + verify
        flags = np.where(spec, SPEC | PAR, gdn.GDN_REQ_FRESH)
        acc = np.where(spec, np.concatenate([d["prev_accepted"], np.zeros(npf, np.int32)]), 0)
        lengths = d["row_len"]
        order = np.argsort(-lengths, kind="stable")
        B = L.batch(d["row_start"], lengths, flags=flags, n_accepted=acc, order=order)
        x, a, b = to_dev(d["x"]), to_dev(d["a"]), to_dev(d["b"])
        y = L.conv(B, x)
        o = L.seq(B, y, a, b) if prefill_entry == "seq" else \
            L.prefill(B, y, a, b, workspace=(prefill_entry == "prefill_ws"))
        o2 = L.verify(B, y, a, b)
        L.ok()
        row_is_spec = np.zeros(d["T"], bool)
        for r in range(R):
            row_is_spec[d["row_start"][r]: d["row_start"][r] + lengths[r]] = spec[r]
        o = torch.where(torch.from_numpy(row_is_spec).cuda()[:, None, None], o2, o)
        # prefills: fp32 conv mirror from a zero window, bf16 rows, fp64 rule
        # (every prefill on the dispatching entry point: both forms run)
        for r in np.nonzero(~spec)[0][: (3 if prefill_entry == "seq" else npf)]:
            sl = slice(d["row_start"][r], d["row_start"][r] + lengths[r])
            yy, _ = oracle.conv_f32(d["x"].value[sl], np.zeros((1, 3, sh.C)), d["conv_w"].value,
                                    [0], [lengths[r]])
            o_ref, S_ref = oracle.gdn_f64(oracle.round_bf16(yy), d["a"].value[sl],
                                          d["b"].value[sl], d["A_log"], d["dt_bias"], [0],
                                          [lengths[r]], sh.Hk, sh.Hv, sh.Dk, sh.Dv)
            # gdn_prefill sends prompts of 64+ rows through the chunked form
            c = CHUNK_ELEM_C if prefill_entry != "seq" else 1.0
            assert_close(f64(o[sl]), o_ref, TOL, what=f"o prefill {r}", c=c)
            assert_close(f64(L.pool.state_math(r)), S_ref[0], TOL, inner=2,
                         what=f"S prefill {r}", c=c)
        # spec requests: the oracle's slot simulation over both steps
        k = 3
        sim = oracle.SlotSim(k, sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, d["conv_w"].value, d["A_log"],
                             d["dt_bias"], S0=S0[:k], hist0=d["hist0"].value[:k],
                             row_store=oracle.round_bf16)
        sim.step(pr["x"].value[:k * n].reshape(k, n, -1), pr["a"].value[:k * n].reshape(k, n, -1),
                 pr["b"].value[:k * n].reshape(k, n, -1), np.zeros(k, np.int32))
        xs = np.stack([d["x"].value[d["row_start"][r]: d["row_start"][r] + n] for r in range(k)])
        As = np.stack([d["a"].value[d["row_start"][r]: d["row_start"][r] + n] for r in range(k)])
        Bs = np.stack([d["b"].value[d["row_start"][r]: d["row_start"][r] + n] for r in range(k)])
        _, o_ref = sim.step(xs, As, Bs, d["prev_accepted"][:k])
        for r in range(k):
            sl = slice(d["row_start"][r], d["row_start"][r] + n)
            assert_close(f64(o[sl]), o_ref[r], TOL, what=f"o spec {r}")


def _at_step_one(d):
    """Four spec pages after one verify step (record width 8, parity 1)."""
    L, _, _ = make_layers(d, 4, gdn.GDN_F32, slots=False)
    x, a, b = step_rows(d, 0, 4, d["n"])
    one_page_step(L, d["row_start"], d["row_len"], spec_flags(0, 4), d["accepted"][0], x, a, b)
    L.ok()
    return L


def _page(L, p):
    lay = L.pool.layout
    return L.pool.buf[p * lay.page_bytes:(p + 1) * lay.page_bytes].clone()


@pytest.mark.parametrize("name", ["GDN_DEV_STALE_STEP", "GDN_DEV_BAD_ACCEPTED",
                                  "GDN_DEV_BAD_FLAG"])
def test_device_errors_skip_only_the_offending_request(name):
    d = synth.spec(R=4, steps=2)
    n = d["n"]
    start, ln = d["row_start"], d["row_len"]
    L = _at_step_one(d)
    x, a, b = step_rows(d, 1, 4, n)
    flags = spec_flags(1, 4)
    acc = d["accepted"][1].copy()
    if name == "GDN_DEV_STALE_STEP":
        flags[2] = SPEC                      # parity 0, the page expects 1
    elif name == "GDN_DEV_BAD_ACCEPTED":
        acc[2] = 8                           # the record holds 8 rows: 0..7
    else:
        flags[2] |= gdn.GDN_REQ_FRESH        # FRESH together with SPEC
    before = _page(L, 2)
    others = [_page(L, p) for p in (0, 1, 3)]
    B = L.batch(start, ln, flags=flags, n_accepted=acc)
    y = L.conv(B, x)
    assert L.status_code() == gdn.CODES[name]
    L.verify(B, y, a, b)
    assert L.status_code() == gdn.CODES[name]
    assert torch.equal(before, _page(L, 2))
    # the other requests completed their step
    for p, old in zip((0, 1, 3), others):
        assert not torch.equal(old, _page(L, p))
        assert (int(L.pool.flag(p).item()) >> 1) & 1 == 0      # parity advanced to 0


def test_device_errors_page_index_and_candidate_count():
    d = synth.spec(R=4, steps=2)
    n = d["n"]
    start, ln = d["row_start"], d["row_len"]
    L = _at_step_one(d)
    x, a, b = step_rows(d, 1, 4, n)
    B = L.batch(start, ln, flags=spec_flags(1, 4), n_accepted=d["accepted"][1], page=[0, 1, 7, 3])
    L.conv(B, x)
    assert L.status_code() == gdn.CODES["GDN_DEV_BAD_PAGE"]
    L.reset_status()
    # 9 candidates for request 0 (rows 0..8 exist: request 1 starts at row 8)
    lens = ln.copy()
    lens[0] = 9
    B = L.batch(start, lens, flags=spec_flags(1, 4), n_accepted=d["accepted"][1])
    L.conv(B, x)
    assert L.status_code() == gdn.CODES["GDN_DEV_TOO_MANY_CANDIDATES"]
    L.reset_status()
    L.verify(B, x, a, b)
    assert L.status_code() == gdn.CODES["GDN_DEV_TOO_MANY_CANDIDATES"]


# (Hk, Hv, Dk): GQA groups of 1, 3 and 8 value heads per q/k head, and the
# three supported head dimensions (one, two or four 32-column blocks per head)
OTHER_SHAPES = [(2, 2, 32), (2, 6, 32), (2, 6, 64), (1, 8, 128)]


def _ragged_vs_slots(sh, io, seed, Kc=8, R=6, steps=5, state=gdn.GDN_F32):
    """1..Kc candidates per request and step, packed in a shuffled row order:
    outputs and the committed state stay bit-identical to the slot layout."""
    rng = np.random.default_rng(seed)
    d = synth.spec(seed=int(rng.integers(1 << 30)), R=R, steps=1, n=1, sh=sh, io=io)
    L1, L2, _ = make_layers(d, R, state, Kc=Kc)
    prev_len = np.zeros(R, np.int64)
    for s in range(steps):
        ln = rng.integers(1, Kc + 1, size=R)
        order = rng.permutation(R)
        start, _, T = synth.pack(ln, order)
        rows = synth.rows(rng, T, sh, io)
        x, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
        acc = np.where(prev_len > 0, rng.integers(0, np.maximum(prev_len, 1)), 0).astype(np.int32)
        flags = spec_flags(s, R)
        B1 = L1.batch(start, ln, flags=flags, n_accepted=acc, max_rows=Kc)
        y1 = L1.conv(B1, x)
        o1 = L1.verify(B1, y1, a, b)
        B2 = L2.batch(start, ln, flags=flags, n_accepted=acc, max_rows=Kc)
        y2, o2 = L2.spec_slots(B2, x, a, b)
        L1.ok()
        L2.ok()
        assert np.array_equal(bits(y1), bits(y2)), f"conv rows differ at step {s}"
        assert np.array_equal(bits(o1), bits(o2)), f"outputs differ at step {s}"
        prev_len = ln
    acc = rng.integers(0, prev_len).astype(np.int32)
    zero = np.zeros(R, np.int32)
    B = L1.batch(np.zeros(R, np.int32), zero, flags=spec_flags(steps, R), n_accepted=acc,
                 num_rows=1)
    L1.conv(B, x)
    L1.verify(B, y1, a, b)
    L1.ok()
    for r in range(R):
        assert np.array_equal(bits(L1.pool.state(r)), bits(L2.slots.state(r, int(acc[r]))))


@pytest.mark.parametrize("io", [synth.BF16, synth.F32])
@pytest.mark.parametrize("hk,hv,dk", OTHER_SHAPES)
def test_one_page_bit_identical_to_slots_other_shapes_ragged(hk, hv, dk, io):
    _ragged_vs_slots(synth.Shapes(Hk=hk, Hv=hv, Dk=dk, Dv=dk), io,
                     100 + hk * 1000 + hv * 10 + dk)


@pytest.mark.parametrize("hk,hv,dk", OTHER_SHAPES)
def test_one_page_bit_identical_to_slots_other_shapes_bf16_state(hk, hv, dk):
    _ragged_vs_slots(synth.Shapes(Hk=hk, Hv=hv, Dk=dk, Dv=dk), synth.BF16,
                     200 + hk * 1000 + hv * 10 + dk, state=gdn.GDN_BF16)


def test_wide_group_verify_bit_identical_to_slots_step_refused():
    """32 value heads on one q/k head at Dk = Dv = 128: the one-page verify
    (bounded only by its own kernels) stays bit-identical to the slot layout,
    and the one-launch step, whose CTA stages the whole group's rows and u,
    refuses the shape on the host with GDN_ERR_UNSUPPORTED."""
    sh = synth.Shapes(Hk=1, Hv=32, Dk=128, Dv=128)
    _ragged_vs_slots(sh, synth.BF16, 4242, R=3, steps=3)
    d = synth.spec(seed=1, R=2, steps=1, n=1, sh=sh, io=synth.BF16)
    L, _, _ = make_layers(d, 2, gdn.GDN_F32, slots=False)
    rows = synth.rows(np.random.default_rng(0), 2, sh, synth.BF16)
    B = L.batch(np.arange(2, dtype=np.int32), np.ones(2, np.int32), flags=spec_flags(0, 2),
                n_accepted=np.zeros(2, np.int32), max_rows=1)
    with pytest.raises(gdn.GdnError) as e:
        L.spec_step(B, to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"]))
    assert e.value.code == gdn.CODES["GDN_ERR_UNSUPPORTED"]
    L.ok()


@pytest.mark.parametrize("Kc", [1, 3])
def test_one_page_bit_identical_to_slots_small_record(Kc):
    """A record of 1 row (no drafts: every step verifies one token, so the
    replay is always row 0) or 3 rows; the window then holds 3 + Kc columns."""
    _ragged_vs_slots(synth.Shapes(Hk=2, Hv=4, Dk=64, Dv=64), synth.BF16, 7 + Kc, Kc=Kc)


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_switch_to_slot_layout_midstream(state):
    """Prefix caching keeps the stock per-candidate pages (r9700-stack v0.2.4,
    "What it does"): a request that ran one-page steps is committed, handed to
    slot 0 of a slot pool by gdn_page_to_slots, and the slot layout continues
    from there, bit-identical to a request that used the slot layout from the
    start."""
    d = synth.spec(R=4, steps=4)
    R, n = 4, d["n"]
    start, ln = d["row_start"][:R], d["row_len"][:R]
    L1, L2, _ = make_layers(d, R, state)          # one-page; slots from the start
    for s in range(2):
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s][:R]
        one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        L2.spec_slots(L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc), x, a, b)
        L1.ok()
        L2.ok()
    # commit the one-page request, then hand its page to a fresh slot pool
    acc = d["accepted"][2][:R]
    zero = np.zeros(R, np.int32)
    B = L1.batch(start, zero, flags=spec_flags(2, R), n_accepted=acc, num_rows=int(start[-1]) + n)
    L1.conv(B, x)
    L1.verify(B, x, a, b)
    L1.ok()
    L3 = Layer(d["shapes"], d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, state=state,
               num_pages=R, slots=True)
    idx = to_dev(np.arange(R, dtype=np.int32))
    gdn.gdn_page_to_slots(L1.dims, R, idx, idx, R, R, L1.pool.buf, L3.slots.buf, L3.status)
    L3.ok()
    for r in range(R):
        assert torch.equal(L3.slots.state(r, 0), L1.pool.state(r))
        assert torch.equal(L3.slots.window(r, 0), L1.pool.window(r)[:3])
    x, a, b = step_rows(d, 2, R, n)
    y2, o2 = L2.spec_slots(L2.batch(start, ln, flags=spec_flags(2, R), n_accepted=acc), x, a, b)
    y3, o3 = L3.spec_slots(L3.batch(start, ln, flags=spec_flags(2, R), n_accepted=zero), x, a, b)
    L2.ok()
    L3.ok()
    assert np.array_equal(bits(y2), bits(y3))
    assert np.array_equal(bits(o2), bits(o3))
    for r in range(R):
        for i in range(n):
            assert np.array_equal(bits(L2.slots.state(r, i)), bits(L3.slots.state(r, i)))


def test_one_page_bit_identical_to_slots_gate_mode_precomputed():
    """Precomputed gates (a = g <= 0, b = beta in [0, 1]): the record carries
    them as given and the replay reads them back, so the one-page verify
    still equals the slot layout bit for bit over several steps."""
    d = synth.spec(R=8, steps=5)
    R, n, steps = d["R"], d["n"], d["steps"]
    sh = d["shapes"]
    rng = np.random.default_rng(12)
    start, ln = d["row_start"][:R], d["row_len"][:R]
    L1 = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R,
               gate_mode=1)
    L2 = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R,
               slots=True, gate_mode=1)
    hist = to_dev(d["hist0"])[:R]
    S0 = d["S0"][:R]
    L1.seed(range(R), S0=S0, hist=hist)
    for r in range(R):
        L2.slots.state(r, 0).copy_(torch.from_numpy(S0[r]).transpose(-1, -2))
        L2.slots.window(r, 0).copy_(hist[r])
    for s in range(steps):
        x = to_dev(d["step_rows"][s]["x"])[: R * n]
        g = synth.as_io(-np.abs(rng.standard_normal((R * n, sh.Hv))) * 0.7, synth.BF16)
        beta = synth.as_io(rng.uniform(0, 1, (R * n, sh.Hv)), synth.BF16)
        a, b = to_dev(g), to_dev(beta)
        acc = d["accepted"][s][:R]
        _, o1 = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        B2 = L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
        _, o2 = L2.spec_slots(B2, x, a, b)
        L1.ok()
        L2.ok()
        assert np.array_equal(bits(o1), bits(o2)), f"outputs differ at step {s}"


def test_bench_configuration_bf16_outputs_vs_slots_and_oracle():
    """The configuration the benchmark times: 64 pages x (1+7) candidates,
    fp32 state, bf16 rows and bf16 outputs. Bit-identical to the slot layout
    over 5 steps; for 4 of the requests, each output is the oracle's slot
    simulation rounded to bf16 or its neighbour (the fp32 result sits
    within 1e-4 of the oracle, so it can cross a rounding boundary)."""
    d = synth.spec()
    R, n = d["R"], d["n"]
    steps = 5
    sh = d["shapes"]
    start, ln = d["row_start"], d["row_len"]
    L1 = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R,
               out=gdn.GDN_BF16)
    L2 = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R,
               out=gdn.GDN_BF16, slots=True)
    hist = to_dev(d["hist0"])[:R]
    S0 = d["S0"][:R]
    L1.seed(range(R), S0=S0, hist=hist)
    for r in range(R):
        L2.slots.state(r, 0).copy_(torch.from_numpy(S0[r]).transpose(-1, -2))
        L2.slots.window(r, 0).copy_(hist[r])
    k = 4
    sim = oracle.SlotSim(k, sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, d["conv_w"].value, d["A_log"],
                         d["dt_bias"], S0=S0[:k], hist0=d["hist0"].value[:k],
                         row_store=oracle.round_bf16)
    for s in range(steps):
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s]
        _, o1 = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        B2 = L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
        _, o2 = L2.spec_slots(B2, x, a, b)
        L1.ok()
        L2.ok()
        assert np.array_equal(bits(o1), bits(o2)), f"outputs differ at step {s}"
        rows = d["step_rows"][s]
        xs = rows["x"].value[: k * n].reshape(k, n, -1)
        As = rows["a"].value[: k * n].reshape(k, n, -1)
        Bs = rows["b"].value[: k * n].reshape(k, n, -1)
        _, o_ref = sim.step(xs, As, Bs, acc[:k])
        o_ref = o_ref.reshape(k * n, sh.Hv, sh.Dv)
        got = f64(o1)[: k * n]
        ref_round = oracle.round_bf16(o_ref)
        spacing = np.spacing(np.abs(ref_round).astype(np.float32)).astype(np.float64) * 2.0 ** 16
        rms = np.sqrt(np.mean(o_ref ** 2))
        assert np.all(np.abs(got - o_ref) <= spacing + 1e-4 * rms), f"step {s}"
        assert np.mean(got != ref_round) < 0.05


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_fused_step_bit_identical_to_conv_verify_and_slots_20_steps(state):
    """gdn_spec_step over the 64-page benchmark batch for 20 steps: outputs
    and whole pages (state, window, record, flag) bit-identical to gdn_conv +
    gdn_spec_verify, outputs bit-identical to the slot layout, and after the
    final commit the checkpoints equal the accepted slots."""
    d = synth.spec()
    R, n, steps = d["R"], d["n"], d["steps"]
    start, ln = d["row_start"], d["row_len"]
    L1, L2, _ = make_layers(d, R, state)
    L3, _, _ = make_layers(d, R, state, slots=False)
    for s in range(steps):
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s]
        _, o1 = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        B3 = L3.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
        o3 = L3.spec_step(B3, x, a, b)
        B2 = L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
        _, o2 = L2.spec_slots(B2, x, a, b)
        L1.ok()
        L2.ok()
        L3.ok()
        assert np.array_equal(bits(o3), bits(o1)), f"fused outputs differ at step {s}"
        assert np.array_equal(bits(o3), bits(o2)), f"fused vs slots outputs differ at step {s}"
        assert torch.equal(L3.pool.buf, L1.pool.buf), f"pages differ at step {s}"
    acc = d["accepted"][steps]
    zero = np.zeros(R, np.int32)
    B = L3.batch(start, zero, flags=spec_flags(steps, R), n_accepted=acc,
                 num_rows=int(start[-1]) + n)
    L3.spec_step(B, x, a, b)
    L3.ok()
    for r in range(R):
        assert np.array_equal(bits(L3.pool.state(r)), bits(L2.slots.state(r, int(acc[r]))))
        assert np.array_equal(bits(L3.pool.window(r)[:3]), bits(L2.slots.window(r, int(acc[r]))))
        assert int(L3.pool.flag(r).item()) & 0xFC == 0


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_fused_and_two_launch_steps_alternate_on_the_same_pages(state):
    """A step's record (the candidates' rows, run coefficients and u) is what
    the next step's replay reads, whichever entry wrote it: the same pages
    driven by gdn_spec_step on even steps and gdn_conv + gdn_spec_verify on
    odd ones, over 12 steps and a final commit, give outputs bit-identical to
    the slot layout at every step and checkpoints equal to the accepted
    slots."""
    d = synth.spec()
    R, n, steps = d["R"], d["n"], 12
    start, ln = d["row_start"], d["row_len"]
    L1, L2, _ = make_layers(d, R, state)
    for s in range(steps):
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s]
        if s % 2 == 0:
            B1 = L1.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
            o1 = L1.spec_step(B1, x, a, b)
        else:
            _, o1 = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        B2 = L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc)
        _, o2 = L2.spec_slots(B2, x, a, b)
        L1.ok()
        L2.ok()
        assert np.array_equal(bits(o1), bits(o2)), f"outputs differ from the slots at step {s}"
    acc = d["accepted"][steps]
    zero = np.zeros(R, np.int32)
    B = L1.batch(start, zero, flags=spec_flags(steps, R), n_accepted=acc,
                 num_rows=int(start[-1]) + n)
    L1.verify(B, x, a, b)   # the commit: replay, checkpoint, close the record
    L1.ok()
    for r in range(R):
        assert np.array_equal(bits(L1.pool.state(r)), bits(L2.slots.state(r, int(acc[r]))))


@pytest.mark.parametrize("io,state", [(synth.BF16, gdn.GDN_F32), (synth.F32, gdn.GDN_F32),
                                      (synth.BF16, gdn.GDN_BF16)])
@pytest.mark.parametrize("hk,hv,dk", OTHER_SHAPES)
def test_fused_step_equals_conv_verify_other_shapes_ragged(hk, hv, dk, io, state):
    """1..8 candidates per request and step in a shuffled row order, the
    three head dimensions and groups of 1, 3 and 8 value heads, fp32 and
    bf16 state: gdn_spec_step leaves every page and output exactly as
    gdn_conv + gdn_spec_verify."""
    _fused_vs_conv_verify(synth.Shapes(Hk=hk, Hv=hv, Dk=dk, Dv=dk), io, state,
                          300 + hk * 1000 + hv * 10 + dk)


@pytest.mark.parametrize("Kc", [1, 3])
def test_fused_step_equals_conv_verify_small_record(Kc):
    """Records of 1 and 3 rows (the window then holds 3 + Kc columns)."""
    _fused_vs_conv_verify(synth.Shapes(Hk=2, Hv=4, Dk=64, Dv=64), synth.BF16, gdn.GDN_F32,
                          900 + Kc, Kc=Kc)


def _fused_vs_conv_verify(sh, io, state, seed, Kc=8):
    rng = np.random.default_rng(seed)
    R, steps = 6, 5
    d = synth.spec(seed=int(rng.integers(1 << 30)), R=R, steps=1, n=1, sh=sh, io=io)
    L1, _, _ = make_layers(d, R, state, slots=False, Kc=Kc)
    L3, _, _ = make_layers(d, R, state, slots=False, Kc=Kc)
    prev_len = np.zeros(R, np.int64)
    for s in range(steps):
        ln = rng.integers(1, Kc + 1, size=R)
        order = rng.permutation(R)
        start, _, T = synth.pack(ln, order)
        rows = synth.rows(rng, T, sh, io)
        x, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
        acc = np.where(prev_len > 0, rng.integers(0, np.maximum(prev_len, 1)), 0).astype(np.int32)
        flags = spec_flags(s, R)
        B1 = L1.batch(start, ln, flags=flags, n_accepted=acc, max_rows=Kc)
        o1 = L1.verify(B1, L1.conv(B1, x), a, b)
        B3 = L3.batch(start, ln, flags=flags, n_accepted=acc, max_rows=Kc)
        o3 = L3.spec_step(B3, x, a, b)
        L1.ok()
        L3.ok()
        assert np.array_equal(bits(o3), bits(o1)), f"outputs differ at step {s}"
        assert torch.equal(L3.pool.buf, L1.pool.buf), f"pages differ at step {s}"
        prev_len = ln


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_fused_step_bf16_outputs_and_gate_modes(gate_mode):
    """gdn_spec_step with bf16 outputs (the benchmark's configuration) and
    with raw or precomputed gates (a = g <= 0, b = beta): outputs, record,
    coefficients, u, windows and states equal gdn_conv + gdn_spec_verify bit
    for bit over 6 steps."""
    d = synth.spec(R=8, steps=6)
    R, n, steps, sh = d["R"], d["n"], d["steps"], d["shapes"]
    start, ln = d["row_start"][:R], d["row_len"][:R]
    rng = np.random.default_rng(77 + gate_mode)
    Ls = []
    for _ in range(2):
        L = Layer(sh, d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, num_pages=R,
                  out=gdn.GDN_BF16, gate_mode=gate_mode)
        L.seed(range(R), S0=d["S0"][:R], hist=to_dev(d["hist0"])[:R])
        Ls.append(L)
    L1, L3 = Ls
    for s in range(steps):
        x, a, b = step_rows(d, s, R, n)
        if gate_mode == 1:
            a = to_dev(synth.as_io(-np.abs(rng.standard_normal((R * n, sh.Hv))) * 0.7, synth.BF16))
            b = to_dev(synth.as_io(rng.uniform(0, 1, (R * n, sh.Hv)), synth.BF16))
        acc = d["accepted"][s][:R]
        _, o1 = one_page_step(L1, start, ln, spec_flags(s, R), acc, x, a, b)
        o3 = L3.spec_step(L3.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc), x, a, b)
        L1.ok()
        L3.ok()
        assert o3.dtype == torch.bfloat16
        assert np.array_equal(bits(o3), bits(o1)), f"outputs differ at step {s}"
        assert torch.equal(L3.pool.buf, L1.pool.buf), f"pages differ at step {s}"


def test_fused_step_device_errors_leave_the_page_alone():
    d = synth.spec(R=4, steps=2)
    n = d["n"]
    start, ln = d["row_start"], d["row_len"]
    L, _, _ = make_layers(d, 4, gdn.GDN_F32, slots=False)
    x, a, b = step_rows(d, 0, 4, n)
    L.spec_step(L.batch(start, ln, flags=spec_flags(0, 4), n_accepted=d["accepted"][0]), x, a, b)
    L.ok()
    x, a, b = step_rows(d, 1, 4, n)
    flags = spec_flags(1, 4)
    flags[2] = SPEC                          # stale parity
    before = _page(L, 2)
    L.spec_step(L.batch(start, ln, flags=flags, n_accepted=d["accepted"][1]), x, a, b)
    assert L.status_code() == gdn.CODES["GDN_DEV_STALE_STEP"]
    assert torch.equal(before, _page(L, 2))


@pytest.mark.parametrize("state", [gdn.GDN_F32, gdn.GDN_BF16])
def test_slots_to_page_and_back_midstream(state):
    """The other direction: a request that ran slot-layout steps is handed
    back to a page from its accepted slot (gdn_slots_to_page) and continues
    one-page, bit-identical to a request that stayed in the slot layout; a
    page with an open record refuses gdn_page_to_slots."""
    d = synth.spec(R=4, steps=5)
    R, n = 4, d["n"]
    start, ln = d["row_start"][:R], d["row_len"][:R]
    _, L2, _ = make_layers(d, R, state)             # slots throughout
    L4, _, _ = make_layers(d, R, state, slots=False)  # pages for the hand-back
    L5 = Layer(d["shapes"], d["io"], d["A_log"], d["dt_bias"], d["conv_w"], Kc=8, state=state,
               num_pages=R, slots=True)
    for s in range(2):
        x, a, b = step_rows(d, s, R, n)
        acc = d["accepted"][s][:R] if s else np.zeros(R, np.int32)
        L2.spec_slots(L2.batch(start, ln, flags=spec_flags(s, R), n_accepted=acc), x, a, b)
        L2.ok()
    acc = d["accepted"][2][:R]
    idx = to_dev(np.arange(R, dtype=np.int32))
    gdn.gdn_slots_to_page(L2.dims, R, idx, to_dev(acc), idx, R, R, L2.slots.buf, L4.pool.buf,
                          L4.status)
    L4.ok()
    for r in range(R):
        assert np.array_equal(bits(L4.pool.state(r)), bits(L2.slots.state(r, int(acc[r]))))
        assert int(L4.pool.flag(r).item()) == 0
    # step 2 both ways: slots resume from the accepted slot, the page starts fresh
    x, a, b = step_rows(d, 2, R, n)
    _, o2 = L2.spec_slots(L2.batch(start, ln, flags=spec_flags(2, R), n_accepted=acc), x, a, b)
    _, o4 = one_page_step(L4, start, ln, spec_flags(0, R), np.zeros(R, np.int32), x, a, b)
    L2.ok()
    L4.ok()
    assert np.array_equal(bits(o2), bits(o4))
    # an open record is not handed over
    before = L5.slots.buf.clone()
    gdn.gdn_page_to_slots(L4.dims, R, idx, idx, R, R, L4.pool.buf, L5.slots.buf, L5.status)
    assert L5.status_code() == gdn.CODES["GDN_DEV_RECORD_OPEN"]
    assert torch.equal(before, L5.slots.buf)
