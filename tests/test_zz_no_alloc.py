"""gdn_chunk_prefill_noalloc: the two-pass chunked prefill on the library's
own device scratch array (no caller workspace, no allocation).

Checked against gdn_chunk_prefill with a caller workspace on the same inputs,
within the chunked tests' tolerance, on two calls in a row (the second call
finds the first call's items in the shared array). Collected last so that it
also runs after every other GPU test in the same process.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_14_gb300 as gdn
import synth
from tests.gpu_util import CHUNK_ELEM_C, Layer, assert_close, f64, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _case(seed, lengths, order):
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    rng = np.random.default_rng(seed)
    start, ln, T = synth.pack(lengths, order)
    d = {"shapes": sh, "io": synth.BF16}
    d.update(synth.params(rng, sh, synth.BF16))
    rows = synth.rows(rng, T, sh, synth.BF16)
    S0 = synth.state(rng, len(lengths), sh, std=0.1)
    return sh, d, start, ln, rows, S0


def _run(sh, d, start, ln, rows, S0, fresh, noalloc):
    R = len(ln)
    L = Layer(sh, synth.BF16, d["A_log"], d["dt_bias"], d["conv_w"], num_pages=R)
    L.seed(range(R), S0=S0)
    B = L.batch(start, ln, flags=np.where(fresh, gdn.GDN_REQ_FRESH, 0))
    o = torch.zeros(B.num_rows, sh.Hv, sh.Dv, dtype=torch.float32, device="cuda")
    qkv, a, b = to_dev(rows["x"]), to_dev(rows["a"]), to_dev(rows["b"])
    if noalloc:
        gdn.gdn_chunk_prefill_noalloc(L.dims, B, L.params, qkv, a, b, o, L.pool.buf, L.status)
    else:
        ws_bytes = gdn.gdn_chunk_prefill_workspace_bytes(L.dims, B)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        gdn.gdn_chunk_prefill(L.dims, B, L.params, qkv, a, b, o, L.pool.buf, ws, ws_bytes,
                              L.status)
    torch.cuda.synchronize()
    L.ok()
    S = np.stack([f64(L.pool.state_math(r)) for r in range(R)])
    return f64(o), S


def test_noalloc_matches_workspace_form_two_calls_in_a_row():
    sh, d, start, ln, rows, S0 = _case(303, [200, 64, 1, 130, 0, 129], [3, 0, 5, 1, 4, 2])
    fresh = np.array([False, True, False, True, True, False])
    o_ref, S_ref = _run(sh, d, start, ln, rows, S0, fresh, noalloc=False)
    for call in range(2):
        o, S = _run(sh, d, start, ln, rows, S0, fresh, noalloc=True)
        assert_close(o, o_ref, TOL, what=f"o, call {call}", c=CHUNK_ELEM_C)
        for r in range(len(ln)):
            assert_close(S[r], S_ref[r], TOL, inner=2, what=f"S request {r}, call {call}",
                         c=CHUNK_ELEM_C)


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    sh = synth.Shapes(Hk=2, Hv=4, Dk=128, Dv=128)
    L = Layer(sh, synth.BF16, np.zeros(sh.Hv), np.zeros(sh.Hv),
              np.zeros((sh.C, sh.W), np.float32), num_pages=1)
    # 4 value heads x 256 chunks of 64 rows = 1024 items of 97 KiB > 64 MiB
    T = 256 * 64
    B = L.batch([0], [T], flags=gdn.GDN_REQ_FRESH)
    assert gdn.gdn_chunk_prefill_workspace_bytes(L.dims, B) > 64 << 20
    rows = torch.zeros(T, sh.C, dtype=torch.bfloat16, device="cuda")
    ab = torch.zeros(T, sh.Hv, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(T, sh.Hv, sh.Dv, dtype=torch.float32, device="cuda")
    with pytest.raises(gdn.GdnError):
        gdn.gdn_chunk_prefill_noalloc(L.dims, B, L.params, rows, ab, ab, o, L.pool.buf, L.status)
    assert L.status_code() == 0
