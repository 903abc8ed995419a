"""CPU oracle for the Gated DeltaNet layer core (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The CUDA library never does, and the two
share no code: the oracle is the plain definition of the method, written in
C++ (fp64, token by token) plus NumPy orchestration.

Contents
  * ``conv_f32``    fp32-accumulate causal conv + SiLU with a fixed tap order:
                    the value the GPU conv must match bit for bit.
  * ``conv_f64``    the same conv in fp64.
  * ``gdn_f64``     the gated delta rule token by token in fp64, q/k L2 norm
                    and gates per token (r9700-stack v0.2.3 release notes,
                    section 1: the "fp64 token-by-token reference").
  * ``SlotSim``     speculative decode in the slot-per-candidate layout: after
                    every candidate the state and conv window are kept, and the
                    next step resumes from the slot of the last accepted
                    candidate (r9700-stack v0.2.4 release notes, "What it
                    does"). This is the definition the one-page verify must
                    reproduce.

Every function here is pinned by the ``-m "not gpu"`` tests against brute
force (``oracle.brute``), closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# The planted mistakes the C++ oracle can be asked to make (tests only).
MUTATIONS = {
    "none": 0,
    "no_decay": 1,
    "u_sign": 2,
    "out_before_update": 3,
    "gqa_modulo": 4,
    "no_q_norm": 5,
    "beta_not_sigmoid": 6,
    "softplus_sign": 7,
    "transposed_read": 8,
}


def build(force: bool = False) -> str:
    """Compile the C++ oracle into ``oracle/liboracle.so`` (host compiler)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_exp_f32.argtypes = [ctypes.c_float]
            lib.oracle_exp_f32.restype = ctypes.c_float
            lib.oracle_silu_f32.argtypes = [ctypes.c_float]
            lib.oracle_silu_f32.restype = ctypes.c_float
            conv_args = [I, P, P, I, I, P, P, P, P, P, P]
            lib.oracle_conv_f32.argtypes = conv_args
            lib.oracle_conv_f32.restype = None
            lib.oracle_conv_f64.argtypes = conv_args
            lib.oracle_conv_f64.restype = None
            lib.oracle_gdn_f64.argtypes = [I, P, P, I, I, I, I, P, P, P, P, P,
                                           D, D, I, P, P, P, I, I]
            lib.oracle_gdn_f64.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def exp_f32(x: float) -> float:
    return _load().oracle_exp_f32(float(x))


def silu_f32(x: float) -> float:
    return _load().oracle_silu_f32(float(x))


def _rows(row_start, row_len):
    rs = np.ascontiguousarray(row_start, dtype=np.int32)
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    assert rs.shape == rl.shape
    return rs, rl


def conv_f32(x, hist, w, row_start, row_len, bias=None):
    """fp32 conv mirror. x [T][C], hist [R][W-1][C], w [C][W] -> (y, hist_out)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hist = np.ascontiguousarray(hist, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rs, rl = _rows(row_start, row_len)
    T, C = x.shape
    W = w.shape[1]
    R = rs.shape[0]
    assert hist.shape == (R, W - 1, C)
    y = np.zeros((T, C), np.float32)
    hout = np.zeros_like(hist)
    _load().oracle_conv_f32(R, _ptr(rs), _ptr(rl), C, W, _ptr(x), _ptr(hist), _ptr(w),
                            _ptr(bias), _ptr(y), _ptr(hout))
    return y, hout


def conv_f64(x, hist, w, row_start, row_len, bias=None):
    """fp64 conv. Same arguments as ``conv_f32``."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    hist = np.ascontiguousarray(hist, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    rs, rl = _rows(row_start, row_len)
    T, C = x.shape
    W = w.shape[1]
    R = rs.shape[0]
    assert hist.shape == (R, W - 1, C)
    y = np.zeros((T, C), np.float64)
    hout = np.zeros_like(hist)
    _load().oracle_conv_f64(R, _ptr(rs), _ptr(rl), C, W, _ptr(x), _ptr(hist), _ptr(w),
                            _ptr(bias), _ptr(y), _ptr(hout))
    return y, hout


def gdn_f64(qkv, a, b, A_log, dt_bias, row_start, row_len, Hk, Hv, Dk, Dv,
            S0=None, scale=None, eps=1e-6, gate_mode=0, threads=None,
            mutate="none"):
    """Token-by-token gated delta rule in fp64.

    qkv [T][2*Hk*Dk + Hv*Dv] conv'd rows; a, b [T][Hv]; S0 [R][Hv][Dk][Dv] or
    None. Returns (o [T][Hv][Dv], S [R][Hv][Dk][Dv]).
    """
    qkv = np.ascontiguousarray(qkv, dtype=np.float64)
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    A_log = np.ascontiguousarray(A_log, dtype=np.float64)
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float64)
    rs, rl = _rows(row_start, row_len)
    R = rs.shape[0]
    T = qkv.shape[0]
    assert qkv.shape[1] == 2 * Hk * Dk + Hv * Dv
    assert a.shape == (T, Hv) and b.shape == (T, Hv)
    if S0 is not None:
        S0 = np.ascontiguousarray(S0, dtype=np.float64)
        assert S0.shape == (R, Hv, Dk, Dv)
    if scale is None:
        scale = Dk ** -0.5
    o = np.zeros((T, Hv, Dv), np.float64)
    S = np.zeros((R, Hv, Dk, Dv), np.float64)
    rc = _load().oracle_gdn_f64(R, _ptr(rs), _ptr(rl), Hk, Hv, Dk, Dv, _ptr(qkv), _ptr(a),
                                _ptr(b), _ptr(A_log), _ptr(dt_bias), float(scale), float(eps),
                                int(gate_mode), _ptr(S0), _ptr(S), _ptr(o),
                                int(threads or default_threads()), MUTATIONS[mutate])
    if rc != 0:
        raise ValueError("oracle_gdn_f64 rejected its arguments")
    return o, S


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64.

    Used only to model where the method stores a value in bf16 (a bf16
    state page): the oracle keeps fp64 everywhere else.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    out = u.astype(np.uint32).view(np.float32).astype(np.float64)
    return out


class SlotSim:
    """Speculative decode, slot-per-candidate layout, fp64.

    Per request the simulation keeps a list of slots. Slot i holds the GDN
    state and the conv window after candidate i of the latest step. A step
    takes n candidate rows (raw conv inputs plus a/b gates) and the number of
    drafts the previous step accepted (a, so rows 0..a were accepted); it
    resumes from slot a, runs the candidates one after another and stores
    the slots again. This is the layout the r9700-stack v0.2.4 notes describe
    for stock vLLM ("What it does": a state page per candidate, resume from
    the last accepted one).

    ``state_round`` models a bf16 state page: every stored slot is rounded.
    ``row_store`` models the storage dtype of conv'd rows: with it set, the
    conv runs in the fp32 mirror (``conv_f32``) and its output is passed
    through ``row_store`` (e.g. ``round_bf16``) before the recurrence, which
    is where the method keeps conv'd rows in the io dtype (the record holds
    them so; the r9700-stack v0.2.4 notes, "What it does"). Without it the
    conv is fp64 and unrounded.
    """

    def __init__(self, R, Hk, Hv, Dk, Dv, W, conv_w, A_log, dt_bias, S0=None,
                 hist0=None, scale=None, eps=1e-6, gate_mode=0, conv_bias=None,
                 state_round=None, row_store=None, threads=None):
        self.R, self.Hk, self.Hv, self.Dk, self.Dv, self.W = R, Hk, Hv, Dk, Dv, W
        self.C = 2 * Hk * Dk + Hv * Dv
        self.conv_w = np.asarray(conv_w, np.float64)
        self.conv_bias = None if conv_bias is None else np.asarray(conv_bias, np.float64)
        self.A_log = np.asarray(A_log, np.float64)
        self.dt_bias = np.asarray(dt_bias, np.float64)
        self.scale, self.eps, self.gate_mode = scale, eps, gate_mode
        self.state_round = state_round
        self.row_store = row_store
        self.threads = threads
        S0 = np.zeros((R, Hv, Dk, Dv)) if S0 is None else np.asarray(S0, np.float64)
        hist0 = (np.zeros((R, W - 1, self.C)) if hist0 is None
                 else np.asarray(hist0, np.float64))
        # slots[r] = list of (S [Hv][Dk][Dv], hist [W-1][C]); before the first
        # spec step the only slot is the prefill's result.
        self.slots = [[(S0[r].copy(), hist0[r].copy())] for r in range(R)]

    def step(self, x, a, b, n_accepted):
        """Run one verify step.

        x [R][n][C] raw candidate rows, a/b [R][n][Hv], n_accepted [R]
        (index of the slot to resume from; 0 for the first step, whose
        single slot is the prefill result). Returns conv'd rows y [R][n][C]
        and outputs o [R][n][Hv][Dv].

        The state runs on unrounded from candidate to candidate; only what a
        slot stores is rounded (``state_round``), as a bf16 state page would.
        """
        x = np.asarray(x, np.float64)
        a = np.asarray(a, np.float64)
        b = np.asarray(b, np.float64)
        R, n, C = x.shape
        assert R == self.R and C == self.C
        y_all = np.zeros_like(x)
        o_all = np.zeros((R, n, self.Hv, self.Dv))
        S = np.stack([self.slots[r][int(n_accepted[r])][0] for r in range(R)])
        hist = np.stack([self.slots[r][int(n_accepted[r])][1] for r in range(R)])
        one = np.arange(R, dtype=np.int32)
        ones = np.ones(R, dtype=np.int32)
        new_slots = [[] for _ in range(R)]
        for i in range(n):
            # candidate i of every request: one row each, windows and states
            # carried from candidate i-1 (or the resumed slot)
            if self.row_store is None:
                y, hist = conv_f64(x[:, i], hist, self.conv_w, one, ones, bias=self.conv_bias)
            else:
                y, hist = conv_f32(x[:, i], hist, self.conv_w, one, ones, bias=self.conv_bias)
                y = self.row_store(y)
                hist = hist.astype(np.float64)
            o, S = gdn_f64(y, a[:, i], b[:, i], self.A_log, self.dt_bias, one, ones,
                           self.Hk, self.Hv, self.Dk, self.Dv, S0=S, scale=self.scale,
                           eps=self.eps, gate_mode=self.gate_mode, threads=self.threads)
            y_all[:, i] = y
            o_all[:, i] = o
            stored = S if self.state_round is None else self.state_round(S)
            for r in range(R):
                new_slots[r].append((stored[r].copy(), hist[r].copy()))
        if n > 0:
            self.slots = new_slots
        return y_all, o_all

    def state(self, r, slot):
        return self.slots[r][slot][0]

    def window(self, r, slot):
        return self.slots[r][slot][1]
