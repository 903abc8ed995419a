"""Seeded synthetic inputs for the Gated DeltaNet layer core.

This module is shared by the CUDA-path tests, the oracle tests and the
benchmark, and holds none of the method's arithmetic: it draws random inputs
with fixed seeds, rounds them to the storage dtype, and lays out row maps.

Workloads (shapes of the Qwen3.5-family GDN layer the pages measure):
  * ``tiny``      1 request, 16 tokens, 2 q/k heads, 2 v heads, Dk=Dv=32,
                  fp32 everything, zero initial state.
  * ``decode``    64 requests x 1 token, 16 q/k heads, 32 v heads,
                  Dk=Dv=128, 8192 conv channels, bf16 rows, fp32 state
                  N(0, 0.02), a 3-column conv window N(0, 1).
  * ``spec``      64 requests, 1+7 candidates per step, 20 steps, accepted
                  drafts per request and step ~ U{0..7}.
  * ``mixed``     8 prefills of U{45..400} tokens packed with 32 spec-decode
                  requests of 8 candidates, through a row map.
  * ``long``      4 sequences of 8192 tokens for the chunked prefill.

Distributions: q/k/v conv inputs, a and b ~ N(0, 1); A_log ~ U(-1, 1);
dt_bias ~ U(-0.5, 0.5); conv taps ~ U(-0.5, 0.5).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclass(frozen=True)
class Shapes:
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    W: int = 4

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv


TINY = Shapes(Hk=2, Hv=2, Dk=32, Dv=32)
FULL = Shapes(Hk=16, Hv=32, Dk=128, Dv=128)

SEEDS = {"tiny": 0, "decode": 1, "spec": 2, "mixed": 3, "long": 4}


def bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns -> their exact fp32 values."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Tensor:
    """A host input in its storage dtype plus its exact value."""
    store: np.ndarray   # float32 or uint16 (bf16 bits)
    value: np.ndarray   # float32 holding exactly the stored value
    dtype: str


def as_io(x, dtype: str) -> Tensor:
    x = np.asarray(x, np.float32)
    if dtype == F32:
        x = np.ascontiguousarray(x)
        return Tensor(x, x, F32)
    bits = bf16_bits(x)
    return Tensor(bits, bf16_value(bits), BF16)


def params(rng, sh: Shapes, io: str):
    return {
        "A_log": rng.uniform(-1.0, 1.0, sh.Hv).astype(np.float32),
        "dt_bias": rng.uniform(-0.5, 0.5, sh.Hv).astype(np.float32),
        "conv_w": as_io(rng.uniform(-0.5, 0.5, (sh.C, sh.W)), io),
    }


def state(rng, R, sh: Shapes, std=0.02):
    """Initial states in the math layout [R][Hv][Dk][Dv], fp32."""
    return (rng.standard_normal((R, sh.Hv, sh.Dk, sh.Dv)) * std).astype(np.float32)


def rows(rng, T, sh: Shapes, io: str):
    return {
        "x": as_io(rng.standard_normal((T, sh.C)), io),
        "a": as_io(rng.standard_normal((T, sh.Hv)), io),
        "b": as_io(rng.standard_normal((T, sh.Hv)), io),
    }


def pack(lengths, order=None):
    """Row map for requests of the given lengths, packed in ``order``."""
    lengths = np.asarray(lengths, np.int32)
    R = lengths.shape[0]
    order = np.arange(R) if order is None else np.asarray(order)
    start = np.zeros(R, np.int32)
    pos = 0
    for r in order:
        start[r] = pos
        pos += int(lengths[r])
    return start, lengths.copy(), int(pos)


def tiny(seed=SEEDS["tiny"], T=16):
    rng = np.random.default_rng(seed)
    sh = TINY
    d = {"shapes": sh, "io": F32, "R": 1}
    d.update(params(rng, sh, F32))
    d.update(rows(rng, T, sh, F32))
    d["row_start"], d["row_len"], d["T"] = pack([T])
    d["S0"] = np.zeros((1, sh.Hv, sh.Dk, sh.Dv), np.float32)
    d["hist0"] = as_io(np.zeros((1, sh.W - 1, sh.C)), F32)
    d["fresh"] = np.array([True])
    return d


def decode(seed=SEEDS["decode"], R=64, sh=FULL, io=BF16):
    rng = np.random.default_rng(seed)
    d = {"shapes": sh, "io": io, "R": R}
    d.update(params(rng, sh, io))
    d.update(rows(rng, R, sh, io))
    d["row_start"], d["row_len"], d["T"] = pack([1] * R)
    d["S0"] = state(rng, R, sh)
    d["hist0"] = as_io(rng.standard_normal((R, sh.W - 1, sh.C)), io)
    d["fresh"] = np.zeros(R, bool)
    return d


def spec(seed=SEEDS["spec"], R=64, steps=20, n=8, sh=FULL, io=BF16):
    """Spec-decode verify steps: per step, n candidate rows per request."""
    rng = np.random.default_rng(seed)
    d = {"shapes": sh, "io": io, "R": R, "steps": steps, "n": n}
    d.update(params(rng, sh, io))
    d["S0"] = state(rng, R, sh)
    d["hist0"] = as_io(rng.standard_normal((R, sh.W - 1, sh.C)), io)
    d["step_rows"] = [rows(rng, R * n, sh, io) for _ in range(steps)]
    # accepted drafts of the previous step, consumed by step s (s >= 1);
    # step 0 has an empty record, so nothing is accepted there.
    acc = rng.integers(0, n, size=(steps + 1, R)).astype(np.int32)
    acc[0] = 0
    d["accepted"] = acc
    d["row_start"], d["row_len"], d["T"] = pack([n] * R)
    return d


def mixed(seed=SEEDS["mixed"], n_prefill=8, n_spec=32, n=8, lo=45, hi=400,
          sh=FULL, io=BF16, shuffled=False):
    """Prefills packed with spec requests (spec rows first, unless shuffled)."""
    rng = np.random.default_rng(seed)
    R = n_prefill + n_spec
    d = {"shapes": sh, "io": io, "R": R, "n": n, "n_prefill": n_prefill, "n_spec": n_spec}
    d.update(params(rng, sh, io))
    plen = rng.integers(lo, hi + 1, size=n_prefill).astype(np.int32)
    # request r < n_spec is a spec request, the rest are prefills
    lengths = np.concatenate([np.full(n_spec, n, np.int32), plen])
    order = rng.permutation(R) if shuffled else np.arange(R)
    d["row_start"], d["row_len"], d["T"] = pack(lengths, order)
    d["is_spec"] = np.arange(R) < n_spec
    d["fresh"] = ~d["is_spec"]
    d.update(rows(rng, d["T"], sh, io))
    d["S0"] = state(rng, R, sh)
    d["S0"][~d["is_spec"]] = 0.0
    d["hist0"] = as_io(rng.standard_normal((R, sh.W - 1, sh.C)), io)
    # one earlier spec step seeds each spec request's record
    d["prev_rows"] = rows(rng, n_spec * n, sh, io)
    d["prev_accepted"] = rng.integers(0, n, size=n_spec).astype(np.int32)
    return d


def long(seed=SEEDS["long"], B=4, T=8192, sh=FULL, io=BF16):
    rng = np.random.default_rng(seed)
    d = {"shapes": sh, "io": io, "R": B}
    d.update(params(rng, sh, io))
    d["row_start"], d["row_len"], d["T"] = pack([T] * B)
    d.update(rows(rng, B * T, sh, io))
    d["S0"] = np.zeros((B, sh.Hv, sh.Dk, sh.Dv), np.float32)
    d["hist0"] = as_io(np.zeros((B, sh.W - 1, sh.C)), io)
    d["fresh"] = np.ones(B, bool)
    return d
