"""Write the oracle's result for the tiny workload as a text fixture.

Calls only ``oracle`` (and ``synth`` for the seeded inputs). The pages print
no worked numeric example of the recurrence, so this fixture is a regression
guard on the oracle itself, not a pin: the pins live in
tests/test_oracle_pins.py. Re-run only when a change to the oracle's
arithmetic is justified by the method's definition, and say which in the
commit message.

Usage: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth   # noqa: E402


def tiny_result():
    d = synth.tiny()
    sh = d["shapes"]
    y, hist = oracle.conv_f64(d["x"].value, d["hist0"].value, d["conv_w"].value,
                              d["row_start"], d["row_len"])
    o, S = oracle.gdn_f64(y, d["a"].value, d["b"].value, d["A_log"], d["dt_bias"],
                          d["row_start"], d["row_len"], sh.Hk, sh.Hv, sh.Dk, sh.Dv)
    return y, o, S


def main():
    y, o, S = tiny_result()
    path = os.path.join(HERE, "tiny_oracle.txt")
    with open(path, "w") as f:
        f.write("# Oracle result for the tiny workload (1 request, 16 tokens, Hk=Hv=2,\n")
        f.write("# Dk=Dv=32, fp32 inputs, seed 0), written by tests/golden/make_golden.py.\n")
        f.write("# Sections: y (conv'd rows [16][192]), o ([16][2][32]), S ([2][32][32]).\n")
        for name, arr in (("y", y), ("o", o), ("S", S[0])):
            f.write(f"{name} {' '.join(str(s) for s in arr.shape)}\n")
            for v in arr.reshape(-1):
                f.write(f"{v:.17g}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
