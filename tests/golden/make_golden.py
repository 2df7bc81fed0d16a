"""Write the stored expected values under tests/golden/ from the oracle alone.

fig4_shape_p4_n8_g2_b4.json: the shape of the worked example of "Echo:
Error-Compensated 4-Bit Tensor-Parallel Communication", appendix Fig. 4 (P=4,
4-bit codes, a group equal to the two values of one segment, inputs shown to one
decimal).  The page prints no values for that figure, so the inputs here are
seeded one-decimal values and the outputs are the oracle's: a regression guard,
not a pin.  Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def bf16_bits_of_one_decimal(vals):
    # one-decimal values rounded to bf16 (nearest even) by the oracle's converter
    return oracle.f32_to_bf16_rn(np.asarray(vals, np.float32)).reshape(np.shape(vals))


def main():
    rng = np.random.default_rng(4)
    vals = np.round(rng.uniform(-2.0, 2.0, (4, 8)), 1)
    x = bf16_bits_of_one_decimal(vals)
    e = np.zeros((4, 8), np.float32)
    r = oracle.allreduce(x, 2, 4, e=e, want_wire=True)
    out = {
        "source": "Echo paper, appendix Fig. 4 (shape only: P=4, b=4, g=2, n=8); "
                  "values written by oracle/ via tests/golden/make_golden.py",
        "inputs_one_decimal": vals.tolist(),
        "x_bf16_bits": x.astype(int).tolist(),
        "out_bf16_bits": r["out"].astype(int).tolist(),
        "state_f32_bits": e.view(np.uint32).astype(int).tolist(),
        "q2": r["q2"].astype(int).tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fig4_shape_p4_n8_g2_b4.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
