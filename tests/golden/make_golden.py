"""Writes oracle_regression.json: the fp64 oracle's outputs on tiny seeded
inputs, stored so that any later change to the oracle's arithmetic shows up.

Calls only ``oracle`` and the seeded input generator.  Run from the repo root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from selective_state_space_111_b300.synth import Spec, make_inputs  # noqa: E402

CASES = {
    "single_f32_B1D2L5": (Spec("single", "f32", B=1, D=2, L=5, N=4, perturb=True), 11),
    "v1_bf16_B1D2L6": (Spec("v1", "bf16", B=1, D=2, L=6, N=4, a_b_noise=0.1), 12),
    "v2_bf16_B1D2L6": (Spec("v2", "bf16", B=1, D=2, L=6, N=4, out_scale=0.5,
                            shared_u=False, perturb=True), 13),
    "ss2d_bf16_B1D1H2W3": (Spec("ss2d", "bf16", B=1, D=1, H=2, W=3, N=4, perturb=True), 14),
}


def run(spec, t):
    if spec.op == "single":
        return oracle.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                     t["delta_bias"])
    if spec.op == "v1":
        return oracle.bimamba_v1(t["u"], t["delta"], t["A"], t["A_b"], t["B"], t["C"], t["D"],
                                 t["z"], t["delta_bias"], out_scale=t["out_scale"])
    if spec.op == "v2":
        return oracle.bimamba_v2(t["u"], t["delta"], t["delta_b"], t["A"], t["A_b"], t["B"],
                                 t["C"], t["B_b"], t["C_b"], t["D"], t["D_b"], t["z"],
                                 t["delta_bias"], t["delta_bias_b"], t["u_b"],
                                 out_scale=t["out_scale"])
    return oracle.ss2d(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                       t["delta_bias"])


def compute_cases():
    return {name: run(spec, make_inputs(spec, seed)).reshape(-1).tolist()
            for name, (spec, seed) in CASES.items()}


def main():
    out = {"about": "fp64 oracle outputs on tiny seeded inputs (see make_golden.py)",
           "cases": compute_cases()}
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as fh:
        json.dump(out, fh, indent=1)


if __name__ == "__main__":
    main()
