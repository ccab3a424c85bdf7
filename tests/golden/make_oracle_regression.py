"""Write tests/golden/oracle_regression.json: fp64 oracle outputs on one tiny
seeded packed case.

This is a regression fixture for the oracle itself (it pins nothing new: the
pins live in tests/test_oracle.py); it makes any later change to the oracle's
arithmetic visible.  It calls only ``oracle`` and ``kda_inputs``.

    python tests/golden/make_oracle_regression.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import kda_inputs as ki  # noqa: E402
import oracle  # noqa: E402

CASE = dict(B=2, T=9, H=2, K=4, V=3, dtype="f32", init_state_std=0.5,
            segments=[[4, ("pad", 1), 3], [2, 7]])
SEED = 11


def compute():
    w = ki.custom_workload(**CASE)
    x = ki.make_inputs(w, seed=SEED)
    o, fs = oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                               initial_state=x["initial_state"],
                               segment_ids=x["segment_ids"], threads=1)
    return o, fs


if __name__ == "__main__":
    o, fs = compute()
    out = dict(case=CASE, seed=SEED, o=[float(f"{x:.17g}") for x in o.ravel()],
               final_state=[float(f"{x:.17g}") for x in fs.ravel()])
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=0)
    print("wrote", path)
