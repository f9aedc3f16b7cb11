"""Writes the stored expected values under tests/golden/ from the fp64 oracle.

Run from the repository root:  python tests/golden/make_golden.py
The values come from oracle/ only (inputs from the seeded generator); nothing
here touches the CUDA path.  Each fixture stores its own inputs, so a test can
re-run the oracle on exactly these numbers and compare.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_recurrence_delta_gb300 import inputs as I  # noqa: E402

CITES = {
    "gated": "GDN & MLA Mechanism Deep-Dive, Step 4 (Gated delta rule)",
    "delta": "HyMo-434M documentation portal, card 01 (GDN recurrence, delta rule)",
}


def fixture(mode):
    w = I.custom(name=f"golden_{mode}", mode=mode, dtype="f32", B=1, H=2, T=10, dk=3, dv=4, seed=2024,
                 h0_std=0.5, backward=True)
    x = I.make_inputs(w)
    rng_dhT = 0.25 * I.normal(2024, 99, 2 * 3 * 4).reshape(1, 2, 3, 4)
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode, threads=1)
    gr = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], rng_dhT,
                        mode=mode, threads=1)
    tol = lambda a: None if a is None else a.tolist()
    return {
        "cite": CITES[mode],
        "written_by": "tests/golden/make_golden.py (oracle/ only)",
        "mode": mode,
        "shape": {"B": 1, "H": 2, "T": 10, "dk": 3, "dv": 4},
        "inputs": {k: tol(x[k]) for k in ("v", "b", "c", "g", "beta", "A_log", "h0", "dO")} | {"dhT": rng_dhT.tolist()},
        "outputs": {"o": o.tolist(), "hT": hT.tolist()} | {k: tol(v) for k, v in gr.items()},
    }


if __name__ == "__main__":
    for mode in ("gated", "delta"):
        path = os.path.join(ROOT, "tests", "golden", f"oracle_{mode}_1x2x10x3x4.json")
        with open(path, "w") as f:
            json.dump(fixture(mode), f, indent=None, separators=(",", ":"))
            f.write("\n")
        print("wrote", path)
