"""The oracle reproduces its stored fixtures (written by tests/golden/make_golden.py).

Guards against the oracle drifting between compilers, platforms or edits: a
change to its arithmetic must come with regenerated fixtures and a reason.
"""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_oracle_matches_stored_fixture(mode):
    fx = json.load(open(os.path.join(HERE, f"oracle_{mode}_1x2x10x3x4.json")))
    x = {k: (None if v is None else np.array(v)) for k, v in fx["inputs"].items()}
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode, threads=1)
    gr = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], x["dhT"],
                        mode=mode, threads=1)
    got = {"o": o, "hT": hT} | gr
    for k, ref in fx["outputs"].items():
        if ref is None:
            assert got[k] is None
            continue
        np.testing.assert_allclose(got[k], np.array(ref), rtol=1e-12, atol=1e-13, err_msg=k)
