"""The oracle reproduces its committed regression fixture (tests/golden)."""
import json
import os

import numpy as np

import synth
from oracle import OracleParams, msa_reference

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_regression_fixture():
    with open(os.path.join(HERE, "golden", "oracle_small_case.json")) as f:
        data = json.load(f)
    c = data["case"]
    w = synth.custom(c["doc_lengths"], c["hq"], c["hkv"], c["d"], c["dp"], c["top_k"], c["seed"],
                     structured=True, block=c["block"])
    inp = synth.make_inputs(w, device="cpu")
    prm = OracleParams(hq=w.hq, hkv=w.hkv, d=w.d, dp=w.dp, top_k=w.top_k, block=w.block)
    ref = msa_reference(inp, prm)
    for name, want in data["outputs"].items():
        np.testing.assert_allclose(ref[name], np.asarray(want), rtol=1e-12, atol=1e-12, err_msg=name)
    assert abs(ref["kl_loss"] - data["kl_loss"]) <= 1e-12 * max(1.0, abs(data["kl_loss"]))
