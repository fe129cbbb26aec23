"""Writes oracle_small_case.json: a small seeded MSA step and the oracle's outputs.

The pages print no worked example with numbers, so this fixture is a regression
record of the fp64 oracle (it calls only ``oracle/`` and the seeded generator),
not an independent pin; the pins live in tests/test_oracle_pins.py.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import OracleParams, msa_reference  # noqa: E402

CASE = dict(doc_lengths=[37, 21], hq=4, hkv=2, d=8, dp=4, top_k=2, block=8, seed=101)


def main():
    w = synth.custom(CASE["doc_lengths"], CASE["hq"], CASE["hkv"], CASE["d"], CASE["dp"],
                     CASE["top_k"], CASE["seed"], structured=True, block=CASE["block"])
    inp = synth.make_inputs(w, device="cpu")
    prm = OracleParams(hq=w.hq, hkv=w.hkv, d=w.d, dp=w.dp, top_k=w.top_k, block=w.block)
    ref = msa_reference(inp, prm)
    keep = ("sel_idx", "sel_arg", "sel_score", "plse", "o", "lse", "mass", "kl", "dq", "dk", "dv",
            "dq_p", "dk_p")
    data = dict(case=CASE, kl_loss=ref["kl_loss"],
                outputs={n: ref[n].tolist() for n in keep})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_case.json")
    with open(path, "w") as f:
        json.dump(data, f, separators=(",", ":"))
    print("wrote", path)


if __name__ == "__main__":
    main()
