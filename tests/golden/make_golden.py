"""Writes tests/golden/oracle_tiny.json from the fp64 oracle alone.

The pages print no worked example; this fixture only guards the oracle
against unintended drift.  It calls nothing but the oracle and the seeded
input generator.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from state_space_model_09_b300 import synth  # noqa: E402

SHAPE = dict(batch=1, seqlen=24, nheads=2, headdim=4, dstate=3, ngroups_b=1, ngroups_c=2,
             chunk=8, io=synth.F32, h0="all")
SEED = 4242
T_STORED = 24

if __name__ == "__main__":
    inp = synth.make_fwd_inputs(synth.FwdShape(**SHAPE), SEED)
    y, h = oracle.ssd_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"])
    out = dict(note="written by tests/golden/make_golden.py from the fp64 oracle",
               shape=SHAPE, seed=SEED, T_stored=T_STORED,
               y_head=y[:, :T_STORED].tolist(), h_final=h.tolist())
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json"), "w") as f:
        json.dump(out, f, indent=1)
