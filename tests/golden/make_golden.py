"""Write the oracle regression fixture ``oracle_small_case.txt``.

The pages print no worked numeric example, so this fixture holds no page
values: it records what the fp64 oracle (and only the oracle) returns on one
small seeded case, so that any later change to the oracle's arithmetic shows
up as a diff.  Run from the repository root: ``python tests/golden/make_golden.py``.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_deltanet_state_chunked_gb300 import synthetic  # noqa: E402

CASE = dict(lengths=[5, 7], h_k=1, h_v=2, d_k=4, d_v=3, dtype="f32", seed=424242, gate_scale=0.1, with_S0=True)


def compute():
    x = synthetic.make_replay_inputs(**CASE)
    S, O = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.S0, l2norm_qk=True, scale=0.5)
    Tc, Sl = oracle.chunk_operator(x.k, x.g, x.beta, x.v, x.cu_seqlens)
    SK = oracle.compose(Tc, Sl, x.S0[0])
    return {"S": S, "O": O, "T": Tc, "S_local": Sl, "S_composed": SK}


def main():
    out = compute()
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_case.txt")
    with open(path, "w") as f:
        f.write("# fp64 oracle outputs for tests/golden/make_golden.py CASE (written by the oracle only)\n")
        for name, arr in out.items():
            f.write(f"{name} {' '.join(str(s) for s in arr.shape)}\n")
            f.write(" ".join(repr(float(v)) for v in arr.ravel()) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
