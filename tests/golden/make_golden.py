"""Writes the golden fixtures of this folder from the fp64 oracle alone (no
CUDA path is involved).  The pages print no worked numerical example of the
attention, so these fixtures are regression records of the oracle, which
the pins in tests/test_oracle.py tie to the pages' definitions; the tests
check that the oracle still reproduces them.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def problem(seed, B, n, Hq, Hkv, d, p):
    rng = np.random.default_rng(seed)
    def r(*shape, std=0.5):
        return np.round(rng.standard_normal(shape) * std, 3)  # short decimal inputs
    return dict(q=r(B, n, Hq, d), k=r(B, n, Hkv, d), v=r(B, n, Hkv, d), kc=r(p, Hkv, d),
                vc=r(p, Hkv, d), do=r(B, n, Hq, d, std=1.0))


def case(name, seed, B, n, Hq, Hkv, d, p, window=0, frozen_prefix=1, theta=1.0e6):
    P = problem(seed, B, n, Hq, Hkv, d, p)
    o, lse = oracle.fwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], frozen_prefix=frozen_prefix,
                        theta=theta, window=window)
    dq, dk, dv, dkc, dvc = oracle.bwd(P["q"], P["k"], P["v"], P["kc"], P["vc"], P["do"],
                                      frozen_prefix=frozen_prefix, theta=theta, window=window)
    out = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dkc=dkc, dvc=dvc)
    return {"name": name,
            "geometry": dict(B=B, n=n, Hq=Hq, Hkv=Hkv, d=d, p=p, window=window,
                             frozen_prefix=frozen_prefix, theta=theta),
            "inputs": {k: v.tolist() for k, v in P.items()},
            "outputs": {k: v.tolist() for k, v in out.items()}}


def main():
    cases = [
        # the end-aligned causal mask behind a 3-row cartridge, row 0 frozen
        case("causal_p3", 1, 1, 5, 2, 1, 8, 3),
        # a sliding window of 4 keys cutting through the cartridge and sink
        case("window4_p3", 2, 1, 5, 2, 1, 8, 3, window=4),
    ]
    for c in cases:
        with open(os.path.join(HERE, c["name"] + ".json"), "w") as f:
            json.dump(c, f, indent=None, separators=(",", ":"))
            f.write("\n")


if __name__ == "__main__":
    main()
