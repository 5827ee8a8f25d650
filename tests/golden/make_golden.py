"""Write tests/golden/scan_tiny.json: a tiny selective-scan problem (gate, skip,
softplus, two groups) and the fp64 oracle's outputs for it.  Calls only the
oracle; the values are a regression fixture for the oracle itself and a fixed
target for the CUDA path (no value here comes from the pages, which print no
worked example)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def problem():
    rng = np.random.default_rng(20261202)
    batch, dim, seqlen, dstate, ngroups = 1, 4, 9, 16, 2
    # values exactly representable in bf16 (at most 8 significant bits)
    q = lambda a: np.round(a * 64) / 64
    return dict(
        u=q(rng.standard_normal((batch, dim, seqlen))),
        delta=q(0.5 * rng.standard_normal((batch, dim, seqlen))),
        A=-np.tile(np.arange(1, dstate + 1, dtype=np.float64), (dim, 1)),
        B=q(rng.standard_normal((batch, ngroups, dstate, seqlen))),
        C=q(rng.standard_normal((batch, ngroups, dstate, seqlen))),
        D=q(rng.standard_normal(dim)),
        z=q(rng.standard_normal((batch, dim, seqlen))),
        delta_bias=q(rng.standard_normal(dim) - 2.0),
    )


if __name__ == "__main__":
    p = problem()
    y, hs = oracle.scan(**p, delta_softplus=True)
    out = {k: v.tolist() for k, v in p.items()}
    out["delta_softplus"] = True
    out["y"] = y.tolist()
    out["final_state"] = hs.tolist()
    with open(os.path.join(HERE, "scan_tiny.json"), "w") as f:
        json.dump(out, f)
    print("wrote scan_tiny.json")
