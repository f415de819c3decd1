"""Write tests/golden/oracle_small.json: a small two-sequence GDN problem and
the oracle's fp64 outputs for it (a regression fixture for the oracle).

Calls only oracle/.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(20260501)
    lens = [5, 6]
    T, H, dk, dv = sum(lens), 2, 4, 3
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    inputs = dict(
        q=rng.standard_normal((T, H, dk)),
        k=k,
        v=rng.standard_normal((T, H, dv)),
        g=-0.5 * rng.random((T, H)),
        beta=rng.random((T, H)),
        initial_state=0.1 * rng.standard_normal((len(lens), H, dk, dv)),
    )
    inputs = {n: np.round(a, 6) for n, a in inputs.items()}   # short decimal text
    cu = [0, lens[0], T]
    scale = 0.5
    o, sf = oracle.gdn_reference(inputs["q"], inputs["k"], inputs["v"], inputs["g"], inputs["beta"],
                                 inputs["initial_state"], np.array(cu), scale=scale)
    fx = dict(
        about="GDN forward, fp64 oracle output for a 2-sequence, 2-head, dk=4, dv=3 case; "
              "layouts: q,k [T,H,dk], v,o [T,H,dv], g,beta [T,H], states [N,H,dk,dv] (k-major)",
        cu_seqlens=cu, scale=scale,
        inputs={n: a.tolist() for n, a in inputs.items()},
        o=o.tolist(), final_state=sf.tolist(),
    )
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as f:
        json.dump(fx, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()
