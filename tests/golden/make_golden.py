"""Write tests/golden/tiny_f32.json: oracle outputs for the tiny workload.

The inputs are the seeded draws of the workload generator (the SDPA tutorial
page's [2, 3, 8] example shape, "Overview" section, with seed 0 because the
page's own example is unseeded); every stored output comes from ``oracle/``
alone. Run from the repository root: ``python tests/golden/make_golden.py``.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import attn_bwd_ref, attn_fwd_ref  # noqa: E402
from exact_attention_softmax_gb300 import workloads as wl  # noqa: E402


def main():
    w = wl.WORKLOADS["tiny_f32"]
    seed = 0
    x = wl.workload_inputs(w, seed=seed)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    o, lse = attn_fwd_ref(q, k, v, w.scale, w.causal)
    dq, dk, dv = attn_bwd_ref(q, k, v, do, w.scale, w.causal)
    doc = {
        "what": "oracle outputs for the tiny fp32 workload [B=2,H=1,L=3,d=8], non-causal",
        "source": "oracle/attention.py (fp64), inputs from the seeded workload generator",
        "seed": seed,
        "scale": w.scale,
        "shape": [w.B, w.H, w.Lq, w.d],
        "inputs": {n: [float(t) for t in x[n].reshape(-1).tolist()] for n in ("q", "k", "v", "do")},
        "outputs": {n: [float(t) for t in a.reshape(-1).tolist()]
                    for n, a in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))},
    }
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_f32.json")
    with open(out, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", out)


if __name__ == "__main__":
    main()
