"""Calibrate the logit-offset scale that skews the synthetic expert load.

Writes nothing: prints the scale lambda for which the expert-load rank law of
the oracle's routing has a least-squares slope of -s (log count against log
rank, ranks 2..E) on full-width synthetic inputs.  The printed value is the
ZIPF_LAMBDA constant of moe_expert_layer_04_gb300/workloads.py.

Only the oracle and the input generator are used.  Exact Zipf(s=1.1) is out of
reach for top-6 routing (the top expert would need more than T/k of the
slots), so the fit excludes rank 1, which saturates near one slot per token.
"""
import argparse

import numpy as np

import oracle
from moe_expert_layer_04_gb300 import workloads as W


def slope(counts):
    c = np.sort(counts)[::-1].astype(np.float64)
    r = np.arange(1, len(c) + 1, dtype=np.float64)
    m = (c > 0) & (r >= 2)
    return np.polyfit(np.log(r[m]), np.log(c[m]), 1)[0]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--s", type=float, default=1.1)
    args = ap.parse_args()
    w = W.scaled(W.WORKLOADS["skewed_mm_fwd"], T=args.tokens, hash_variant=False)
    inp = W.make_inputs(w)
    z0 = oracle.gate_logits(inp["x"], inp["W_g"], exact=True)
    vis = inp["is_vision"].numpy()

    def fit(lam):
        off = W.zipf_offsets(w.E, args.s, w.seed, "cpu", lam=lam).numpy().astype(np.float64)
        ids, _, _, _ = oracle.route(z0 + off, inp["bias"], w.k, w.rho, is_vision=vis)
        return slope(np.bincount(ids.ravel(), minlength=w.E)), ids

    lo, hi = 0.0, 4.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        sl, _ = fit(mid)
        if sl > -args.s:
            lo = mid
        else:
            hi = mid
    lam = 0.5 * (lo + hi)
    sl, ids = fit(lam)
    counts = np.sort(np.bincount(ids.ravel(), minlength=w.E))[::-1]
    print(f"lambda={lam:.4f} slope={sl:.4f} top counts={counts[:6].tolist()} "
          f"tail={counts[-6:].tolist()} T={w.T}")


if __name__ == "__main__":
    main()
