"""Writes ``oracle_small.json``: oracle outputs on two small fixed cases (a regression lock).

Calls only the oracle.  The first case is the dyadic worked example of the pin tests (T=3,
lambda=1/2, scale=1/2); the second is a seeded 130-token case with H=2, dk=96, dv=192 and h0,
from which a few sampled outputs are kept.  Rerun this script only when a change to the oracle's
arithmetic is justified by the source (the commit must say which passage)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import glasynth as gs  # noqa: E402
import oracle  # noqa: E402


def cases():
    q = np.array([[1, 2], [0, 1], [3, -1]], np.float32)[:, None, :]
    k = np.array([[1, 0], [2, 1], [-1, 1]], np.float32)[:, None, :]
    v = np.array([[1, 1], [0, 2], [4, -3]], np.float32)[:, None, :]
    h0 = np.array([[1, 0], [0, 2]], np.float32)[None, None]
    ll = np.array([np.log(0.5)], np.float32)
    yield "dyadic_T3", dict(q=q, k=k, v=v, h0=h0, ll=ll, scale=0.5)
    T, H = 130, 2
    q = gs.bf16_round(gs.normal(0, 1, (T, H, 96), 1 / np.sqrt(96)))
    k = gs.bf16_round(gs.normal(0, 2, (T, H, 96), 1 / np.sqrt(96)))
    v = gs.bf16_round(gs.normal(0, 3, (T, H, 192)))
    h0 = gs.normal(0, 4, (1, H, 96, 192), 0.1)
    ll = np.log(np.array([0.97, 0.999], np.float32))
    yield "seeded_T130", dict(q=q, k=k, v=v, h0=h0, ll=ll, scale=float(gs.SCALE))


SAMPLES = {"o": [(0, 0, 0), (1, 1, 5), (127, 0, 191), (128, 1, 64), (129, 0, 100)],
           "hT": [(0, 0, 0, 0), (0, 1, 95, 191), (0, 0, 50, 7)]}


def main():
    out = {}
    for name, c in cases():
        o, hT = oracle.fwd(c["q"], c["k"], c["v"], c["ll"], c["scale"], h0=c["h0"])
        if name == "dyadic_T3":
            out[name] = {"o": o.tolist(), "hT": hT.tolist()}
        else:
            out[name] = {"o": {str(i): float(o[i]) for i in SAMPLES["o"]},
                         "hT": {str(i): float(hT[i]) for i in SAMPLES["hT"]}}
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
