"""Write the stored oracle outputs used as regression fixtures.

Calls only ``oracle`` and ``synth``; nothing here touches the CUDA library.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def toy_fixture(seed=0):
    wl = synth.TOY
    L, M = wl.layer, wl.Ms[0]
    x = synth.hidden(M, L.H, seed)
    ids, w = synth.routing(M, L, seed)
    w13, s13, w2, s2 = synth.layer_weights(L, seed)
    r = oracle.forward(x, ids, w, w13, s13, w2, s2, L.E, L.H, L.I, want_intermediates=True)
    return {
        "what": "oracle output of the toy layer (E=8, H=256, I=128, top-2, M=4), seed 0",
        "made_by": "tests/golden/make_golden.py (oracle + synth only)",
        "ids": ids.tolist(), "topk_w": [[float(v) for v in row] for row in w],
        "counts": r["counts"].tolist(), "offsets": r["offsets"].tolist(),
        "perm": r["perm"].tolist(), "inv_perm": r["inv_perm"].tolist(),
        "out_hex": [[float(v).hex() for v in row] for row in r["out"]],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "toy_seed0_oracle.json"), "w") as f:
        json.dump(toy_fixture(), f, indent=0)
    print("wrote toy_seed0_oracle.json")
