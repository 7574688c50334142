"""Write tests/golden/oracle_small.json from the float64 oracle alone.

The pages print no worked numeric example, so this fixture is a regression
record of the oracle on three tiny, hand-written inputs; the independent pins
live in tests/pins.py.  A change to the oracle's arithmetic that alters these
numbers must name, in its commit message, the passage that justifies it, and
re-run this script:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def cases():
    # BatchNorm2d [B=2, C=2, H=1, W=3]
    bn_x = [[[[1.0, 2.0, 4.0]], [[100.0, 100.5, 99.0]]],
            [[[0.0, -1.0, 3.0]], [[101.0, 98.5, 100.25]]]]
    bn_dy = [[[[0.5, -1.0, 2.0]], [[1.0, 0.0, -0.5]]],
             [[[1.5, 0.25, -2.0]], [[-1.0, 2.0, 0.75]]]]
    bn = dict(x=bn_x, dy=bn_dy, gamma=[1.25, 0.75], beta=[0.1, -0.2],
              running_mean=[0.0, 0.0], running_var=[1.0, 1.0],
              momentum=0.1, eps=1e-5)
    # RMSNorm [R=2, H=4]
    rms = dict(x=[[1.0, -2.0, 0.5, 3.0], [0.25, 0.5, -1.5, 2.0]],
               dy=[[1.0, 0.5, -1.0, 2.0], [-0.5, 1.5, 0.25, -1.0]],
               w=[1.0, 0.5, 1.5, 0.75], eps=1e-5)
    # bias + dropout + add + LayerNorm [R=2, H=4]
    ln = dict(inp=[[0.5, -1.0, 2.0, 0.0], [1.0, 1.5, -0.5, -2.0]],
              residual=[[1.0, 0.0, -1.0, 2.0], [0.5, -0.5, 1.0, 0.25]],
              bias=[0.1, -0.2, 0.3, 0.0],
              mask=[[1, 0, 1, 1], [1, 1, 0, 1]],
              dy=[[1.0, -0.5, 0.25, 2.0], [0.5, 1.0, -1.5, -0.25]],
              gamma=[1.0, 1.25, 0.75, 1.5],
              dz_extra=[[0.1, 0.0, -0.2, 0.3], [0.0, 0.5, 0.25, -0.1]],
              scale=1.25, eps=1e-5)
    return bn, rms, ln


def compute():
    bn, rms, ln = cases()
    f = oracle.batch_norm_forward_train(
        np.array(bn["x"]), bn["gamma"], bn["beta"], bn["running_mean"],
        bn["running_var"], bn["momentum"], bn["eps"])
    b = oracle.batch_norm_backward(np.array(bn["x"]), np.array(bn["dy"]),
                                   bn["gamma"], bn["eps"])
    rstd = oracle.rms_norm_rstd(np.array(rms["x"]), rms["eps"])
    r = oracle.rms_norm_backward(np.array(rms["x"]), np.array(rms["dy"]),
                                 np.array(rms["w"]), rstd)
    z = oracle.dropout_add(ln["inp"], ln["residual"], ln["bias"],
                           np.array(ln["mask"]), ln["scale"])
    mu, lrstd = oracle.layer_norm_saved_stats(z, ln["eps"])
    l = oracle.fused_bias_dropout_add_layer_norm_backward(
        ln["dy"], ln["inp"], ln["residual"], ln["bias"],
        np.array(ln["mask"]), ln["scale"], mu, lrstd, ln["gamma"],
        dz_extra=ln["dz_extra"])
    tolist = lambda d: {k: np.asarray(v).tolist() for k, v in d.items()}
    return {
        "bn": {"inputs": bn, "forward": tolist(f), "backward": tolist(b)},
        "rms": {"inputs": rms, "rstd": rstd.tolist(), "backward": tolist(r)},
        "ln": {"inputs": ln, "mean": mu.tolist(), "rstd": lrstd.tolist(),
               "backward": tolist(l)},
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as fh:
        json.dump(compute(), fh, indent=1)
        fh.write("\n")
