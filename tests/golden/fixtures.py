"""Readers of the text fixtures in this folder (no arithmetic of the
method here)."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def worked_example_2x2():
    """Inputs [1, 3, 1, 2] (B, T, H, d), expected o [1, 3, 1, 2] and final
    state [1, 1, 2, 2] of kla_worked_example_2x2.txt, as float64 arrays."""
    toks, state = [], []
    with open(os.path.join(HERE, "kla_worked_example_2x2.txt")) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "token":
                toks.append([float(x) for x in parts[2:]])
            elif parts[0] == "state":
                state.append([float(x) for x in parts[1:]])
    a = np.array(toks)
    alpha, eta = a[:, 0], a[:, 1]
    k, v, q, o = a[:, 2:4], a[:, 4:6], a[:, 6:8], a[:, 8:10]
    shape = lambda x: x.reshape(1, len(toks), 1, 2)
    return dict(q=shape(q), k=shape(k), v=shape(v),
                log_alpha=np.log(alpha).reshape(1, len(toks), 1),
                eta=eta.reshape(1, len(toks), 1), eps=0.0,
                o=shape(o), hT=np.array(state).reshape(1, 1, 2, 2))


def precond_squash_2d():
    """x, delta, A0 [1, 1, 2], k [1, 1, 1, 2], expected write key kw
    [1, 1, 1, 2] and A_T [1, 1, 2] of precond_squash_2d.txt (float64)."""
    vals = {}
    with open(os.path.join(HERE, "precond_squash_2d.txt")) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            vals[parts[0]] = np.array([float(x) for x in parts[1:]])
    return dict(x=float(vals["x"][0]), delta=float(vals["delta"][0]),
                A0=vals["A0"].reshape(1, 1, 2), k=vals["k"].reshape(1, 1, 1, 2),
                kw=vals["kw"].reshape(1, 1, 1, 2),
                AT=vals["AT"].reshape(1, 1, 2))
