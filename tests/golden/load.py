"""Parser for the hand-worked golden cases in this folder."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def cases(name="hand_worked.txt"):
    out, cur = [], None
    with open(os.path.join(HERE, name)) as fh:
        for raw in fh:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "op":
                cur = {"op": vals[0]}
                out.append(cur)
            else:
                cur[key] = np.array([float(v) for v in vals], dtype=np.float32)
    return out
