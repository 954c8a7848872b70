"""Reader for the hand-written fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_cases(name):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = {"name": parts[1]}
            elif parts[0] == "end":
                cases.append(cur)
                cur = None
            elif parts[0] == "N":
                cur["N"] = int(parts[1])
            else:
                cur[parts[0]] = np.array([int(v) for v in parts[1:]], dtype=np.int64)
    return cases
