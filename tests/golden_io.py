"""Reader for the fixtures under tests/golden (format: name dtype shape values)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out, meta = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line:
                continue
            if line.startswith("#"):
                for tok in line[1:].split():
                    if "=" in tok:
                        k, v = tok.rstrip(",").split("=", 1)
                        try:
                            meta[k] = int(v)
                        except ValueError:
                            meta[k] = float(v)
                continue
            key, kind, shape, *vals = line.split(" ")
            shape = tuple(int(s) for s in shape.split(","))
            if kind == "f32hex":
                a = np.array([int(v, 16) for v in vals], np.uint32).view(np.float32)
            else:
                a = np.array([int(v) for v in vals], dtype=kind)
            out[key] = a.reshape(shape)
    return out, meta
