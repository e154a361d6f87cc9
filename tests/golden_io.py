"""Reader for the hand-worked schedule fixtures under tests/golden/."""

import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
KINDS = {"A": 0, "H": 1, "U": 2, "L": 3}


def read_schedule(name):
    """-> {k: [(chunk, stage, dest, [(kind, chunk, j, page, tpos), ...]), ...]}"""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, ctx = line.split(":")
            k, chunk, stage, dest = map(int, head.split())
            ents = []
            for item in ctx.split(";"):
                kind, c, j, p, t = item.split()
                ents.append((KINDS[kind], int(c), int(j), int(p), int(t)))
            out.setdefault(k, []).append((chunk, stage, dest, ents))
    return out
