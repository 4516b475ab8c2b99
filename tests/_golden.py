"""Reader for the hand-worked fixtures in tests/golden/ (key: value lines)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _records(name):
    """Yield dicts; a new record starts at each 'case:' line (or file start)."""
    rec = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            key, val = key.strip(), val.strip()
            if key == "case" and rec:
                yield rec
                rec = {}
            rec[key] = val
    if rec:
        yield rec


def load(name):
    recs = list(_records(name))
    return recs[0] if len(recs) == 1 else recs


def hexbytes(s):
    return bytes(int(t, 16) for t in s.split())


def ints(s):
    return [int(t) for t in s.split()]


def hexwords(s):
    return [int(t, 16) for t in s.split()]


def assignments(s, value_base=16):
    """'3=7F80 65536=0000' -> {3: 0x7F80, 65536: 0}."""
    out = {}
    for tok in s.split():
        k, _, v = tok.partition("=")
        out[int(k)] = int(v, value_base)
    return out
