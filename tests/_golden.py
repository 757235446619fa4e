"""Reader for the hand-derived fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            k, v = line.split("=", 1)
            out[k.strip()] = v.strip()
    return out


def sym_map(text, default_key="others"):
    """'3:2 7:1 others:1' -> ({3: 2, 7: 1}, 1 or None)."""
    vals, rest = {}, None
    for tok in text.split():
        k, v = tok.split(":")
        if k in (default_key, "rest"):
            rest = int(v)
        else:
            vals[int(k)] = int(v)
    return vals, rest


def int_list(text):
    return [int(t) for t in text.split()] if text else []
