"""Reader for the text fixtures under tests/golden/ (each cites its source)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def parse(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            toks = val.split()
            vals = []
            for t in toks:
                try:
                    vals.append(int(t))
                except ValueError:
                    vals.append(t)
            out[key.strip()] = vals if len(vals) != 1 else vals[0]
    return out


def load_all():
    res = {}
    for name in sorted(os.listdir(GOLDEN)):
        if name.endswith(".txt"):
            res[name[:-4]] = parse(os.path.join(GOLDEN, name))
    return res
