"""Reader for the small text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Returns {key: list of ints or list of int lists for repeated keys}."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            vals = [int(v) for v in vals]
            if key in out:
                if not isinstance(out[key][0], list):
                    out[key] = [out[key]]
                out[key].append(vals)
            else:
                out[key] = vals
    return out
