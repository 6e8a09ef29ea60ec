"""Reader for the small text fixtures under tests/golden (values printed on the pages)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    """Return {key: value-string} for the non-comment lines of a fixture file."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.strip()
    return out


def ints(s):
    return [int(x) for x in s.split()]
