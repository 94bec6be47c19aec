"""Reader for the text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_pairs(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split(None, 1)
                out.append((k, v))
    return out


def read_table(name):
    return {k: v for k, v in read_pairs(name)}
