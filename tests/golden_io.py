"""Readers for the small text fixtures under tests/golden/ (comment lines start with #)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for raw in f:
            raw = raw.strip()
            if raw and not raw.startswith("#"):
                yield raw.split()


def table(name):
    """key -> list of remaining fields (last occurrence wins), plus the ordered list."""
    d, seq = {}, []
    for parts in lines(name):
        d[parts[0]] = parts[1:]
        seq.append(parts)
    return d, seq
