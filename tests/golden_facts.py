"""Readers for the fixtures under tests/golden/ (values the pages print)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def e2m1_magnitudes():
    vals = []
    with open(os.path.join(GOLDEN, "e2m1_magnitudes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                vals.append(float(line))
    return vals


def facts():
    out = {}
    with open(os.path.join(GOLDEN, "format_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = float(v) if "." in v else int(v)
    return out
