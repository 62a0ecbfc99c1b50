"""Parser for the hand-worked fixtures under tests/golden/.

Each data line holds groups of hex bf16 bit patterns separated by '|'; lines
starting with '#' are the derivation and the citation.
"""
import os

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    rows = []
    with open(os.path.join(HERE, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([[int(tok, 16) for tok in grp.split()] for grp in line.split("|")])
    return rows
