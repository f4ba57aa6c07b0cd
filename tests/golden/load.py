"""Reader for the text fixtures in this directory."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def page_numbers():
    rows = []
    with open(os.path.join(HERE, "pages_numbers.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                kind, *vals = line.split()
                rows.append((kind, [int(v) for v in vals]))
    return rows
