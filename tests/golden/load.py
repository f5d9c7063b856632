"""Reader for the small text fixtures in this folder (no arithmetic)."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def read_matrices(name):
    """{label: array} from a fixture: '# ...' comments, then blocks of
    'label rows cols' followed by `rows` lines of `cols` numbers."""
    out, lines = {}, []
    for raw in open(os.path.join(HERE, name)):
        line = raw.split("#", 1)[0].strip()
        if line:
            lines.append(line)
    i = 0
    while i < len(lines):
        label, r, c = lines[i].split()
        r, c = int(r), int(c)
        rows = [[float(v) for v in lines[i + 1 + k].split()] for k in range(r)]
        assert all(len(row) == c for row in rows), label
        out[label] = np.array(rows, dtype=np.float64)
        i += 1 + r
    return out
