"""Writes the stored mixing-matrix fixtures in this folder.  Calls only ``oracle/``.

The MHLA pages print no numeric example, so the fixtures here are the oracle's
own W for small block grids (after its closed-form and invariant pins pass),
stored as float32 bit patterns.  They guard against drift of the oracle and let
the host-side initialiser of the library be checked bit for bit without a GPU.

Run from the repository root:  python tests/golden/write_golden.py
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402

CASES = [
    # (grid, block, transform, local_thres, exp_sigma)
    ((16, 16), (4, 4), "linear", 1.5, 3.0),
    ((16, 16), (4, 4), "cos", 1.5, 3.0),
    ((16, 16), (4, 4), "exp", 1.5, 3.0),
    ((16, 16), (4, 4), "gaussian", 1.5, 3.0),
    ((16, 16), (4, 4), "local", 1.5, 3.0),
    ((14, 14), (2, 2), "linear", 1.5, 3.0),
    ((8, 12), (4, 4), "exp", 1.5, 2.0),
    ((8, 16, 24), (4, 8, 8), "linear", 1.5, 3.0),
    ((4, 4, 6), (2, 2, 2), "local", 1.8, 3.0),
]


def case_name(grid, block, transform, local_thres, exp_sigma):
    g = "x".join(map(str, grid))
    b = "x".join(map(str, block))
    return f"{g}_b{b}_{transform}_t{local_thres}_s{exp_sigma}"


def main():
    path = os.path.join(HERE, "mixing_w.txt")
    with open(path, "w") as f:
        f.write("# MHLA mixing matrices W (row-major, W[i][j], i = query block), float32 bits in hex.\n")
        f.write("# Written by tests/golden/write_golden.py from oracle.mixing_matrix; the\n")
        f.write("# construction is BlockDistanceConv._compute_block_distances / _apply_transform of\n")
        f.write("# the MHLA module walkthrough (171host.com/767426.html), section 7.\n")
        for c in CASES:
            W = oracle.mixing_matrix(c[0], c[1], c[2], local_thres=c[3], exp_sigma=c[4])
            bits = W.astype(np.float32).view(np.uint32).reshape(-1)
            f.write(f"case {case_name(*c)} M={W.shape[0]}\n")
            for r in range(0, bits.size, 16):
                f.write(" ".join(f"{x:08x}" for x in bits[r:r + 16]) + "\n")
    print("wrote", path)


def load():
    """{case_name: float32 W} from mixing_w.txt."""
    out, cur, vals, M = {}, None, [], 0
    with open(os.path.join(HERE, "mixing_w.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            if line.startswith("case "):
                if cur is not None:
                    out[cur] = np.array(vals, dtype=np.uint32).view(np.float32).reshape(M, M)
                parts = line.split()
                cur, M, vals = parts[1], int(parts[2][2:]), []
            else:
                vals.extend(int(x, 16) for x in line.split())
    if cur is not None:
        out[cur] = np.array(vals, dtype=np.uint32).view(np.float32).reshape(M, M)
    return out


if __name__ == "__main__":
    main()
