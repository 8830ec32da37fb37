"""Writes the derived fixtures under tests/golden/ from the oracle alone.

rank1_f5.txt: f^5(1) for the quintic of eq. (2) ("Muon is Scalable" blog,
Background), i.e. the single singular value NS5 gives a rank-1 input.
Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import muon_ref as R  # noqa: E402

with open(os.path.join(HERE, "rank1_f5.txt"), "w") as f:
    f.write("# f^5(1) with (a,b,c) = (3.4445, -4.7750, 2.0315); written by make_golden.py\n")
    f.write("%.17g\n" % R.quintic_iter(1.0, 5))
