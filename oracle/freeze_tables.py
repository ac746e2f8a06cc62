"""Write oracle/zo_frozen_tables.h: the oracle's copy of the code tables of
stream format v1, frozen as integers.

Test infrastructure, like the rest of oracle/.  The tables are regenerated
here from the oracle's own closed-form pmf and package-merge (``zo_phase_table``
in zipccl_oracle.c) and nothing else; the oracle's encoder and predictor read
the frozen copy, so that its streams no longer depend on the host's libm
``erf``.  The CPU tests rebuild the tables and check that they still equal
the frozen ones.

usage: python oracle/freeze_tables.py
"""
from __future__ import annotations

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402

OUT = os.path.join(HERE, "zo_frozen_tables.h")


def render() -> str:
    offs, lens = oracle.rebuilt_phase_tables()
    rows = ",\n".join("    {" + ", ".join(str(v) for v in row) + "}" for row in lens)
    return (
        "/* zo_frozen_tables.h -- the oracle's frozen code tables of stream format v1.\n"
        " * Written by oracle/freeze_tables.py from the oracle's package-merge over the\n"
        " * closed-form Gaussian exponent pmf at sigma = 2^(r/16), r = 0..15 (window of\n"
        " * the 15 exponents of largest mass, escape symbol 15, lengths limited to 10).\n"
        " * Test infrastructure: read by zipccl_oracle.c only. */\n"
        "static const int zo_frozen_base_off[16] = {" + ", ".join(str(v) for v in offs) + "};\n"
        "static const int zo_frozen_lens[16][16] = {\n" + rows + "\n};\n")


def main() -> None:
    text = render()
    with open(OUT, "w") as f:
        f.write(text)
    print(f"wrote {OUT}")


if __name__ == "__main__":
    main()
