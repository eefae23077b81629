"""Shared-memory load cost of the address patterns the scan kernels' lane
layouts produce, measured on the current GPU by libssmprobe.so
(unit_rates.cu, ``ssmprobe_lds_patterns``): cycles per warp-wide load, i.e.
the shared-memory wavefronts it takes.  Prints one JSON line.

    python selective_state_space_fwd_gb300/probe/lds_patterns.py
"""
import ctypes
import json
import os
import sys

PATTERNS = [
    "16 B, every lane its own address",
    "16 B, one address for the warp",
    "16 B B/C slice of 4 states, state groups in consecutive lanes",
    "16 B B/C slice of 4 states, lane pairs sharing a state group",
    "16 B first chunk of an 8-state B/C slice, consecutive lanes",
    "16 B first chunk of an 8-state B/C slice, lane pairs sharing a state group",
    "8 B delta/x pair, 4-lane channel groups",
    "8 B delta/x pair, the pair-shared layout's channel groups",
]


def main() -> int:
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
    from selective_state_space_fwd_gb300 import build as B
    lib = ctypes.CDLL(B.build_probe())
    out = (ctypes.c_double * len(PATTERNS))()
    rc = lib.ssmprobe_lds_patterns(out, len(PATTERNS))
    if rc != 0:
        print(json.dumps({"error": f"probe status {rc}"}))
        return 1
    print(json.dumps({"cycles_per_warp_load": {name: round(out[i], 3)
                                               for i, name in enumerate(PATTERNS)}}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
