"""Writes the stored expected values under tests/golden/ from the oracle alone.

Run: python tests/golden/make_golden.py
It calls only the oracle package; nothing here comes from the CUDA library.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402


def main():
    thr, lv = oracle.tables()
    out = {
        "source": "oracle.tables(): alpha-law thresholds (fp32 bits, index 0 unused) and "
                  "level values (fp16 bits), Lynx reading section 3",
        "alpha": oracle.alpha(),
        "thr_f32_bits": [int(v) for v in thr.view(np.uint32)],
        "lv_f16_bits": [int(v) for v in lv],
    }
    with open(os.path.join(HERE, "tables_alpha255.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
