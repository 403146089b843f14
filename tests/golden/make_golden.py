"""Writes the oracle fixtures of this folder.  Calls only the CPU oracle (and
the seeded input generators); never the CUDA library.

    python tests/golden/make_golden.py

The pages print no worked numeric example for decode attention, so these
fixtures are not the pages' numbers: they freeze the oracle's own results on
small seeded inputs, so that a later change of the oracle's arithmetic, or a
platform whose libm rounds differently, shows up as a failing CPU test
(tests/test_oracle.py::test_golden_fixtures) instead of passing silently.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fd_workloads as fw  # noqa: E402
import oracle  # noqa: E402


def cases():
    """(file name, workload, description) of every fixture."""
    tiny = fw.tiny_mqa()
    paged = fw.to_paged(fw.make_contiguous("golden-fp8-paged", 21, [1, 9, 40], 8, 2, 64, "f16",
                                           "e4m3", gap=1), 8, 22)
    i8tok = fw.with_scales(fw.make_contiguous("golden-i8-token", 23, [5, 33], 4, 1, 64, "bf16",
                                              "i8", gap=2), fw.SCALE_TOKEN, 24,
                           powers_of_two=True)
    multi = fw.make_contiguous("golden-q3", 25, [2, 17], 4, 2, 64, "f16", "f16", q_len=3)
    return [
        ("tiny_mqa_f16.json", tiny, "B=2, seq_len {7, 33}, 4/1 heads, D=64, fp16, contiguous"),
        ("fp8_paged8.json", paged, "B=3, seq_len {1, 9, 40}, 8/2 heads, D=64, e4m3, page 8"),
        ("i8_token_scales.json", i8tok, "B=2, seq_len {5, 33}, 4/1 heads, D=64, bf16 q, int8 "
                                        "with per-token scales (powers of two)"),
        ("multi_token_q3.json", multi, "B=2, seq_len {2, 17}, 4/2 heads, D=64, fp16, q_len 3"),
    ]


def main():
    for name, w, desc in cases():
        out, lse = oracle.decode_attention(w)
        doc = {
            "about": "oracle output (fp64) on seeded inputs from fd_workloads; written by "
                     "make_golden.py from the CPU oracle only",
            "workload": desc,
            "out": [float(x).hex() for x in out.ravel()],
            "out_shape": list(out.shape),
            "lse": [float(x).hex() for x in lse.ravel()],
            "lse_shape": list(lse.shape),
        }
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(doc, f, indent=0)
            f.write("\n")
        print(name, out.shape, float(np.abs(out).max()))


if __name__ == "__main__":
    main()
