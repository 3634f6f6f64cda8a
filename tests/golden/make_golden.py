"""Write the stored expected values under tests/golden/ by calling the oracle only.

    python tests/golden/make_golden.py

Inputs are hand-chosen edge cases (each with the reason it is there); every
expected value is the oracle's. The pin tests re-derive each expected value from
the exact rational model (tests/exact_model.py) and from PyTorch's conversion, so
a wrong oracle cannot hide behind these files; the GPU tests then hold the CUDA
path to them bit for bit.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402

# (binary64 input as a hex float, why it is here). The pages round to BF16 a single
# time (drafter/linears module text; drafter/comm ArNorm); the mode is read as
# IEEE 754 round-to-nearest-even.
ROUND_INPUTS = [
    ("0x1.0000000000000p+0", "1.0 exactly"),
    ("0x1.0100000000000p+0", "1 + 2^-8: tie between 1.0 (even) and 1 + 2^-7"),
    ("0x1.0300000000000p+0", "1 + 3*2^-8: tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)"),
    ("0x1.0100004000000p+0", "1 + 2^-8 + 2^-30: above the tie; via binary32 it would round twice"),
    ("0x1.00fffffffff00p+0", "just below the 1 + 2^-8 tie"),
    ("-0x1.0100004000000p+0", "negative mirror of the double-rounding trap"),
    ("-0x0.0p+0", "negative zero keeps its sign"),
    ("0x0.0p+0", "positive zero"),
    ("0x1.0p-133", "smallest BF16 subnormal"),
    ("0x1.0p-134", "half the smallest subnormal: tie to even gives +0"),
    ("0x1.8p-133", "1.5 * 2^-133: tie between 2^-133 (odd) and 2^-132 (even)"),
    ("0x1.0000001p-134", "just above half the smallest subnormal"),
    ("0x1.0p-126", "smallest normal"),
    ("0x1.fcp-127", "2^-126 - 2^-133 = 127 * 2^-133: the largest subnormal, exactly"),
    ("0x1.fep-127", "2^-126 - 2^-134: tie between 127*2^-133 (odd) and 2^-126 (even)"),
    ("0x1.fep+127", "largest finite BF16"),
    ("0x1.ffp+127", "tie between the largest finite and 2^128: rounds to +Inf"),
    ("0x1.fefffp+127", "just below that tie: the largest finite"),
    ("0x1.0p+1000", "far beyond binary32: +Inf"),
    ("-0x1.0p+1000", "far beyond binary32: -Inf"),
    ("0x1.92p+1", "3.140625, exactly on the grid"),
    ("0x1.5555555555555p-2", "1/3: rounds up"),
    ("-0x1.5555555555555p-2", "-1/3"),
]

# Reduce columns: (slots as BF16 patterns, residual pattern or None, why).
# The rule: FP32 sum of the TP slots in rank order 0..TP-1 starting from slot 0,
# one BF16 rounding, FP32 add of the residual, one BF16 rounding
# (drafter/comm, module text and ArNorm.kernel; cutedsl/common/twoshot, reduce).
REDUCE_INPUTS = [
    ([0x3F80, 0x3380, 0xBF80], None,
     "1 + 2^-24 - 1 in rank order: 1 + 2^-24 ties to 1, then 0 (FP64 would give 2^-24)"),
    ([0xBF80, 0x3380, 0x3F80], None,
     "the same three values in the other order: -(1 - 2^-24) is exact, then 2^-24"),
    ([0x8000, 0x8000], None, "all -0: the sum starts from slot 0 and stays -0"),
    ([0x8000, 0x0000], None, "-0 + +0 = +0"),
    ([0x0000, 0x8000], None, "+0 + -0 = +0"),
    ([0x8000], None, "TP = 1: identity, -0 included"),
    ([0x8000, 0x8000, 0x8000, 0x8000, 0x8000, 0x8000, 0x8000, 0x8000], None, "TP = 8 of -0"),
    ([0x3F80, 0x3B00, 0x3B00, 0x3B00, 0x3B00], None,
     "1 + 4 * 2^-9 in FP32 is 1 + 2^-7; rounding to BF16 after each add would stay at 1"),
    ([0x3F80, 0x3B80], 0x3B80,
     "AR(1, 2^-8) rounds to 1 (tie), then 1 + 2^-8 ties to 1 again: two roundings, not one"),
    ([0x3F80, 0x3B80], None, "AR(1, 2^-8) alone: tie to even gives 1"),
    ([0x4049, 0xC049], 0x8000, "x + (-x) = +0, then +0 + -0 = +0"),
    ([0x8000, 0x8000], 0x8000, "-0 all through: -0"),
    ([0x7F7F, 0x7F7F], None, "largest finite twice: the binary32 sum overflows to +Inf"),
    ([0x0001, 0x0001], None, "two smallest subnormals: exact in FP32, 2^-132 in BF16"),
    ([0x7F00, 0x7F00], None, "2^127 twice: 2^128 overflows binary32 to +Inf"),
    ([0x7F7F, 0xFF7F, 0x7F7F], None, "max - max + max: finite all the way in rank order"),
    ([0x3F80, 0x3380, 0xBF80, 0x3380], 0x3F80,
     "order-sensitive sum then residual: rank order gives 2^-24, plus 1 rounds to 1"),
]


def main():
    lines = ["# BF16 rounding cases: binary64 input (hex float) -> BF16 pattern.",
             "# Expected values written by tests/golden/make_golden.py from the oracle;",
             "# the pages round to BF16 a single time (drafter/linears module text,",
             "# drafter/comm ArNorm); the mode is read as IEEE 754 round-to-nearest-even.",
             "# input expected  # reason"]
    for text, why in ROUND_INPUTS:
        v = float.fromhex(text)
        lines.append(f"{text} 0x{oracle.bf16_from_f64(v):04x}  # {why}")
    with open(os.path.join(HERE, "bf16_round_cases.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")

    lines = ["# Reduce + residual columns: slot patterns | residual pattern or - | expected.",
             "# Expected values written by tests/golden/make_golden.py from the oracle;",
             "# rule: drafter/comm module text and ArNorm.kernel (rank-order FP32 sum from",
             "# slot 0, one BF16 rounding, FP32 residual add, one BF16 rounding);",
             "# cutedsl/common/twoshot reduce (the same rank-order sum).",
             "# slots | residual | expected  # reason"]
    for slots, res, why in REDUCE_INPUTS:
        p = np.array(slots, dtype=np.uint16).reshape(len(slots), 1, 1)
        r = None if res is None else np.array([[res]], dtype=np.uint16)
        out = int(oracle.reduce_residual(p, r)[0, 0])
        s = " ".join(f"0x{b:04x}" for b in slots)
        rs = "-" if res is None else f"0x{res:04x}"
        lines.append(f"{s} | {rs} | 0x{out:04x}  # {why}")
    with open(os.path.join(HERE, "reduce_cases.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
