"""Default tile and depth per problem class, frozen from the sweep.

Chapter 11 "Pipeline and autotuning", section 3.8, recommends writing the
tuned config back as the function's defaults per compute capability and
keeping a switch to turn tuning off; this table is that frozen result for
compute capability 10.3 (GB300).  ``sweep.py`` regenerates it by measurement.
"""

from __future__ import annotations

# (operand dtype code, output dtype code) -> list of (max tiles, block, num_stages)
# The first entry whose tile budget covers the problem wins.
TABLE = {
    "large": ((256, 256, 64), 3),
    "small": ((128, 128, 64), 4),
}


def choose(M: int, N: int, K: int, dtype: int, out_dtype: int):
    """(block, num_stages) for a problem; small outputs use narrower tiles to cover more SMs."""
    tiles_wide = -(-M // 256) * -(-N // 256)
    if tiles_wide >= 152:
        block, stages = TABLE["large"]
    else:
        block, stages = TABLE["small"]
    # fp32 output needs twice the staging of 16-bit output; 3 stages of
    # 256x256x64 still fit the 227 KiB block limit either way.
    return block, stages
