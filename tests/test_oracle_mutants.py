"""Every deliberately broken oracle build must fail at least one pin.

Each mutant plants one plausible mistake in the oracle's C source (a dropped
term, a wrong sign, an inclusive instead of exclusive offset, a strided
expert-to-rank map, a stride that ignores padding, an unstable order, bf16
truncation, pairs counted instead of tokens, the wrong alignment, floor
instead of ceiling division, padded rows that route somewhere, a NaN result
other than the canonical one, a double rounding). The pins are
only trusted if each of these is caught.
"""
import pytest

from oracle import Oracle
from oracle_pins import PINS

MUTANTS = {
    1: "combine drops the last top-k term",
    2: "combine subtracts instead of adds",
    3: "expert offsets inclusive instead of exclusive",
    4: "expert-to-rank map strided instead of contiguous",
    5: "per-rank stride ignores the padding to 4",
    6: "rows handed out in reverse token order",
    7: "bf16 cast truncates",
    8: "tokens_in_rank counts pairs",
    9: "padding to a multiple of 8",
    10: "capacity uses floor division",
    11: "padded rows route to experts",
    12: "combine backward scales every row by the first score",
    13: "dispatch backward drops the first term",
    14: "packed layout placed like the strided one",
    15: "expert GEMM uses the next expert's weights",
    16: "dedupe writes one row per pair instead of per rank",
    17: "combine accumulates in descending k",
    18: "rank prefix exclusive instead of inclusive",
    19: "receive source records the token, not the pair",
    20: "expert GEMM sums in fp32",
    21: "dedupe records global expert ids",
    22: "dedupe expansion reads another rank's row",
    23: "combine backward score gradient summed in fp32",
    24: "combine flushes subnormal results to zero",
    25: "bf16 cast rounds NaNs like numbers",
    26: "capacity from the call's T instead of num_tokens_per_rank",
    27: "expert GEMM reads the weights transposed",
    28: "bf16 ties round away from zero",
    29: "arithmetic NaN results keep the host's NaN instead of the canonical one",
    30: "bf16 cast of a NaN drops its sign and payload",
    31: "expert GEMM rounds twice, through fp32",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_mutant_is_caught(mutant):
    o = Oracle(mutant)
    assert o.lib.oracle_mutant_id() == mutant
    caught = []
    for pin in PINS:
        try:
            pin(o)
        except Exception:       # a failed assertion or a rejected call
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
