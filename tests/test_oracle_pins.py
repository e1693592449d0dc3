"""The oracle against its pins (CPU only), and the pins against planted mistakes."""

import os

import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    fails = pin(orc)
    assert not fails, fails


# Each planted mistake (oracle.c, ORACLE_MUTANT) must make at least one pin fail.
MUTANTS = {
    1: "rotation by the negative angle",
    2: "interleaved pairs instead of half-split",
    3: "global token index as the position",
    4: "exclusive window |i-j| < w",
    5: "scale dropped",
    6: "log base 2 in the lse",
    7: "keys used as values",
    8: "key range one short at the window's far edge",
    9: "key range one too wide at the window's near edge",
    10: "group of short sequences one row over the tile",
    11: "group of short sequences crossing its window",
    12: "rope op: inverse rotates forwards",
    13: "rope op: interleaved layout ignored",
    14: "rope op: features past dims not copied",
    15: "backward: D term dropped from dS",
    16: "backward: key gradient rotated forwards",
    17: "backward: scale missing from the query gradient",
    18: "backward: query gradient rotated forwards",
    19: "backward: value gradient weighted by dS instead of P",
    20: "backward: probabilities not normalised",
    21: "rope op: partial dims paired across the whole head",
    22: "rope op: cos and sin tables swapped",
    23: "values rotated like the keys",
    24: "lse without the row maximum",
    25: "schedule: key range not clipped at the sequence end",
    26: "schedule: last piece of a long sequence given a full tile of rows",
    27: "rows: a sequence's first token given to the sequence before",
    28: "rows: the row's head ignored",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_pins_catch_planted_mistake(tmp_path, mutant):
    path = oracle.compile_oracle(str(tmp_path / f"liboracle_m{mutant}.so"), mutant=mutant)
    bad = oracle.Oracle(path)
    assert P.all_failures(bad), f"no pin fails for mutant {mutant}: {MUTANTS[mutant]}"


def test_oracle_rejects_malformed_offsets(orc):
    # the offsets must run from 0 and never decrease (the GPU path reports the same cases as
    # PK_ERR_BAD_CU); the oracle refuses them rather than computing something
    import numpy as np

    for cu in ([1, 4, 9], [0, 6, 4, 9]):
        cu = np.asarray(cu, dtype=np.uint32)
        with pytest.raises(ValueError):
            orc.schedule(cu, 0)
        T = int(cu[-1])
        qkv = np.zeros((T, 3 * 64), dtype=np.float64)
        tbl = np.zeros((T, 32), dtype=np.float64)
        with pytest.raises(ValueError):
            orc.attend(qkv, tbl, tbl, cu, 1, 0, 0.125, "f64")
