"""The CPU oracle against independent ground truth (no GPU needed).

See tests/oracle_checks.py for what each check compares with.  The mutant test
compiles the oracle again with one planted mistake at a time (a dropped K
group, a transposed scale index, a flushed subnormal, truncation instead of
round-to-nearest-even, a dropped sign, a transposed operand, a dropped scale,
padding rows computed, the mask ignored, the quantiser's 448 left out,
truncation in the e4m3 encoder, the addend C dropped, a K-grouped segment
starting one K group early, A's storage layout ignored, a UE8M0 bias of 128,
packed UE8M0 bytes read in reverse, the UE8M0 quantiser's scale rounded down)
and shows that at least one check
fails for each, so the checks are able to see such mistakes.
"""
import pytest

import oracle
from oracle import build as oracle_build
from tests import oracle_checks as C


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("check", C.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    check(orc)


MUTANTS = {
    1: "last K group dropped",
    2: "sb read transposed",
    3: "sa read row-major",
    4: "e4m3 subnormals flushed",
    5: "bf16 truncation",
    6: "B read as [K][N]",
    7: "e4m3 sign dropped",
    8: "B scale dropped",
    9: "padding rows computed",
    10: "mask ignored",
    11: "quantiser scale without 448",
    12: "e4m3 encode truncates",
    13: "addend C dropped",
    14: "k-grouped segment starts a K group early",
    15: "A's storage layout ignored",
    16: "UE8M0 bias 128",
    17: "UE8M0 bytes unpacked in reverse order",
    18: "UE8M0 quantiser scale rounded down",
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return str(tmp_path_factory.mktemp("mutants"))


@pytest.mark.parametrize("n", sorted(MUTANTS), ids=lambda n: MUTANTS[n].replace(" ", "_"))
def test_planted_mistake_is_caught(mutant_dir, n):
    path = oracle_build.build_mutant(n, mutant_dir)
    mut = oracle.Oracle(path)
    caught = []
    for check in C.ALL_CHECKS:
        try:
            check(mut)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"mutant {n} ({MUTANTS[n]}) passed every check"
