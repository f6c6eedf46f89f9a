"""Each planted mistake in the oracle (a dropped term, a wrong sign, a transposed
operand, a wrong selection, a missing renormalisation, a wrong histogram) must
fail at least one pin; this is what makes the pins worth trusting.  Mutations are
compiled from oracle/moe_oracle.c with -DORACLE_MUTATION=n, on the CPU."""
import pytest

import pins

MUTATIONS = {
    1: "shared expert dropped",
    2: "silu sign flipped",
    3: "down projection transposed",
    4: "no renormalisation over the chosen experts",
    5: "smallest logits selected",
    6: "router weight transposed",
    7: "gated activation dropped",
    8: "histogram counts first choice only",
    9: "4-bit codes read with the nibbles swapped",
}


@pytest.mark.parametrize("m", sorted(MUTATIONS), ids=lambda m: f"m{m}")
def test_mutation_is_caught(m):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(m)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutation {m} ({MUTATIONS[m]}) passed every pin"


QUANT_MUTATIONS = {
    1: "odd column packed in the low nibble",
    2: "codes rounded down",
    3: "range divided into 16 steps",
}


@pytest.mark.parametrize("m", sorted(QUANT_MUTATIONS), ids=lambda m: f"q{m}")
def test_quantiser_mutation_is_caught(m):
    failed = []
    for pin in pins.QUANT_PINS:
        try:
            pin(m)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"quantiser mutation {m} ({QUANT_MUTATIONS[m]}) passed every pin"


GDN_MUTATIONS = {
    1: "alpha dropped from the recall in the delta",
    2: "state not decayed",
    3: "output read before the write",
    4: "value head h mapped to key head h % H_k",
    5: "recall with the state transposed",
    6: "beta scales only the new value",
}


@pytest.mark.parametrize("m", sorted(GDN_MUTATIONS), ids=lambda m: f"g{m}")
def test_gdn_mutation_is_caught(m):
    failed = []
    for pin in pins.GDN_PINS:
        try:
            pin(m)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"scan mutation {m} ({GDN_MUTATIONS[m]}) passed every pin"
