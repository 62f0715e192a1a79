"""The float64 oracle against its pins (library routines, closed forms, invariants)
and against the pages' own worked arithmetic."""
import os

import pytest

import oracle
from mla_latent_kv_attention_gb300 import accounting
from tests import oracle_pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


def test_kv_footprint_matches_page():
    """The page's 1.96 GB / 245 MB for 142,000 tokens x 24 layers x 576 B (and DCP8)."""
    rows = []
    with open(os.path.join(HERE, "golden", "kv_footprint.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    assert rows
    for positions, layers, bpp, shards, page_fig, unit in rows:
        assert bpp == accounting.D
        got = accounting.kv_cache_bytes(int(positions), int(layers), int(shards))
        assert abs(got - page_fig) <= unit / 2, (got, page_fig)
    assert accounting.kv_cache_bytes(142000, 24) == 1_963_008_000
    assert accounting.kv_cache_bytes(142000, 24, 8) == 245_376_000
