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


def test_attention_flop_accounting_closed_forms():
    """The roofline numerators: visible (row, key) pairs of a causal chunk of T new
    positions at the end of L cached ones are T (L - T) + T (T + 1) / 2 per head; decode
    sees all L keys; the per-pair flops are 2 (576 + 512) absorbed and 2 (192 + 128) in the
    MHA form; the up-projection is 2 L 512 H 256."""
    from mla_latent_kv_attention_gb300 import accounting as A
    for T, L, H in ((1, 1, 1), (4, 32772, 12), (8192, 40960, 12), (100, 100, 3)):
        pairs = (T * (L - T) + T * (T + 1) // 2) * H
        assert A.visible_pairs([L], T, H) == pairs
        assert A.attention_flops([L], T, H) == pairs * 2 * (576 + 512)
        assert A.mha_attention_flops(T, L, H) == pairs * 2 * (192 + 128)
    assert A.visible_pairs([10, 0, 7], 1, 2) == (10 + 0 + 7) * 2
    assert A.mha_projection_flops(40960, 12) == 2 * 40960 * 512 * 12 * 256
    # the full prefill chunk the pages' TTFT case stands for: 7.886e12 absorbed flops
    assert abs(A.attention_flops([40960], 8192, 12) / 1e12 - 7.886) < 0.001


def test_decode_byte_accounting():
    """Every cached row once (576 B), the queries (bf16, 576 wide), the outputs (bf16, 512),
    the LSE (fp32), the lengths and the page-table entries read."""
    from mla_latent_kv_attention_gb300 import accounting as A
    lens = [4096, 1, 65, 0]
    rows = len(lens) * 2 * 12
    pages = 64 + 1 + 2 + 0
    assert A.decode_bytes(lens, 2, 12) == sum(lens) * 576 + rows * (1152 + 1024 + 4) + 4 * 4 + 4 * pages
