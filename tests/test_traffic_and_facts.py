"""Byte counts and geometry against the figures the pages print (tests/golden/pages_facts.json)."""

import json
import os

from linear_attention_ssm_step_gb300 import traffic, workloads

FACTS = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")))


def test_state_round_trip_is_the_pages_786kb():
    assert 2 * traffic.STATE_BYTES == FACTS["state_round_trip_bytes_per_row"]["value"]


def test_activation_bytes_are_about_15kb():
    assert abs(traffic.TOKEN_IO_BYTES - FACTS["activation_bytes_per_row_approx"]["value"]) < 1000


def test_b512_state_is_about_402mb():
    assert abs(512 * 2 * traffic.STATE_BYTES - FACTS["state_bytes_at_b512_approx"]["value"]) < 1e6


def test_decode_and_verify_bytes():
    assert traffic.decode_bytes(1) - traffic.PER_CALL_BYTES == 801820
    assert traffic.verify_bytes(1, 8) - traffic.PER_CALL_BYTES == 909508
    assert traffic.decode_bytes(0, 1) - traffic.PER_CALL_BYTES == 4 + 3072


def test_ring_bytes():
    # no fold, 4 live entries: checkpoint + 12 entries + 8 tokens of activations + index + hist_len
    assert traffic.ring_row_bytes(4, 8, False) == 393216 + 12 * 12288 + 8 * 15384 + 8
    assert traffic.ring_row_bytes(12, 8, True) - traffic.ring_row_bytes(12, 8, False) == 393216


def test_geometry_and_packed_row():
    g = FACTS["geometry"]
    assert (traffic.H, traffic.K, traffic.V) == (g["heads"], g["key_dim"], g["value_dim"])
    w = workloads.decode_inputs(2, 3, layout="packed")
    assert w.qkv.shape[-1] == g["packed_row_elems"]
    assert w.q.shape == (2, 12, 128) and w.q.stride() == (4608, 128, 1)
    assert w.k.data_ptr() - w.q.data_ptr() == 1536 * 2 and w.v.data_ptr() - w.q.data_ptr() == 3072 * 2


def test_ring_modes_satisfy_the_capacity_rule():
    r = FACTS["ring"]
    for T, fm in ((8, r["flush_min_t8"]), (4, r["flush_min_t4"])):
        assert fm == r["default_width"] + 1 - T  # fold exactly when history + T would overflow W16
        assert (fm - 1) + T <= r["default_width"] <= r["deep_window_width"]
