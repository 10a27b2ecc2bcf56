"""Pins of the oracle's schedules, all-to-all and memory closed forms.

The memory forms are checked against the values the pages print
(tests/golden/upipe_memory_forms.json, each with its citation); the exchange
is checked against a direct index formula; the schedules against the
properties the pages state (every head once; out of order, all KV heads in
stage 0 and none afterwards).
"""
import json
import os

import numpy as np
import pytest

from oracle import upipe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "upipe_memory_forms.json")


def test_memory_forms_match_printed_values():
    g = json.load(open(GOLDEN))
    S, d = 1 << 20, 128
    q = g["qwen3_32b"]
    H, C, U = q["H"], q["C"], q["U"]
    uly = orc.ulysses_attention_bytes_per_rank(S, C, H, d)
    up = orc.upipe_stage_bytes_per_rank(S, C, U, d)
    assert uly == 96 * S * d
    assert up == 12 * S * d
    assert 100.0 * (1 - up / uly) == q["printed_reduction_percent"]
    # Core method: at U = C the per-device peak is 12*S*d_head whatever H is
    for H2 in (8, 32, 64, 128):
        assert orc.upipe_stage_bytes_per_rank(S, 8, 8, d) == 12 * S * d
    # U = H is plain Ulysses
    assert orc.upipe_stage_bytes_per_rank(S, C, H, d) == uly
    # output buffers (steps 3, 4; d_model read as d_head) are a third of QKV+exchange
    assert 3 * orc.upipe_output_bytes_per_rank(S, C, U, d) == up


@pytest.mark.parametrize("H,G,U,C", [(8, 2, 2, 2), (32, 8, 8, 8), (64, 8, 8, 8), (32, 8, 16, 8),
                                     (32, 8, 32, 8), (12, 3, 6, 3), (8, 2, 8, 4)])
def test_schedules_cover_every_head_once(H, G, U, C):
    for order in (orc.IN_ORDER, orc.GQA_OUT_OF_ORDER):
        if order == orc.GQA_OUT_OF_ORDER and not (G % C == 0 or C % G == 0):
            continue
        s = orc.stage_heads(H, G, U, C, order)
        assert s.shape == (H // U, C, U // C)
        assert sorted(s.ravel().tolist()) == list(range(H))
        if order == orc.IN_ORDER:
            for i in range(H // U):
                assert sorted(s[i].ravel().tolist()) == list(range(i * U, (i + 1) * U))


@pytest.mark.parametrize("H,G,U,C", [(8, 2, 2, 2), (32, 8, 8, 8), (64, 8, 8, 8), (32, 8, 16, 8),
                                     (32, 2, 8, 8), (32, 8, 8, 2)])
def test_out_of_order_moves_each_kv_head_once_in_stage_zero(H, G, U, C):
    o = orc.GQA_OUT_OF_ORDER
    moves = orc.kv_moves(H, G, U, C, o)
    assert {st for st, _, _ in moves} == {0}
    assert {g for _, _, g in moves} == set(range(G))
    # a rank's KV set never changes across stages
    s = orc.stage_heads(H, G, U, C, o)
    for r in range(C):
        kvs = orc.rank_kv_heads(H, G, U, C, r, o)
        for i in range(H // U):
            assert {orc.kv_head(int(h), H, G) for h in s[i, r]} <= set(kvs)
    # one copy per KV head when C | G, C/G copies when G | C
    assert len(moves) == max(G, C)
    # in order, every query slot of every stage receives its KV head
    assert len(orc.kv_moves(H, G, U, C, orc.IN_ORDER)) == H


def test_exchange_is_the_ulysses_index_map_and_round_trips():
    rng = np.random.default_rng(0)
    C, Sc, d, heads = 4, 3, 2, [5, 1, 7, 2, 0, 6, 3, 4]
    S = C * Sc
    shards = [{h: rng.standard_normal((Sc, d)) for h in heads} for _ in range(C)]
    wanted = [heads[2 * r:2 * r + 2] for r in range(C)]
    held = orc.seq_to_head(shards, wanted)
    for r in range(C):
        for j, h in enumerate(wanted[r]):
            for t in range(S):
                assert np.array_equal(held[r][j, t], shards[t // Sc][h][t % Sc])
    back = orc.head_to_seq(held, wanted, S)
    for c in range(C):
        got = dict(back[c])
        assert sorted(got) == sorted(heads)
        for h in heads:
            assert np.array_equal(got[h], shards[c][h])


def test_check_shape_rejects_what_the_method_cannot_run():
    with pytest.raises(ValueError):
        orc.check_shape(16, 8, 8, 2, 4, 3, 1)      # U does not divide H
    with pytest.raises(ValueError):
        orc.check_shape(16, 8, 8, 2, 4, 4, 3)      # C does not divide U
    with pytest.raises(ValueError):
        orc.check_shape(15, 8, 8, 2, 4, 4, 2)      # C does not divide S
    with pytest.raises(ValueError):
        orc.check_shape(16, 8, 8, 3, 4, 4, 2)      # G does not divide H
    with pytest.raises(ValueError):
        orc.check_shape(24, 8, 12, 4, 4, 6, 3, orc.GQA_OUT_OF_ORDER)  # neither C|G nor G|C
    orc.check_shape(1024, 512, 8, 2, 64, 2, 2, orc.GQA_OUT_OF_ORDER)


def test_model_flops_of_the_named_layers():
    # 3x forward; attention is the causal half of the dense S^2 work
    f = orc.layer_model_flops(32768, 4096, 32, 8, 128)
    assert f == 2 * 32768 * 4096 * 6144 + 2 * 32768 * 4096 * 4096 + 2 * 32768 ** 2 * 32 * 128
    assert abs(3 * f / 32768 - 1.057e9) / 1.057e9 < 0.01
