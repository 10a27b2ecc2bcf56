"""Pins of the oracle's head stages combined with sequence chunks.

Chunking the sequence only regroups the work: with the online merge of
partial softmax results the chunked layer must equal the plain definition
(which is pinned by finite differences and by torch's SDPA elsewhere) for
every U, C and chunk count, up to fp64 rounding.  Planted slips in the chunk
mask or in the merge must break that equality.
"""
import numpy as np
import pytest

from oracle import upipe_oracle as orc


def _layer(S=32, d_model=12, H=4, G=2, d=8, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((S, d_model))
    W_qkv = rng.standard_normal((d_model, (H + 2 * G) * d)) / np.sqrt(d_model)
    W_o = rng.standard_normal((H * d, d_model)) / np.sqrt(d_model)
    dY = rng.standard_normal((S, d_model))
    return X, W_qkv, W_o, dY


def _gaps(H, G, d, U, C, n, S=32, d_model=12):
    X, W_qkv, W_o, dY = _layer(S, d_model, H, G, d)
    ref_f = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    ref_b = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    Y, O, lse = orc.chunked_forward(X, W_qkv, W_o, H, G, d, U, C, n)
    got_b = orc.chunked_backward(X, W_qkv, W_o, H, G, d, U, C, n, dY, O, lse)
    return [float(np.abs(a - b).max() / np.abs(b).max()) for a, b in zip((Y, O, lse) + got_b, ref_f + ref_b)]


@pytest.mark.parametrize("H,G,U,C,n", [(4, 2, 4, 2, 1), (4, 2, 2, 2, 2), (4, 2, 2, 1, 4), (4, 2, 1, 1, 8),
                                       (4, 2, 4, 4, 2), (8, 2, 4, 2, 4), (8, 2, 2, 2, 16), (4, 4, 2, 2, 4),
                                       (4, 1, 2, 2, 2)])
def test_chunked_layer_equals_the_definition(H, G, U, C, n):
    assert max(_gaps(H, G, 8, U, C, n)) < 1e-12


def test_merge_of_two_key_sets_is_the_softmax_over_their_union():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((5, 7)) * 4
    v = rng.standard_normal((7, 3))
    full = np.exp(a - a.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    parts = []
    for cols in (slice(0, 3), slice(3, 7)):
        s = a[:, cols]
        m = s.max(1, keepdims=True)
        e = np.exp(s - m)
        parts.append(((e / e.sum(1, keepdims=True)) @ v[cols], (m + np.log(e.sum(1, keepdims=True)))[:, 0]))
    o, lse = orc.merge_partials(*parts[0], *parts[1])
    assert np.abs(o - full @ v).max() < 1e-13
    assert np.abs(lse - np.log(np.exp(a).sum(1))).max() < 1e-13
    o2, lse2 = orc.merge_partials(*parts[1], *parts[0])
    assert np.abs(o2 - o).max() < 1e-13 and np.abs(lse2 - lse).max() < 1e-13


def test_chunk_scores_mask_by_sequence_position():
    q = np.ones((4, 2))
    k = np.ones((4, 2))
    A = orc.chunk_scores(q, k, 4, 0)      # every key before every query
    assert np.isfinite(A).all()
    A = orc.chunk_scores(q, k, 4, 4)      # the diagonal block: causal
    assert (np.isinf(A) == (np.arange(4)[None, :] > np.arange(4)[:, None])).all()
    A = orc.chunk_scores(q, k, 4, 6)      # keys 6..9 against queries 4..7
    assert (np.isinf(A) == (6 + np.arange(4)[None, :] > 4 + np.arange(4)[:, None])).all()


def test_chunk_count_must_split_ranks_evenly():
    X, W_qkv, W_o, _ = _layer()
    with pytest.raises(ValueError):
        orc.chunked_forward(X, W_qkv, W_o, 4, 2, 8, 2, 2, 3)
    with pytest.raises(ValueError):
        orc.chunked_forward(X, W_qkv, W_o, 4, 2, 8, 4, 4, 16)  # 2 rows per chunk, 4 ranks


def _local_mask(q, k, q_pos, k_pos):
    A = (q @ k.T) / np.sqrt(q.shape[1])
    A[np.triu_indices(q.shape[0], k=1)] = -np.inf
    return A


def _swapped_offsets(q, k, q_pos, k_pos):
    A = (q @ k.T) / np.sqrt(q.shape[1])
    qi = k_pos + np.arange(q.shape[0])[:, None]
    kj = q_pos + np.arange(k.shape[0])[None, :]
    A[kj > qi] = -np.inf
    A[:, 0] = np.where(np.isinf(A).all(1), 0.0, A[:, 0])
    return A


def _plain_average(o_a, lse_a, o_b, lse_b):
    return 0.5 * (o_a + o_b), np.logaddexp(lse_a, lse_b)


def _unshifted_weights(o_a, lse_a, o_b, lse_b):
    lse = np.logaddexp(lse_a, lse_b)
    return o_a * np.exp(lse_a)[:, None] + o_b * np.exp(lse_b)[:, None], lse


@pytest.mark.parametrize("name,fn", [("chunk_scores", _local_mask), ("chunk_scores", _swapped_offsets),
                                     ("merge_partials", _plain_average), ("merge_partials", _unshifted_weights)])
def test_planted_chunking_slips_fail_the_pin(monkeypatch, name, fn):
    monkeypatch.setattr(orc, name, fn)
    assert max(_gaps(4, 2, 8, 2, 2, 4)) > 1e-3
