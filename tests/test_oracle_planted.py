"""Plant plausible mistakes in the oracle (on the CPU, via monkeypatch) and
check that the pins catch each one.  This shows the pins can fail."""
import numpy as np
import pytest

from oracle import upipe_oracle as orc
from tests.test_oracle_pins import _rand_layer, _torch_layer


def _sdpa_gap(H=4, G=2, d=8):
    S, d_model = 20, 12
    X, W_qkv, W_o, dY = _rand_layer(S, d_model, H, G, d, seed=1)
    Y_t, _, dX_t, dWqkv_t, dWo_t = _torch_layer(X, W_qkv, W_o, H, G, d, dY)
    Y = orc.layer_forward(X, W_qkv, W_o, H, G, d)[0]
    dX, dW_qkv, dW_o = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    return max(np.linalg.norm(a - b) / np.linalg.norm(b)
               for a, b in ((Y, Y_t), (dX, dX_t), (dW_qkv, dWqkv_t), (dW_o, dWo_t)))


def _fd_gap():
    H, G, d, S, d_model = 2, 1, 4, 6, 5
    X, W_qkv, W_o, dY = _rand_layer(S, d_model, H, G, d, seed=2)
    dX = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)[0]
    num = np.zeros_like(X)
    for i in range(S):
        for j in range(d_model):
            o = X[i, j]
            X[i, j] = o + 1e-6
            lp = (orc.layer_forward(X, W_qkv, W_o, H, G, d)[0] * dY).sum()
            X[i, j] = o - 1e-6
            lm = (orc.layer_forward(X, W_qkv, W_o, H, G, d)[0] * dY).sum()
            X[i, j] = o
            num[i, j] = (lp - lm) / 2e-6
    return np.linalg.norm(num - dX) / np.linalg.norm(num)


def test_unplanted_oracle_passes_both_pins():
    assert _sdpa_gap() < 1e-12
    assert _fd_gap() < 1e-6


def _no_mask(q, k):
    return (q @ k.T) / np.sqrt(q.shape[1])


def _wrong_scale(q, k):
    A = (q @ k.T) / q.shape[1]
    A[np.triu_indices(q.shape[0], k=1)] = -np.inf
    return A


def _strict_mask(q, k):
    A = (q @ k.T) / np.sqrt(q.shape[1])
    A[np.triu_indices(q.shape[0], k=0)] = -1e300
    A[0, 0] = 0.0
    return A


@pytest.mark.parametrize("fn", [_no_mask, _wrong_scale, _strict_mask])
def test_forward_slips_fail_the_library_pin(monkeypatch, fn):
    monkeypatch.setattr(orc, "causal_scores", fn)
    assert _sdpa_gap() > 1e-3


def test_wrong_kv_grouping_fails_the_library_pin(monkeypatch):
    monkeypatch.setattr(orc, "kv_head", lambda h, H, G: h % G)
    assert _sdpa_gap() > 1e-3


_GOOD_BWD = orc.attention_head_backward


def _bwd_no_D(q, k, v, P, o, do):
    d = q.shape[1]
    dA = P * (do @ v.T)
    return dA @ k / np.sqrt(d), dA.T @ q / np.sqrt(d), P.T @ do


def _bwd_dk_unscaled(q, k, v, P, o, do):
    dq, dk, dv = _GOOD_BWD(q, k, v, P, o, do)
    return dq, dk * np.sqrt(q.shape[1]), dv


def _bwd_dv_transposed(q, k, v, P, o, do):
    dq, dk, dv = _GOOD_BWD(q, k, v, P, o, do)
    return dq, dk, P @ do


@pytest.mark.parametrize("fn", [_bwd_no_D, _bwd_dk_unscaled, _bwd_dv_transposed])
def test_backward_slips_fail_finite_differences(monkeypatch, fn):
    monkeypatch.setattr(orc, "attention_head_backward", fn)
    assert _fd_gap() > 1e-3
