"""Pins of the fp64 oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign, index or scale, a transposed operand, a leaky mask, a wrong KV
group) fails at least one of them:

* central finite differences of L = <Y, dY>         -> every analytic gradient
* softmax rows sum to one, masked entries exactly 0 -> normaliser and mask
* torch CPU fp64 scaled_dot_product_attention (causal, GQA) with autograd
                                                    -> forward, lse and backward
* closed-form special cases (S = 1, W_q = 0 cumulative mean, MHA, MQA)
* staged == plain for every U | H, C | U, both schedules (U = H is Ulysses)
"""
import itertools

import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import LayerShape, layer_inputs, bf16_bits_to_f64


def _rand_layer(S, d_model, H, G, d, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((S, d_model))
    W_qkv = rng.standard_normal((d_model, (H + 2 * G) * d)) / np.sqrt(d_model)
    W_o = rng.standard_normal((H * d, d_model)) / np.sqrt(d_model)
    dY = rng.standard_normal((S, d_model))
    return X, W_qkv, W_o, dY


# --------------------------------------------------------------------------
# finite differences: brute force on tiny shapes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("H,G", [(4, 2), (4, 1), (4, 4)])
def test_gradients_match_central_differences(H, G):
    S, d_model, d = 12, 16, 4
    X, W_qkv, W_o, dY = _rand_layer(S, d_model, H, G, d, seed=H * 10 + G)

    def loss(X_, Wqkv_, Wo_):
        return float((orc.layer_forward(X_, Wqkv_, Wo_, H, G, d)[0] * dY).sum())

    dX, dW_qkv, dW_o = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    eps = 1e-6
    for name, arr, grad in (("X", X, dX), ("W_qkv", W_qkv, dW_qkv), ("W_o", W_o, dW_o)):
        num = np.zeros_like(arr)
        for idx in itertools.product(*map(range, arr.shape)):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss(X, W_qkv, W_o)
            arr[idx] = old - eps
            lm = loss(X, W_qkv, W_o)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        rel = np.linalg.norm(num - grad) / np.linalg.norm(num)
        assert rel < 1e-6, (name, rel)


# --------------------------------------------------------------------------
# softmax normaliser and causal mask
# --------------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_mask_is_exact():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((37, 8)) * 3 for _ in range(3))
    o, lse, P = orc.attention_head_forward(q, k, v)
    assert np.abs(P.sum(axis=1) - 1).max() < 1e-12
    assert np.all(P[np.triu_indices(37, k=1)] == 0.0)
    assert np.all(P[np.tril_indices(37)] > 0.0)
    # lse is the log of the unnormalised row sum
    A = (q @ k.T) / np.sqrt(8)
    for i in (0, 5, 36):
        assert abs(lse[i] - np.log(np.exp(A[i, :i + 1]).sum())) < 1e-12
    # row 0 sees only key 0
    assert np.allclose(o[0], v[0], atol=0, rtol=1e-15)


# --------------------------------------------------------------------------
# library routine: torch fp64 SDPA with autograd
# --------------------------------------------------------------------------

def _torch_layer(X, W_qkv, W_o, H, G, d, dY):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in (("X", X), ("W_qkv", W_qkv), ("W_o", W_o))}
    S = X.shape[0]
    qkv = t["X"] @ t["W_qkv"]
    q = qkv[:, :H * d].reshape(S, H, d).transpose(0, 1)[None]
    k = qkv[:, H * d:(H + G) * d].reshape(S, G, d).transpose(0, 1)[None]
    v = qkv[:, (H + G) * d:].reshape(S, G, d).transpose(0, 1)[None]
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    O = o[0].transpose(0, 1).reshape(S, H * d)
    Y = O @ t["W_o"]
    (Y * torch.tensor(dY)).sum().backward()
    return (Y.detach().numpy(), O.detach().numpy(), t["X"].grad.numpy(),
            t["W_qkv"].grad.numpy(), t["W_o"].grad.numpy())


@pytest.mark.parametrize("H,G,d", [(8, 2, 16), (6, 3, 8), (4, 4, 8), (4, 1, 8)])
def test_layer_matches_torch_sdpa_fp64(H, G, d):
    S, d_model = 70, 24
    X, W_qkv, W_o, dY = _rand_layer(S, d_model, H, G, d, seed=H + G + d)
    Y_t, O_t, dX_t, dWqkv_t, dWo_t = _torch_layer(X, W_qkv, W_o, H, G, d, dY)
    Y, O, lse = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    dX, dW_qkv, dW_o = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    for a, b in ((Y, Y_t), (O, O_t), (dX, dX_t), (dW_qkv, dWqkv_t), (dW_o, dWo_t)):
        assert np.linalg.norm(a - b) <= 1e-12 * np.linalg.norm(b)


# --------------------------------------------------------------------------
# closed forms and degenerate cases
# --------------------------------------------------------------------------

def test_single_token_output_is_sum_of_value_projections():
    H, G, d, d_model = 6, 2, 4, 10
    X, W_qkv, W_o, _ = _rand_layer(1, d_model, H, G, d, seed=11)
    Y, _, lse = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    _, _, Wv = orc.split_w_qkv(W_qkv, H, G, d)
    want = sum((X @ Wv[h // (H // G)]) @ W_o[h * d:(h + 1) * d] for h in range(H))
    assert np.allclose(Y, want, rtol=1e-13, atol=1e-13)
    # one visible key: lse equals that single score
    Wq, Wk, _ = orc.split_w_qkv(W_qkv, H, G, d)
    s = float(((X @ Wq[1]) @ (X @ Wk[0]).T)[0, 0]) / np.sqrt(d)
    assert abs(lse[1, 0] - s) < 1e-12


def test_zero_query_weights_give_cumulative_means():
    S, d_model, H, G, d = 9, 8, 4, 2, 4
    X, W_qkv, W_o, _ = _rand_layer(S, d_model, H, G, d, seed=5)
    W_qkv[:, :H * d] = 0.0
    _, O, lse = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    _, _, Wv = orc.split_w_qkv(W_qkv, H, G, d)
    for h in range(H):
        V = X @ Wv[h // (H // G)]
        cm = np.cumsum(V, axis=0) / np.arange(1, S + 1)[:, None]
        assert np.allclose(O[:, h * d:(h + 1) * d], cm, rtol=1e-13, atol=1e-13)
        assert np.allclose(lse[h], np.log(np.arange(1, S + 1)), rtol=0, atol=1e-13)


def test_mha_and_mqa_groupings():
    # G = H: head h uses KV head h; G = 1: every head uses KV head 0.
    assert [orc.kv_head(h, 8, 8) for h in range(8)] == list(range(8))
    assert [orc.kv_head(h, 8, 1) for h in range(8)] == [0] * 8
    assert [orc.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    # MQA layer equals MHA layer whose KV weights are G copies of one head
    S, d_model, H, d = 10, 8, 4, 4
    X, W1, W_o, _ = _rand_layer(S, d_model, H, 1, d, seed=7)
    Wq, Wk, Wv = orc.split_w_qkv(W1, H, 1, d)
    W4 = np.concatenate(Wq + Wk * H + Wv * H, axis=1)
    assert np.allclose(orc.layer_forward(X, W1, W_o, H, 1, d)[0],
                       orc.layer_forward(X, W4, W_o, H, H, d)[0], rtol=1e-13, atol=1e-13)


def test_sampled_rows_equal_full_forward():
    S, d_model, H, G, d = 40, 12, 4, 2, 4
    X, W_qkv, W_o, _ = _rand_layer(S, d_model, H, G, d, seed=9)
    Y, O, lse = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    rows = [0, 3, 17, 39]
    Yr, Or, lser = orc.layer_forward_rows(X, W_qkv, W_o, H, G, d, rows)
    assert np.allclose(Yr, Y[rows], rtol=1e-13, atol=1e-13)
    assert np.allclose(lser, lse[:, rows], rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# the method is exact: staged == plain for every U and both schedules
# --------------------------------------------------------------------------

def _valid_u_c(H, G, S):
    for U in range(1, H + 1):
        if H % U:
            continue
        for C in range(1, U + 1):
            if U % C or S % C:
                continue
            for order in (orc.IN_ORDER, orc.GQA_OUT_OF_ORDER):
                if order == orc.GQA_OUT_OF_ORDER and not (G % C == 0 or C % G == 0):
                    continue
                yield U, C, order


@pytest.mark.parametrize("H,G", [(8, 2), (4, 4), (4, 1), (8, 4)])
def test_staged_equals_plain_for_every_u(H, G):
    S, d_model, d = 16, 8, 4
    X, W_qkv, W_o, dY = _rand_layer(S, d_model, H, G, d, seed=H * 3 + G)
    Y, O, lse = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    dX, dW_qkv, dW_o = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    seen = 0
    for U, C, order in _valid_u_c(H, G, S):
        Ys, Os, lses = orc.staged_forward(X, W_qkv, W_o, H, G, d, U, C, order)
        assert np.linalg.norm(Ys - Y) <= 1e-12 * np.linalg.norm(Y), (U, C, order)
        assert np.array_equal(Os, O) or np.allclose(Os, O, rtol=1e-13, atol=1e-13)
        assert np.allclose(lses, lse, rtol=1e-13, atol=1e-13)
        g = orc.staged_backward(X, W_qkv, W_o, H, G, d, U, C, dY, Os, lses, order)
        for a, b in zip(g, (dX, dW_qkv, dW_o)):
            assert np.linalg.norm(a - b) <= 1e-12 * np.linalg.norm(b), (U, C, order)
        seen += 1
    assert seen >= 4


def test_ulysses_is_the_single_stage_case():
    H, G, S, d_model, d = 8, 2, 16, 8, 4
    X, W_qkv, W_o, _ = _rand_layer(S, d_model, H, G, d, seed=2)
    assert orc.stage_heads(H, G, H, 4).shape == (1, 4, 2)
    Y1 = orc.staged_forward(X, W_qkv, W_o, H, G, d, H, 4)[0]
    assert np.allclose(Y1, orc.layer_forward(X, W_qkv, W_o, H, G, d)[0], rtol=1e-13, atol=1e-13)


def test_tiny_workload_bf16_inputs_staged_equals_plain():
    sh = LayerShape(S=64, d_model=32, H=8, G=2, d_head=8, U=2, C=2)
    inp = layer_inputs(sh, seed=0)
    X, W_qkv, W_o, dY = (bf16_bits_to_f64(inp[k]) for k in ("X", "W_qkv", "W_o", "dY"))
    Y = orc.layer_forward(X, W_qkv, W_o, sh.H, sh.G, sh.d_head)[0]
    for order in (orc.IN_ORDER, orc.GQA_OUT_OF_ORDER):
        Ys = orc.staged_forward(X, W_qkv, W_o, sh.H, sh.G, sh.d_head, sh.U, sh.C, order)[0]
        assert np.linalg.norm(Ys - Y) <= 1e-12 * np.linalg.norm(Y)


def test_attention_rows_match_the_whole_head():
    """The row-wise forward and dQ (used to check full-size launches on sampled
    rows) against the whole-head oracle."""
    rng = np.random.default_rng(9)
    S, d = 48, 8
    q, k, v, do = (rng.standard_normal((S, d)) for _ in range(4))
    o, l, P = orc.attention_head_forward(q, k, v)
    dq, _, _ = orc.attention_head_backward(q, k, v, P, o, do)
    rows = [0, 1, 17, 47]
    ro, rl, rdq = orc.attention_rows(q, k, v, do, rows)
    assert np.abs(ro - o[rows]).max() < 1e-13 and np.abs(rl - l[rows]).max() < 1e-13
    assert np.abs(rdq - dq[rows]).max() < 1e-13


def test_layer_backward_rows_match_the_whole_layer():
    """The row-wise dX (used to check full-size backward launches on the last
    rows) against the whole-layer oracle on every row of a small case."""
    rng = np.random.default_rng(10)
    S, dm, H, G, d = 24, 10, 4, 2, 6
    X = rng.standard_normal((S, dm))
    W_qkv = rng.standard_normal((dm, (H + 2 * G) * d)) / np.sqrt(dm)
    W_o = rng.standard_normal((H * d, dm)) / np.sqrt(dm)
    dY = rng.standard_normal((S, dm))
    dX, _, _ = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    for rows in ([S - 1], [S - 1, S - 2, 17], [0, 5, S - 1]):
        got = orc.layer_backward_rows(X, W_qkv, W_o, H, G, d, dY, rows)
        assert np.abs(got - dX[rows]).max() < 1e-12


# --------------------------------------------------------------------------
# the backward for an upstream gradient that is zero outside a few rows
# --------------------------------------------------------------------------

@pytest.mark.parametrize("H,G,rows", [(4, 2, [0, 7, 8, 25, 39]), (4, 4, [39]), (4, 1, [0]),
                                      (6, 3, [3, 4, 5, 17, 30, 31])])
def test_sparse_dy_backward_is_the_whole_layer_backward(H, G, rows):
    """layer_backward_sparse_dy leaves out only the rows where dY is zero:
    it must equal the whole-layer backward (pinned by finite differences
    above) run on dY zeroed outside those rows, for every output."""
    S, d_model, d = 40, 16, 4
    X, W_qkv, W_o, dY = _rand_layer(S, d_model, H, G, d, seed=len(rows) + H)
    rows = np.array(rows)
    dY_sparse = np.zeros_like(dY)
    dY_sparse[rows] = dY[rows]
    want = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY_sparse)
    got = orc.layer_backward_sparse_dy(X, W_qkv, W_o, H, G, d, dY[rows], rows)
    for name, a, b in zip(("dX", "dW_qkv", "dW_o"), got, want):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max()), name
    # the K/V gradients reach every key row up to the last listed query, and
    # rows of dX below it are nonzero although dY is zero there
    assert rows.max() == 0 or np.abs(got[0][: rows.max()]).max() > 0


# --------------------------------------------------------------------------
# fp32 sum of a KV head's gradient copies, in rank order
# --------------------------------------------------------------------------

def test_replica_gradient_sum_order_and_rounding():
    e = 2.0 ** -24  # half an fp32 unit at 1.0
    # left to right: 1 + e rounds back to 1 (tie, even), twice
    s32, r = orc.replica_gradient_sum([[1.0], [e], [e]])
    assert s32[0] == np.float32(1.0)
    # the small copies first: e + e = 2e, then 1 + 2e is exact in fp32
    s32, r = orc.replica_gradient_sum([[e], [e], [1.0]])
    assert s32[0] == np.float32(1.0 + 2 * e)
    # one copy: just its bf16 rounding; ties go to the even mantissa
    for x, want in ((1.0 + 2.0 ** -8, 1.0), (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6), (-(1.0 + 2.0 ** -8), -1.0),
                    (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7)):
        s32, r = orc.replica_gradient_sum([[x]])
        assert r[0] == want, (x, r[0], want)
    # small integers add exactly in any order
    rng = np.random.default_rng(5)
    c = rng.integers(-50, 50, size=(8, 3, 4)).astype(np.float32)
    s32, r = orc.replica_gradient_sum(c)
    assert np.array_equal(s32, c.sum(axis=0)) and np.array_equal(r, c.sum(axis=0).astype(np.float64))
