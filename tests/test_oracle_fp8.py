"""Pins of the oracle's FP8 (E4M3) heads.

The E4M3 rounding is pinned to the format's definition (every code decoded
from its bit fields is a fixed point; midpoints go to the even mantissa;
overflow saturates) and to torch's own float8_e4m3fn conversion.  The FP8
attention is pinned to the exact attention when Q and K are already FP8 values
under power-of-two scales, and to the plain layer within the error the
format's 3-bit mantissa allows.  Planted slips (truncation, a wrong exponent
bias, a missing scale) must fail a pin.
"""
import numpy as np
import pytest

from oracle import upipe_oracle as orc


def _all_e4m3_values():
    """Every finite E4M3 value from the bit fields: (-1)^s 2^(e-7) (1 + m/8),
    e = 1..15, with e = 15, m = 7 the NaN; subnormals 2^-6 m/8."""
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            v = 2.0 ** -6 * m / 8 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8)
            vals += [v, -v]
    return np.array(sorted(set(vals)))


def test_every_code_is_a_fixed_point():
    v = _all_e4m3_values()
    assert len(v) == 253  # 2 x 126 nonzero magnitudes + one zero
    assert v.max() == 448.0
    assert np.array_equal(orc.e4m3_round(v), v)


def test_midpoints_round_to_even_and_overflow_saturates():
    v = _all_e4m3_values()
    pos = v[v >= 0]
    mid = (pos[:-1] + pos[1:]) / 2
    got = orc.e4m3_round(mid)
    lo, hi = pos[:-1], pos[1:]
    # the even neighbour has an even mantissa code: its index among positives is even
    idx_lo = np.arange(len(lo))
    want = np.where(idx_lo % 2 == 0, lo, hi)
    assert np.array_equal(got, want)
    assert np.array_equal(orc.e4m3_round(np.array([449.0, 464.0, 1e6, -1e6])), [448.0, 448.0, 448.0, -448.0])
    assert orc.e4m3_round(np.array([2.0 ** -10]))[0] == 0.0  # half the smallest subnormal: to even (0)


def test_rounding_matches_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 in this torch")
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-14, 6, 20000))
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(orc.e4m3_round(x), want)


def test_fp8_attention_is_exact_on_fp8_inputs():
    """Q rows and K blocks whose amax is exactly 448 * 2^k and whose entries are
    E4M3 values times 2^k quantize to themselves: the FP8 attention is then the
    exact attention of those inputs."""
    rng = np.random.default_rng(1)
    v_all = _all_e4m3_values()
    S, d = 256, 16
    q = rng.choice(v_all, size=(S, d)) / 8.0
    k = rng.choice(v_all, size=(S, d)) / 4.0
    q[:, 0] = 448.0 / 8.0
    k[::128, 0] = 448.0 / 4.0
    v = rng.standard_normal((S, d))
    o8, l8 = orc.attention_head_forward_fp8(q, k, v)
    o, l, _ = orc.attention_head_forward(q, k, v)
    assert np.abs(o8 - o).max() < 1e-13 and np.abs(l8 - l).max() < 1e-13


def test_fp8_scales_follow_rows_and_key_blocks():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((256, 8)).astype(np.float32)
    codes, sc = orc.fp8_rows(q)
    assert sc.shape == (256,) and np.abs(codes).max() <= 448
    assert np.allclose(np.abs(codes).max(axis=1), 448.0)  # each row's largest entry maps to the top code
    kc, ks = orc.fp8_key_blocks(q)
    assert ks.shape == (2,)
    assert np.isclose(np.abs(kc[:128]).max(), 448.0) and np.isclose(np.abs(kc[128:]).max(), 448.0)
    z, zs = orc.fp8_rows(np.zeros((4, 8), np.float32))
    assert (z == 0).all() and (zs == 1).all()


def _layer_gap(fp8_heads):
    rng = np.random.default_rng(3)
    S, dm, H, G, d = 256, 32, 4, 2, 16
    X = rng.standard_normal((S, dm))
    W_qkv = rng.standard_normal((dm, (H + 2 * G) * d)) / np.sqrt(dm)
    W_o = rng.standard_normal((H * d, dm)) / np.sqrt(dm)
    Y, O, lse = orc.layer_forward(X, W_qkv, W_o, H, G, d)
    Y8, O8, lse8 = orc.layer_forward_fp8(X, W_qkv, W_o, H, G, d, fp8_heads)
    per_head = [np.linalg.norm(O8[:, h * d:(h + 1) * d] - O[:, h * d:(h + 1) * d]) /
                np.linalg.norm(O[:, h * d:(h + 1) * d]) for h in range(H)]
    return per_head, np.linalg.norm(Y8 - Y) / np.linalg.norm(Y)


def test_fp8_heads_stay_within_the_format_error_and_others_are_untouched():
    per_head, gy = _layer_gap({1, 2})
    assert per_head[0] == 0.0 and per_head[3] == 0.0
    # 3 mantissa bits: relative rounding error <= 2^-4 per entry; the scores'
    # error is an average of d such errors, and softmax and P V average again
    assert 1e-4 < per_head[1] < 5e-2 and 1e-4 < per_head[2] < 5e-2
    assert gy < 5e-2


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-30, 30, 50000))).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]  # ties: to even (down, then up)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_round(x)
    assert np.array_equal(got, want)
    assert got[2] == 1.0 and got[3] == 1.0 + 2.0 ** -6


def _truncate(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
    q = 2.0 ** (e - 3)
    return np.sign(x) * np.minimum(np.floor(a / q) * q, 448.0)


def _wrong_bias(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -7.0)
    q = 2.0 ** (e - 3)
    return np.sign(x) * np.minimum(np.round(a / q) * q, 448.0)


@pytest.mark.parametrize("fn", [_truncate, _wrong_bias])
def test_planted_rounding_slips_fail_the_pins(monkeypatch, fn):
    monkeypatch.setattr(orc, "e4m3_round", fn)
    v = _all_e4m3_values()
    pos = v[v >= 0]
    mid = (pos[:-1] + pos[1:]) / 2
    fixed = np.array_equal(orc.e4m3_round(v), v)
    idx_lo = np.arange(len(mid))
    mids_ok = np.array_equal(orc.e4m3_round(mid), np.where(idx_lo % 2 == 0, pos[:-1], pos[1:]))
    assert not (fixed and mids_ok)


def _scale_gap():
    """Q entries near 3e-3 and K entries near 3e3: without per-group scales Q
    falls into E4M3's subnormals and K saturates at 448."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal((128, 8)) * 3e-3
    k = rng.standard_normal((128, 8)) * 3e3
    v = rng.standard_normal((128, 8))
    o, _, _ = orc.attention_head_forward(q, k, v)
    o8, _ = orc.attention_head_forward_fp8(q, k, v)
    return np.linalg.norm(o8 - o) / np.linalg.norm(o)


def test_scales_keep_small_and_large_heads_in_range():
    assert _scale_gap() < 0.2


def test_planted_missing_scale_fails_the_pin(monkeypatch):
    monkeypatch.setattr(orc, "fp8_scale", lambda amax: np.float32(1.0))
    assert _scale_gap() > 0.5


# ---------------------------------------------------------------------------
# the backward of FP8-scored heads
# ---------------------------------------------------------------------------

def _fp8_valued_qk(S=256, d=16, seed=5):
    """Q rows and K blocks that are E4M3 values times power-of-two scales with
    their amax at 448 x scale: they quantize to themselves."""
    rng = np.random.default_rng(seed)
    v_all = _all_e4m3_values()
    q = rng.choice(v_all, size=(S, d)) / 8.0
    k = rng.choice(v_all, size=(S, d)) / 4.0
    q[:, 0] = 448.0 / 8.0
    k[::128, 0] = 448.0 / 4.0
    return q / 64.0 * 8.0, k / 64.0 * 4.0, rng  # scores of moderate size (scales 2^-6, 2^-6)


def test_fp8_backward_is_the_exact_backward_on_fp8_inputs():
    """On inputs the quantizer leaves unchanged, every FP8 gradient is the
    plain attention gradient of those inputs."""
    q, k, rng = _fp8_valued_qk()
    qd, kd = orc.fp8_dequantized(q, k)
    assert np.array_equal(qd, q) and np.array_equal(kd, k)
    v = rng.standard_normal(q.shape)
    do = rng.standard_normal(q.shape)
    o, _, P = orc.attention_head_forward(q, k, v)
    want = orc.attention_head_backward(q, k, v, P, o, do)
    got = orc.attention_head_backward_fp8(q, k, v, do)
    for a, b in zip(got, want):
        assert np.abs(a - b).max() <= 1e-12 * np.abs(b).max()


def _fp8_backward_fd_gap(seed=6):
    """Largest gap between the FP8 backward and central differences of
    L = <O, dO>: in v directly (v is not quantized), and in the dequantized
    q~, k~ (O is smooth in them) -- the straight-through gradient in q and k is
    the gradient in q~ and k~.  Sampled entries, two key blocks (the second
    one short)."""
    rng = np.random.default_rng(seed)
    S, d = 130, 4
    q, k, v, do = (rng.standard_normal((S, d)) for _ in range(4))
    qd, kd = orc.fp8_dequantized(q, k)
    dq, dk, dv = orc.attention_head_backward_fp8(q, k, v, do)

    def loss(qq, kk, vv):
        return float((orc.attention_head_forward(qq, kk, vv)[0] * do).sum())

    eps, worst = 1e-6, 0.0
    for arr, grad, call in ((v.copy(), dv, lambda a: loss(qd, kd, a)), (qd.copy(), dq, lambda a: loss(a, kd, v)),
                            (kd.copy(), dk, lambda a: loss(qd, a, v))):
        for idx in [(i, j) for i in range(0, S, 7) for j in range(d)]:
            old = arr[idx]
            arr[idx] = old + eps
            lp = call(arr)
            arr[idx] = old - eps
            lm = call(arr)
            arr[idx] = old
            worst = max(worst, abs((lp - lm) / (2 * eps) - grad[idx]) / max(1.0, np.abs(grad).max()))
    return worst


def test_fp8_backward_matches_differences_in_the_dequantized_operands():
    assert _fp8_backward_fd_gap() < 1e-6


def test_fp8_layer_backward_without_fp8_heads_is_the_layer_backward():
    rng = np.random.default_rng(7)
    S, dm, H, G, d = 128, 16, 4, 2, 8
    X = rng.standard_normal((S, dm))
    W_qkv = rng.standard_normal((dm, (H + 2 * G) * d)) / np.sqrt(dm)
    W_o = rng.standard_normal((H * d, dm)) / np.sqrt(dm)
    dY = rng.standard_normal((S, dm))
    want = orc.layer_backward(X, W_qkv, W_o, H, G, d, dY)
    got = orc.layer_backward_fp8(X, W_qkv, W_o, H, G, d, dY, set())
    for a, b in zip(got, want):
        assert np.abs(a - b).max() <= 1e-12 * np.abs(b).max()
    # with FP8 heads the gradients move by about the format's error, no more
    got8 = orc.layer_backward_fp8(X, W_qkv, W_o, H, G, d, dY, {0, 3})
    for a, b in zip(got8, want):
        gap = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert 1e-5 < gap < 5e-2


def test_planted_unquantized_operand_in_the_fp8_backward_fails(monkeypatch):
    """A backward that forms dq~ from the unquantized k instead of k~ (a
    plausible slip) fails the difference pin."""
    plain_backward = orc.attention_head_backward

    def slipped(q_, k_, v_, do_):
        qd, kd = orc.fp8_dequantized(q_, k_)
        o, _, P = orc.attention_head_forward(qd, kd, v_)
        dq, _, _ = plain_backward(qd, k_, v_, P, o, do_)  # k, not k~
        _, dk, dv = plain_backward(qd, kd, v_, P, o, do_)
        return dq, dk, dv

    monkeypatch.setattr(orc, "attention_head_backward_fp8", slipped)
    assert _fp8_backward_fd_gap() > 1e-3


def test_planted_straight_through_on_the_wrong_side_fails(monkeypatch):
    """Differentiating with the unquantized q and k altogether (no FP8 in the
    backward at all) fails the pin on FP8-valued inputs' neighbours too."""
    def slipped(q_, k_, v_, do_):
        o, _, P = orc.attention_head_forward(q_, k_, v_)
        return orc.attention_head_backward(q_, k_, v_, P, o, do_)

    monkeypatch.setattr(orc, "attention_head_backward_fp8", slipped)
    assert _fp8_backward_fd_gap() > 1e-3
