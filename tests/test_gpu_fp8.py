"""FP8 (E4M3) heads on the GPU against the oracle.

The encoding is bit-exact: both sides decide each code from the same bf16
value in fp32 (scale = amax / 448 and x / scale as IEEE fp32 divisions, round
to nearest even, saturating), so codes and scales must match exactly.  The
FP8 attention is compared with the oracle's FP8 attention (the same codes,
then exact arithmetic) at the layer tolerance, 1e-2.  Against the plain
definition the budget is restated for FP8: E4M3 keeps 3 mantissa bits, a
relative rounding error up to 2^-4 per score operand; the scores average d
such errors and the softmax output averages again, so the outputs of FP8
heads stay within 5e-2 (relative Frobenius) of the bf16-free definition.
"""
import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import LayerShape, SHAPES, layer_inputs, bf16_bits_to_f64, normal_bf16
from tests.helpers import to_dev, f64_of, rel

pytestmark = pytest.mark.gpu
TOL = 1e-2
FP8_BUDGET = 5e-2


@pytest.fixture(scope="module")
def up():
    import headwise_chunked_ulysses_gb300 as u
    u.lib()
    return u


def _decode(codes):
    """E4M3 code bytes -> values: sign bit 7, exponent bits 3..6 (bias 7),
    mantissa bits 0..2; exponent 0 is subnormal."""
    c = codes.astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7.0))
    return sign * mag


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_quantization_is_bit_exact(up, per_row, d):
    import torch
    S, n, stride = 512, 3, 3 * d + 64
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((S, stride)) * np.exp(rng.uniform(-6, 6, (S, 1)))).astype(np.float32)
    x[7] = 0.0                        # an all-zero row (scale 1)
    x[130:140, :d] *= 1e4             # values far above 448 before scaling
    bits = x.view(np.uint32)
    bits = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)  # RNE to bf16
    src = to_dev(bits)
    codes, scales = up.quantize_e4m3(src, S, n, d, stride, per_row)
    torch.cuda.synchronize()
    up.sync_status()
    xs = bf16_bits_to_f64(bits).astype(np.float32)
    got_c = _decode(codes.cpu().numpy())
    got_s = scales.cpu().numpy()
    for h in range(n):
        xh = xs[:, h * d:(h + 1) * d]
        want_c, want_s = orc.fp8_rows(xh) if per_row else orc.fp8_key_blocks(xh)
        assert np.array_equal(got_s[h], want_s)
        assert np.array_equal(got_c[h], want_c)


@pytest.mark.parametrize("n_q,n_kv,S,kv", [(4, 2, 1024, [0, 0, 1, 1]), (2, 2, 384, [1, 0]), (1, 1, 2048, [0])])
def test_fp8_attention_matches_the_oracle(up, n_q, n_kv, S, kv):
    import torch
    d = 128
    Qb = normal_bf16((S, n_q * d), 11)
    Kb = normal_bf16((S, n_kv * d), 12)
    Vb = normal_bf16((n_kv, S, d), 13)
    q8, qs = up.quantize_e4m3(to_dev(Qb), S, n_q, d, n_q * d, True)
    k8, ks = up.quantize_e4m3(to_dev(Kb), S, n_kv, d, n_kv * d, False)
    O, lse = up.attention_fwd_fp8(q8, qs, k8, ks, to_dev(Vb), kv)
    torch.cuda.synchronize()
    up.sync_status()
    q64, k64, v64 = bf16_bits_to_f64(Qb), bf16_bits_to_f64(Kb), bf16_bits_to_f64(Vb)
    for h in range(n_q):
        g = kv[h]
        o, l = orc.attention_head_forward_fp8(q64[:, h * d:(h + 1) * d], k64[:, g * d:(g + 1) * d], v64[g])
        assert rel(f64_of(O[h]), o) <= TOL
        assert np.abs(f64_of(lse[h]) - l).max() < 3e-2
        oo, ll, _ = orc.attention_head_forward(q64[:, h * d:(h + 1) * d], k64[:, g * d:(g + 1) * d], v64[g])
        assert rel(f64_of(O[h]), oo) <= FP8_BUDGET


TINY128 = LayerShape(S=1024, d_model=512, H=4, G=2, d_head=128, U=2, C=2)


@pytest.mark.parametrize("fp8_heads", [set(), {0, 1}, {2, 3}, {0, 1, 2, 3}])
def test_layer_with_fp8_stages(up, fp8_heads):
    import torch
    sh = TINY128
    bits = layer_inputs(sh, 0)
    d = {k: to_dev(v) for k, v in bits.items()}
    f = {k: bf16_bits_to_f64(v) for k, v in bits.items()}
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, 0)
    Y, O, lse, st = up.attn_fwd_fp8(d["X"], d["W_qkv"], d["W_o"], s, fp8_heads)
    torch.cuda.synchronize()
    up.sync_status()
    Y8, O8, l8 = orc.layer_forward_fp8(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, fp8_heads)
    Yd, Od, ld = orc.layer_forward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head)
    assert rel(f64_of(Y), Y8) <= TOL and rel(f64_of(O), O8) <= TOL
    assert np.abs(f64_of(lse) - l8).max() < 3e-2
    assert rel(f64_of(Y), Yd) <= FP8_BUDGET
    if not fp8_heads:  # no FP8 stage: the bf16 forward, bit for bit
        Yb, Ob, lb, _ = up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], s)
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Yb.view(torch.int16)) and torch.equal(lse, lb)
    # the bf16 backward from the FP8 forward's O and lse
    dX, dWq, dWo, _ = up.attn_bwd(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s)
    torch.cuda.synchronize()
    up.sync_status()
    gX, gWq, gWo = orc.layer_backward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, f["dY"])
    for a, b in ((dX, gX), (dWq, gWq), (dWo, gWo)):
        assert rel(f64_of(a), b) <= FP8_BUDGET


def test_llama_widths_4k_all_fp8(up):
    import torch
    sh = SHAPES["llama3_8b_4k"]
    bits = layer_inputs(sh, 0)
    d = {k: to_dev(v) for k, v in bits.items() if k != "dY"}
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, 0)
    Y, O, lse, st = up.attn_fwd_fp8(d["X"], d["W_qkv"], d["W_o"], s, set(range(sh.H)))
    torch.cuda.synchronize()
    up.sync_status()
    f = {k: bf16_bits_to_f64(bits[k]) for k in ("X", "W_qkv", "W_o")}
    Y8, O8, l8 = orc.layer_forward_fp8(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, set(range(sh.H)))
    assert rel(f64_of(Y), Y8) <= TOL and rel(f64_of(O), O8) <= TOL


def test_fp8_argument_errors(up):
    sh = TINY128
    bits = layer_inputs(sh, 0)
    d = {k: to_dev(v) for k, v in bits.items()}
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, 0)
    with pytest.raises(up.UpipeError) as e:
        up.attn_fwd_fp8(d["X"], d["W_qkv"], d["W_o"], s, {0})  # half of stage 0
    assert e.value.code == up.EINVAL
    t = SHAPES["tiny"]  # d_head 64
    tb = layer_inputs(t, 0)
    td = {k: to_dev(v) for k, v in tb.items()}
    ts = up.Shape(t.S, t.d_model, t.H, t.G, t.d_head, t.U, t.C, 0)
    with pytest.raises(up.UpipeError) as e:
        up.attn_fwd_fp8(td["X"], td["W_qkv"], td["W_o"], ts, {0, 1})
    assert e.value.code == up.EUNSUPPORTED


# ---------------------------------------------------------------------------
# the FP8 backward: the exact gradient of the FP8-scored attention in its
# dequantized operands (straight-through for the rounding), as the oracle's
# attention_head_backward_fp8 / layer_backward_fp8 define it
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n_q,n_kv,S,kv", [(4, 2, 1024, [0, 0, 1, 1]), (2, 2, 384, [1, 0]), (3, 1, 256, [0, 0, 0])])
def test_fp8_attention_backward_matches_the_oracle(up, n_q, n_kv, S, kv):
    import torch
    d = 128
    Qb = normal_bf16((S, n_q * d), 21)
    Kb = normal_bf16((S, n_kv * d), 22)
    Vb = normal_bf16((n_kv, S, d), 23)
    dOb = normal_bf16((n_q, S, d), 24)
    q8, qs = up.quantize_e4m3(to_dev(Qb), S, n_q, d, n_q * d, True)
    k8, ks = up.quantize_e4m3(to_dev(Kb), S, n_kv, d, n_kv * d, False)
    V, dO = to_dev(Vb), to_dev(dOb)
    O, lse = up.attention_fwd_fp8(q8, qs, k8, ks, V, kv)
    dQ, dK, dV = up.attention_bwd_fp8(q8, qs, k8, ks, V, O, dO, lse, kv)
    torch.cuda.synchronize()
    up.sync_status()
    q64, k64, v64, do64 = (bf16_bits_to_f64(x) for x in (Qb, Kb, Vb, dOb))
    dK_ref, dV_ref = np.zeros((n_kv, S, d)), np.zeros((n_kv, S, d))
    for h in range(n_q):
        g = kv[h]
        dq, dk, dv = orc.attention_head_backward_fp8(q64[:, h * d:(h + 1) * d], k64[:, g * d:(g + 1) * d], v64[g],
                                                     do64[h])
        assert rel(f64_of(dQ[h]), dq) <= TOL, ("dQ", h)
        dK_ref[g] += dk
        dV_ref[g] += dv
    for g in range(n_kv):
        assert rel(f64_of(dK[g]), dK_ref[g]) <= TOL, ("dK", g)
        assert rel(f64_of(dV[g]), dV_ref[g]) <= TOL, ("dV", g)


@pytest.mark.parametrize("fp8_heads", [{0, 1}, {2, 3}, {0, 1, 2, 3}])
def test_layer_backward_with_fp8_stages(up, fp8_heads):
    """The layer backward of FP8 stages against the oracle's FP8 layer
    backward; with every stage FP8 the backward arena shrinks by the codes."""
    import torch
    sh = TINY128
    bits = layer_inputs(sh, 0)
    d = {k: to_dev(v) for k, v in bits.items()}
    f = {k: bf16_bits_to_f64(v) for k, v in bits.items()}
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, 0)
    Y, O, lse, _ = up.attn_fwd_fp8(d["X"], d["W_qkv"], d["W_o"], s, fp8_heads)
    dX, dWq, dWo, stb = up.attn_bwd_fp8(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s, fp8_heads)
    torch.cuda.synchronize()
    up.sync_status()
    want = orc.layer_backward_fp8(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, f["dY"], fp8_heads)
    for name, a, b in zip(("dX", "dW_qkv", "dW_o"), (dX, dWq, dWo), want):
        assert rel(f64_of(a), b) <= TOL, name
    plain = up.bwd_workspace_bytes(s)
    fp8 = up.bwd_workspace_bytes_fp8(s, fp8_heads)
    if len(fp8_heads) == sh.H:
        slot = sh.S * sh.d_head
        assert plain - fp8 >= 2 * sh.U * slot - 8 * sh.U * sh.S - 1024  # Q, K codes: 1 byte instead of 2
    else:
        assert fp8 == plain


def test_llama_widths_4k_all_fp8_backward(up):
    import torch
    sh = SHAPES["llama3_8b_4k"]
    bits = layer_inputs(sh, 0)
    d = {k: to_dev(v) for k, v in bits.items()}
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, 0)
    heads = set(range(sh.H))
    Y, O, lse, _ = up.attn_fwd_fp8(d["X"], d["W_qkv"], d["W_o"], s, heads)
    dX, dWq, dWo, stb = up.attn_bwd_fp8(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s, heads)
    torch.cuda.synchronize()
    up.sync_status()
    f = {k: bf16_bits_to_f64(v) for k, v in bits.items()}
    want = orc.layer_backward_fp8(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, f["dY"], heads)
    for name, a, b in zip(("dX", "dW_qkv", "dW_o"), (dX, dWq, dWo), want):
        assert rel(f64_of(a), b) <= TOL, name
    _, _, _, stp = up.attn_bwd(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s)
    assert stb["arena_peak_bytes"] < stp["arena_peak_bytes"]
