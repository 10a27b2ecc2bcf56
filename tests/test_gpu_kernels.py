"""Parity of the individual CUDA kernels, called through the C ABI.

* the Ulysses exchange (seq->head, head->seq): bit-exact against the oracle's
  all-to-all of C virtual ranks;
* the tensor-core contraction in all four operand layouts and four output
  modes (incl. split-K with atomic partial sums over K ranges of equal and
  unequal length), on one SM and on CTA pairs (M and N multiples of 256):
  against an fp64 product of the same bf16 operands;
* causal GQA attention forward and backward: against the oracle's attention
  core (fp64), per head; dK, dV summed over the query heads of each group.
"""
import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import normal_bf16, bf16_bits_to_f64
from tests.helpers import to_dev, bits_of, f64_of, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def up():
    import torch
    import headwise_chunked_ulysses_gb300 as u
    u.lib()
    assert torch.cuda.is_available()
    return u


# ---------------------------------------------------------------------------
# exchange
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,n_heads,d,C,pad", [(1024, 8, 64, 2, 0), (384, 6, 128, 3, 0), (256, 4, 64, 4, 64),
                                               (512, 12, 128, 4, 128), (96, 3, 64, 3, 0)])
def test_exchange_is_bit_exact(up, S, n_heads, d, C, pad):
    import torch
    rng = np.random.default_rng(S + n_heads + d + C)
    ld = n_heads * d + pad
    src_bits = rng.integers(0, 1 << 16, size=(S, ld), dtype=np.uint16)
    src = to_dev(src_bits)
    dst = torch.empty(n_heads, S, d, dtype=torch.bfloat16, device="cuda")
    up.layout_seq2head(src, dst, S, n_heads, d, C, ld)
    got = bits_of(dst)
    Sc = S // C
    shards = [{h: src_bits[c * Sc:(c + 1) * Sc, h * d:(h + 1) * d] for h in range(n_heads)} for c in range(C)]
    per = n_heads // C
    wanted = [list(range(r * per, (r + 1) * per)) for r in range(C)]
    held = orc.seq_to_head(shards, wanted)
    want = np.concatenate(held, axis=0)
    assert np.array_equal(got, want)
    # and back: every head lands in its columns, padding untouched
    back_bits = rng.integers(0, 1 << 16, size=(S, ld), dtype=np.uint16)
    back = to_dev(back_bits)
    up.layout_head2seq(dst, back, S, n_heads, d, C, ld)
    got_back = bits_of(back)
    assert np.array_equal(got_back[:, :n_heads * d], src_bits[:, :n_heads * d])
    assert np.array_equal(got_back[:, n_heads * d:], back_bits[:, n_heads * d:])


# ---------------------------------------------------------------------------
# contraction
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(256, 384, 320), (128, 512, 128), (384, 64, 192), (256, 256, 1024),
                                   (128, 256, 8192), (512, 512, 512), (768, 1280, 576), (256, 256, 16384),
                                   # M a multiple of 64 only: a last row tile of 64 rows
                                   (64, 256, 192), (192, 384, 320), (320, 1536, 8192),
                                   # split-K ranges of unequal length (on 152 SMs: 2 splits over 21
                                   # K blocks on one SM; 8 and 7 splits over 65 on CTA pairs)
                                   (128, 768, 1344), (256, 512, 4160), (1280, 512, 4160),
                                   # CTA pairs on 152 SMs: 80 tiles, a second round of 4
                                   (5120, 1024, 128)])
@pytest.mark.parametrize("a_trans,b_trans", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_layouts_and_modes(up, M, N, K, a_trans, b_trans):
    import torch
    seed = M + N + K + 10 * a_trans + 20 * b_trans
    A_bits = normal_bf16((K, M) if a_trans else (M, K), seed)
    B_bits = normal_bf16((N, K) if b_trans else (K, N), seed + 1)
    A64, B64 = bf16_bits_to_f64(A_bits), bf16_bits_to_f64(B_bits)
    want = (A64.T if a_trans else A64) @ (B64.T if b_trans else B64)
    A, B = to_dev(A_bits), to_dev(B_bits)
    # fp32 accumulation: rounding error grows like sqrt(K)
    tol32 = 1e-5 * max(1.0, np.sqrt(K / 1024))
    D32 = up.gemm(A, B, M, N, K, a_trans, b_trans, out_mode=1)
    assert rel(f64_of(D32), want) < tol32
    D16 = up.gemm(A, B, M, N, K, a_trans, b_trans, out_mode=0)
    assert rel(f64_of(D16), want) < 1e-2
    base = torch.randn(M, N, dtype=torch.float32, device="cuda")
    base0 = f64_of(base)
    up.gemm(A, B, M, N, K, a_trans, b_trans, out_mode=2, D=base)
    assert rel(f64_of(base), base0 + want) < tol32
    base = torch.randn(M, N, dtype=torch.float32, device="cuda")
    base0 = f64_of(base)
    up.gemm(A, B, M, N, K, a_trans, b_trans, out_mode=3, D=base)  # split-K, atomic partial sums
    assert rel(f64_of(base), base0 + want) < tol32
    up.sync_status()


# ---------------------------------------------------------------------------
# attention core
# ---------------------------------------------------------------------------

def _attn_inputs(n_q, n_kv, S, d, seed):
    Q = normal_bf16((n_q, S, d), seed)
    K = normal_bf16((n_kv, S, d), seed + 1)
    V = normal_bf16((n_kv, S, d), seed + 2)
    dO = normal_bf16((n_q, S, d), seed + 3)
    return Q, K, V, dO


CASES = [(4, 2, 384, 64, [0, 0, 1, 1]), (4, 2, 256, 128, [0, 0, 1, 1]), (2, 2, 1024, 128, [0, 1]),
         (3, 1, 128, 64, [0, 0, 0]), (2, 4, 512, 64, [3, 1]),
         # more than 8 slots: the kernels order their CTAs in groups of 8 slots
         (16, 16, 512, 128, list(range(16))), (16, 8, 384, 64, [k // 2 for k in range(16)])]


@pytest.mark.parametrize("n_q,n_kv,S,d,kv", CASES)
def test_attention_forward_and_backward(up, n_q, n_kv, S, d, kv):
    Qb, Kb, Vb, dOb = _attn_inputs(n_q, n_kv, S, d, seed=S + d + n_q)
    Q, K, V, dO = (to_dev(x) for x in (Qb, Kb, Vb, dOb))
    O, lse = up.attention_fwd(Q, K, V, kv)
    dQ, dK, dV = up.attention_bwd(Q, K, V, O, dO, lse, kv)
    up.sync_status()
    q64, k64, v64, do64 = (bf16_bits_to_f64(x) for x in (Qb, Kb, Vb, dOb))
    Og, lseg, dQg, dKg, dVg = (f64_of(x) for x in (O, lse, dQ, dK, dV))
    dK_ref = np.zeros_like(k64)
    dV_ref = np.zeros_like(v64)
    used = set(kv)
    for h in range(n_q):
        g = kv[h]
        o, l, P = orc.attention_head_forward(q64[h], k64[g], v64[g])
        assert rel(Og[h], o) < 1e-2, ("O", h)
        assert np.abs(lseg[h] - l).max() < 2e-3, ("lse", h)
        dq, dk, dv = orc.attention_head_backward(q64[h], k64[g], v64[g], P, o, do64[h])
        assert rel(dQg[h], dq) < 1e-2, ("dQ", h)
        dK_ref[g] += dk
        dV_ref[g] += dv
    for g in range(n_kv):
        if g in used:
            assert rel(dKg[g], dK_ref[g]) < 1e-2, ("dK", g)
            assert rel(dVg[g], dV_ref[g]) < 1e-2, ("dV", g)
        else:  # a KV slot no query reads has zero gradient
            assert np.all(dKg[g] == 0) and np.all(dVg[g] == 0)


def test_attention_first_row_copies_first_value(up):
    # query 0 sees only key 0: O[0] = V[0] and lse[0] = q0.k0/sqrt(d), whatever the scores
    import torch
    S, d = 256, 128
    Qb, Kb, Vb, _ = _attn_inputs(1, 1, S, d, seed=77)
    O, lse = up.attention_fwd(to_dev(Qb), to_dev(Kb), to_dev(Vb), [0])
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(O)[0, 0], Vb[0, 0])
    s00 = float(bf16_bits_to_f64(Qb)[0, 0] @ bf16_bits_to_f64(Kb)[0, 0]) / np.sqrt(d)
    assert abs(f64_of(lse)[0, 0] - s00) < 1e-4


def test_attention_core_full_size_32k(up):
    """The attention launches of the Llama3-8B layer at S=32768 as the bench
    times them (8 query slots, each with its own KV slot copy, d_head=128):
    O, lse and dQ on sampled rows against the row-wise oracle, and two exact
    identities of the whole backward: per KV slot, the rows of dV sum to the
    sum of dO over its queries (rows of P sum to 1), and the rows of dK sum to
    zero (each row of dS sums to dO.O - D = 0)."""
    import torch
    n, S, d = 8, 32768, 128
    Qb = normal_bf16((n, S, d), 101)
    Kb = normal_bf16((2, S, d), 102)
    Vb = normal_bf16((2, S, d), 103)
    dOb = normal_bf16((n, S, d), 104)
    kv_head = [k // 4 for k in range(n)]
    Kc = np.ascontiguousarray(Kb[kv_head])  # per-slot copies, as the in-order exchange makes them
    Vc = np.ascontiguousarray(Vb[kv_head])
    Q, K, V, dO = (to_dev(x) for x in (Qb, Kc, Vc, dOb))
    O, lse = up.attention_fwd(Q, K, V, list(range(n)))
    dQ, dK, dV = up.attention_bwd(Q, K, V, O, dO, lse, list(range(n)))
    torch.cuda.synchronize()
    up.sync_status()
    rows = np.array([0, 1, 127, 128, 4095, 16384, 32767])
    idx = torch.as_tensor(rows, device="cuda")
    for h in (0, 5):
        q, k, v, do = (bf16_bits_to_f64(x) for x in (Qb[h], Kb[kv_head[h]], Vb[kv_head[h]], dOb[h]))
        o, l, dq = orc.attention_rows(q, k, v, do, rows)
        assert rel(f64_of(O[h][idx]), o) < 1e-2
        assert np.abs(f64_of(lse[h][idx]) - l).max() < 2e-3
        assert rel(f64_of(dQ[h][idx]), dq) < 1e-2
    dVs = dV.double().sum(dim=1).cpu().numpy()
    dKs = dK.double().sum(dim=1).cpu().numpy()
    dKn = dK.double().norm(dim=2).sum(dim=1).cpu().numpy()
    do_sum = bf16_bits_to_f64(dOb).sum(axis=1)
    for k in range(n):
        assert rel(dVs[k], do_sum[k]) < 1e-2
        assert np.linalg.norm(dKs[k]) < 1e-2 * dKn[k]
