"""The attention backward for callers that cannot allocate device memory.

upipe_attention_bwd_noalloc takes no workspace: its scratch is a fixed array
inside the library, because some callers (engines that reserve all device
memory up front, plugins inside frameworks that forbid allocation on their
call path) have no way to provide one.  These tests call it through the C ABI
twice in a row and check each result against upipe_attention_bwd, which uses
a caller-provided workspace: the two run the same kernels, so dK and dV (each
reduced inside one CTA, in a fixed order) are bit-identical and dQ (added by
reduce-adds whose order varies) agrees within the tolerance the other GPU
tests use.  They also check the result against the fp64 oracle, and run the
largest size the fixed scratch accepts.  This file is collected last, and
also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import normal_bf16, bf16_bits_to_f64
from tests.helpers import to_dev, f64_of, rel

pytestmark = pytest.mark.gpu
TOL = 1e-2
SCRATCH_LIMIT = 1 << 20  # n_q * S the fixed 8 MiB scratch holds (8 bytes per query row)


def _i32(seq):
    return (ctypes.c_int32 * len(seq))(*seq)


def _inputs(n_q, n_kv, S, d, seed):
    return tuple(normal_bf16(shape, seed + i) for i, shape in
                 enumerate(((n_q, S, d), (n_kv, S, d), (n_kv, S, d), (n_q, S, d))))


def _noalloc_twice(up, Q, K, V, O, dO, lse, kv):
    """Two calls in a row into NaN-filled outputs; returns both results."""
    import torch
    lib = up.lib()
    n_q, S, d = Q.shape
    n_kv = K.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    outs = []
    for _ in range(2):
        dQ = torch.full((n_q, S, d), float("nan"), dtype=torch.float32, device="cuda")
        dK = torch.full((n_kv, S, d), float("nan"), dtype=torch.float32, device="cuda")
        dV = torch.full((n_kv, S, d), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.upipe_attention_bwd_noalloc(P(Q), P(K), P(V), P(O), P(dO), P(lse), n_q, n_kv, S, d, _i32(kv),
                                             P(dQ), P(dK), P(dV), stream)
        assert rc == up.OK, lib.upipe_status_str(rc)
        torch.cuda.synchronize()
        up.sync_status()
        outs.append((dQ, dK, dV))
    return outs


@pytest.mark.parametrize("n_q,n_kv,S,d,kv", [(4, 2, 512, 128, [0, 0, 1, 1]), (4, 2, 384, 64, [0, 0, 1, 1]),
                                             (3, 3, 256, 64, [2, 0, 1])])
def test_noalloc_backward_matches_workspace_backward_and_oracle(n_q, n_kv, S, d, kv):
    import torch
    import headwise_chunked_ulysses_gb300 as up
    bits = _inputs(n_q, n_kv, S, d, seed=11 + S + d)
    Q, K, V, dO = (to_dev(x) for x in bits)
    O, lse = up.attention_fwd(Q, K, V, kv)
    want = up.attention_bwd(Q, K, V, O, dO, lse, kv)
    q64, k64, v64, do64 = (bf16_bits_to_f64(x) for x in bits)
    dq_ref = np.zeros_like(q64)
    dk_ref, dv_ref = np.zeros_like(k64), np.zeros_like(v64)
    for h in range(n_q):
        g = kv[h]
        o, _, P = orc.attention_head_forward(q64[h], k64[g], v64[g])
        dq_ref[h], dk, dv = orc.attention_head_backward(q64[h], k64[g], v64[g], P, o, do64[h])
        dk_ref[g] += dk
        dv_ref[g] += dv
    for call, (dQ, dK, dV) in enumerate(_noalloc_twice(up, Q, K, V, O, dO, lse, kv)):
        assert torch.equal(dK, want[1]) and torch.equal(dV, want[2]), call
        assert bool(torch.isfinite(dQ).all()), call
        assert rel(f64_of(dQ), f64_of(want[0])) <= TOL, call
        assert rel(f64_of(dQ), dq_ref) <= TOL, call
        assert rel(f64_of(dK), dk_ref) <= TOL, call
        assert rel(f64_of(dV), dv_ref) <= TOL, call


def test_noalloc_backward_at_the_largest_size_its_scratch_holds():
    """n_q * S exactly at the limit: the last query slot's D and lse entries
    sit at the end of the fixed array."""
    import torch
    import headwise_chunked_ulysses_gb300 as up
    n_q, n_kv, S, d = 64, 8, 16384, 64
    assert n_q * S == SCRATCH_LIMIT
    kv = [h // 8 for h in range(n_q)]
    Q, K, V, dO = (to_dev(x) for x in _inputs(n_q, n_kv, S, d, seed=91))
    O, lse = up.attention_fwd(Q, K, V, kv)
    want = up.attention_bwd(Q, K, V, O, dO, lse, kv)
    for call, (dQ, dK, dV) in enumerate(_noalloc_twice(up, Q, K, V, O, dO, lse, kv)):
        assert torch.equal(dK, want[1]) and torch.equal(dV, want[2]), call
        assert bool(torch.isfinite(dQ).all()), call
        # the last slot, whose scratch entries end the array, on its own
        assert rel(f64_of(dQ[-1]), f64_of(want[0][-1])) <= TOL, call
        assert rel(f64_of(dQ), f64_of(want[0])) <= TOL, call


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    """One query row past the limit, and a larger case: UPIPE_ENOSPC before
    anything is enqueued.  The buffers have the full sizes the shapes name, so
    the call reads nothing out of bounds whatever it does."""
    import torch
    import headwise_chunked_ulysses_gb300 as up
    lib = up.lib()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    d = 64
    for n_q, S in ((1, SCRATCH_LIMIT + 128), (9, 131072)):
        assert n_q * S > SCRATCH_LIMIT
        x = torch.empty(n_q * S * d, dtype=torch.bfloat16, device="cuda")
        f = torch.empty(n_q * S * d, dtype=torch.float32, device="cuda")
        lse = torch.empty(n_q * S, dtype=torch.float32, device="cuda")
        rc = lib.upipe_attention_bwd_noalloc(P(x), P(x), P(x), P(x), P(x), P(lse), n_q, 1, S, d,
                                             _i32([0] * n_q), P(f), P(f), P(f), None)
        assert rc == up.ENOSPC, (n_q, S, rc)
        del x, f, lse
