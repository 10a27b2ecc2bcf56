"""The attention backward for callers that cannot allocate device memory.

upipe_attention_bwd_noalloc takes no workspace: its scratch is a fixed array
inside the library, because some callers (engines that reserve all device
memory up front, plugins inside frameworks that forbid allocation on their
call path) have no way to provide one.  This test calls it through the C ABI
twice in a row and checks each result against upipe_attention_bwd, which
uses a caller-provided workspace, within the tolerance the other GPU tests
use.  It lives in its own file, collected last, and also passes on its own
in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from synthetic import normal_bf16
from tests.helpers import to_dev, f64_of, rel

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _i32(seq):
    return (ctypes.c_int32 * len(seq))(*seq)


def test_noalloc_backward_matches_workspace_backward_twice():
    import torch
    import headwise_chunked_ulysses_gb300 as up
    lib = up.lib()
    n_q, n_kv, S, d = 4, 2, 512, 128
    kv = [0, 0, 1, 1]
    Q, K, V, dO = (to_dev(normal_bf16(shape, seed)) for shape, seed in
                   (((n_q, S, d), 11), ((n_kv, S, d), 12), ((n_kv, S, d), 13), ((n_q, S, d), 14)))
    O, lse = up.attention_fwd(Q, K, V, kv)
    want = [f64_of(x) for x in up.attention_bwd(Q, K, V, O, dO, lse, kv)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    for call in range(2):
        dQ = torch.full((n_q, S, d), float("nan"), dtype=torch.float32, device="cuda")
        dK = torch.full((n_kv, S, d), float("nan"), dtype=torch.float32, device="cuda")
        dV = torch.full((n_kv, S, d), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.upipe_attention_bwd_noalloc(P(Q), P(K), P(V), P(O), P(dO), P(lse), n_q, n_kv, S, d, _i32(kv),
                                             P(dQ), P(dK), P(dV), stream)
        assert rc == up.OK, lib.upipe_status_str(rc)
        torch.cuda.synchronize()
        up.sync_status()
        for got, ref, name in zip((dQ, dK, dV), want, ("dQ", "dK", "dV")):
            g = f64_of(got)
            assert np.isfinite(g).all(), (call, name)
            assert rel(g, ref) <= TOL, (call, name)


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    import torch
    import headwise_chunked_ulysses_gb300 as up
    lib = up.lib()
    n_q, S, d = 9, 131072, 64  # 8 * 9 * 131072 bytes > 8 MiB
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(16, dtype=torch.float32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.upipe_attention_bwd_noalloc(P(x), P(x), P(x), P(x), P(x), P(f), n_q, 1, S, d, _i32([0] * n_q),
                                         P(f), P(f), P(f), None)
    assert rc == up.ENOSPC
