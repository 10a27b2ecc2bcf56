"""Exact checks of the layer's bookkeeping, through the C ABI.

* The backward's reverse exchange sums the gradients of a KV head's copies
  (one per query slot in the in-order exchange) in ascending rank order, in
  fp32, then rounds once to bf16: bit-exact against the oracle's fp32 loop in
  the same order.
* The workspace a layer call touches: every byte of the forward and backward
  workspaces is filled with a sentinel, the call runs, and the highest byte
  that changed (with two different sentinels, so a byte written with the
  sentinel's own value still shows) must be the last byte of the plan, and
  the stage arena's touched bytes must stay within the closed forms.
* The failure detection: a kernel whose bounded wait runs out (an mbarrier
  nothing arrives at) is reported by upipe_sync_status as UPIPE_ETIMEOUT,
  which the read clears; the context stays usable.
"""
import ctypes

import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import SHAPES, layer_inputs
from tests.helpers import to_dev, f64_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def up():
    import headwise_chunked_ulysses_gb300 as u
    u.lib()
    return u


# ---------------------------------------------------------------------------
# reverse exchange with the fixed-order replica sum
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n_src,head_of_src,S,d,pad", [
    (8, [k // 4 for k in range(8)], 512, 128, 0),      # Llama in order: 8 slots, 4 copies of each of 2 KV heads
    (6, [2, 0, 1, 0, 2, 1], 384, 64, 64),               # copies spread over non-adjacent slots, padded rows
    (4, [0, 1, 2, 3], 256, 128, 0),                     # one copy per head: a conversion to bf16
    (16, [k // 8 for k in range(16)], 128, 64, 0),     # 8 copies per head
])
def test_reverse_exchange_sum_is_bit_exact(up, n_src, head_of_src, S, d, pad):
    import torch
    rng = np.random.default_rng(n_src * 1000 + S + d)
    # copies of very different magnitudes, so the fp32 sum depends on its order
    scale = 2.0 ** rng.integers(-20, 12, size=(n_src, S, 1))
    src = (rng.standard_normal((n_src, S, d)) * scale).astype(np.float32)
    n_heads = max(head_of_src) + 1
    ld = n_heads * d + pad
    dst_init = rng.integers(0, 1 << 16, size=(S, ld), dtype=np.uint16)
    dst = to_dev(dst_init)
    up.layout_head2seq_sum(torch.from_numpy(src).cuda(), head_of_src, dst, n_heads, ld)
    torch.cuda.synchronize()
    got = f64_of(dst[:, :n_heads * d])  # (the padding holds random bits, some of them NaN patterns)
    for h in range(n_heads):
        copies = src[[k for k in range(n_src) if head_of_src[k] == h]]
        _, want = orc.replica_gradient_sum(copies)
        g = got[:, h * d:(h + 1) * d]
        assert np.array_equal(g, want), h
        assert np.array_equal(np.signbit(g), np.signbit(want)), h
    # padding columns untouched
    assert np.array_equal(dst.view(torch.int16).cpu().numpy().view(np.uint16)[:, n_heads * d:],
                          dst_init[:, n_heads * d:])


# ---------------------------------------------------------------------------
# touched bytes of the workspace
# ---------------------------------------------------------------------------

def _touched(run, n_bytes):
    """Bytes of an n_bytes workspace that `run(ws)` changes, over two runs with
    the sentinels 0xA5 and 0x5A."""
    import torch
    masks = []
    for sentinel in (0xA5, 0x5A):
        ws = torch.full((n_bytes,), sentinel, dtype=torch.uint8, device="cuda")
        stats = run(ws)
        torch.cuda.synchronize()
        masks.append(ws != sentinel)
        del ws
    touched = masks[0] | masks[1]
    idx = torch.nonzero(touched)
    high = int(idx.max()) + 1 if idx.numel() else 0
    return touched, high, stats


@pytest.mark.parametrize("sched", [0, 1])
def test_workspace_high_water_is_the_plan(up, sched):
    """Llama3-8B widths at S=4096, both schedules: the highest byte the forward
    and the backward write is the last byte of their workspace plans (stage
    arena + persistent part), and the stage arena's touched bytes stay within
    the forward form 12 S U d (in order) and the backward plan."""
    import torch
    s = SHAPES["llama3_8b_4k"]
    sh = up.Shape(s.S, s.d_model, s.H, s.G, s.d_head, s.U, s.C, sched)
    bits = layer_inputs(s, 0)
    d = {k: to_dev(v) for k, v in bits.items()}
    nf, nb = up.fwd_workspace_bytes(sh), up.bwd_workspace_bytes(sh)
    tf, hf, stf = _touched(lambda ws: up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], sh, ws=ws)[3], nf)
    Y, O, lse, _ = up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], sh)
    tb, hb, stb = _touched(lambda ws: up.attn_bwd(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], sh, ws=ws)[3], nb)
    up.sync_status()
    for t, high, st, n in ((tf, hf, stf, nf), (tb, hb, stb, nb)):
        plan = st["arena_peak_bytes"] + st["persistent_bytes"]
        assert plan == n
        assert high == plan, (high, plan)
        arena_touched = int(t[:st["arena_peak_bytes"]].sum())
        # every buffer of the arena is written; only alignment gaps stay
        assert st["arena_peak_bytes"] - 8 * 256 <= arena_touched <= st["arena_peak_bytes"]
        if st is stf and sched == 0:
            assert arena_touched <= 12 * s.S * s.U * s.d_head
    if sched == 0:
        kv = max(1, s.U * s.G // s.H)
        form = 2 * s.S * s.d_head * (s.U + 2 * kv) + 20 * s.S * s.U * s.d_head + 8 * s.S * s.U
        assert int(tb[:stb["arena_peak_bytes"]].sum()) <= form


# ---------------------------------------------------------------------------
# failure detection
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("warp_form", [0, 1])
def test_bounded_wait_timeout_is_reported_and_cleared(up, warp_form):
    import torch
    lib = up.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.upipe_sync_status(stream) == up.OK
    up.watchdog_selftest(200_000, warp_form)  # ~0.1 ms of SM clocks, then the wait gives up
    assert lib.upipe_sync_status(stream) == up.ETIMEOUT
    assert lib.upipe_sync_status(stream) == up.OK  # the read cleared the word
    # the context is still usable
    Q = torch.randn(1, 128, 64, device="cuda").to(torch.bfloat16)
    O, lse = up.attention_fwd(Q, Q, Q, [0])
    torch.cuda.synchronize()
    assert bool(torch.isfinite(lse).all())
    assert lib.upipe_sync_status(stream) == up.OK
