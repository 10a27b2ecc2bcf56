"""CUDA-graph replay of layer calls (upipe_graphs_enable).

A replayed call runs the captured launch sequence on the same buffers, so the
forward is bit-identical to a direct call (its kernels are deterministic) and
the backward differs at most by the order of its fp32 atomic accumulations.
A replay must read the buffers' current contents, not the ones seen at
capture, and a call with other pointers must capture a graph of its own.
"""
import numpy as np
import pytest

from synthetic import SHAPES, layer_inputs, bf16_bits_to_f64
from tests.helpers import to_dev, f64_of, rel
from oracle import upipe_oracle as orc

pytestmark = pytest.mark.gpu
TOL = 1e-2
ORDER_TOL = 1e-3  # graph vs direct backward: atomic-order rounding only


@pytest.fixture(scope="module")
def up():
    import headwise_chunked_ulysses_gb300 as u
    u.lib()
    yield u
    u.graphs_enable(False)


def _buffers(up, sh, s):
    import torch
    S, dm, H, G, d = sh.S, sh.d_model, sh.H, sh.G, sh.d_head
    bf, f32 = torch.bfloat16, torch.float32
    b = dict(
        Y=torch.empty(S, dm, dtype=bf, device="cuda"), O=torch.empty(S, H * d, dtype=bf, device="cuda"),
        lse=torch.empty(H, S, dtype=f32, device="cuda"), dX=torch.empty(S, dm, dtype=bf, device="cuda"),
        dWq=torch.empty(dm, (H + 2 * G) * d, dtype=f32, device="cuda"),
        dWo=torch.empty(H * d, dm, dtype=f32, device="cuda"),
        wsf=torch.empty(up.fwd_workspace_bytes(s), dtype=torch.uint8, device="cuda"),
        wsb=torch.empty(up.bwd_workspace_bytes(s), dtype=torch.uint8, device="cuda"))
    return b


def _step(up, d, s, b):
    import torch
    for k in ("Y", "O", "lse", "dX", "dWq", "dWo"):
        b[k].view(torch.uint8).fill_(0xA5)  # a replay must write every output again
    _, _, _, sf = up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], s, Y=b["Y"], O_saved=b["O"], lse=b["lse"], ws=b["wsf"])
    _, _, _, sb = up.attn_bwd(d["X"], d["W_qkv"], d["W_o"], b["O"], b["lse"], d["dY"], s, dX=b["dX"],
                              dW_qkv=b["dWq"], dW_o=b["dWo"], ws=b["wsb"])
    torch.cuda.synchronize()
    up.sync_status()
    out = {k: b[k].clone() for k in ("Y", "O", "lse", "dX", "dWq", "dWo")}
    return out, sf, sb


def _same(a, c):
    import torch
    for k in ("Y", "O", "lse"):
        assert torch.equal(a[k].view(torch.uint8), c[k].view(torch.uint8)), k
    for k in ("dX", "dWq", "dWo"):
        assert rel(f64_of(a[k]), f64_of(c[k])) <= ORDER_TOL, k


@pytest.mark.parametrize("name,U,C,sched", [("tiny", 2, 2, 0), ("tiny", 4, 2, 1), ("tiny", 8, 4, 0),
                                            ("llama3_8b_4k", 8, 8, 0), ("llama3_8b_4k", 8, 8, 1)])
def test_graph_replay_matches_direct_calls(up, name, U, C, sched):
    import torch
    sh = SHAPES[name]
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, U, C, sched)
    d = {k: to_dev(v) for k, v in layer_inputs(sh, 0).items()}
    b = _buffers(up, sh, s)
    up.graphs_enable(False)
    direct, sf0, sb0 = _step(up, d, s, b)
    up.graphs_enable(True)
    try:
        first, sf1, sb1 = _step(up, d, s, b)    # captures, then launches the graph
        again, sf2, sb2 = _step(up, d, s, b)    # replays
        _same(direct, first)
        _same(direct, again)
        for a, c in ((sf0, sf1), (sf0, sf2), (sb0, sb1), (sb0, sb2)):
            assert a["launches"] == c["launches"] and a["arena_peak_bytes"] == c["arena_peak_bytes"]
        # new contents in the same buffers: the replay must see them
        d2 = {k: to_dev(v) for k, v in layer_inputs(sh, 1).items()}
        for k in d:
            d[k].copy_(d2[k])
        replay_new, _, _ = _step(up, d, s, b)
        up.graphs_enable(False)
        direct_new, _, _ = _step(up, d, s, b)
        _same(direct_new, replay_new)
        assert not torch.equal(replay_new["Y"], direct["Y"])
        # other pointers: a graph of their own, on their own buffers
        up.graphs_enable(True)
        b2 = _buffers(up, sh, s)
        other, _, _ = _step(up, d2, s, b2)
        _same(direct_new, other)
    finally:
        up.graphs_enable(False)
    if name == "tiny":
        f = {k: bf16_bits_to_f64(v) for k, v in layer_inputs(sh, 1).items()}
        Y, _, _ = orc.layer_forward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head)
        dX, dWq, dWo = orc.layer_backward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, f["dY"])
        assert rel(f64_of(replay_new["Y"]), Y) <= TOL
        assert rel(f64_of(replay_new["dX"]), dX) <= TOL
        assert rel(f64_of(replay_new["dWq"]), dWq) <= TOL
        assert rel(f64_of(replay_new["dWo"]), dWo) <= TOL


def test_graphs_step_aside_while_profiling(up):
    """With timing on, calls run directly so every launch gets its events."""
    sh = SHAPES["tiny"]
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, 2, 2, 0)
    d = {k: to_dev(v) for k, v in layer_inputs(sh, 0).items()}
    b = _buffers(up, sh, s)
    up.graphs_enable(True)
    try:
        _step(up, d, s, b)
        up.profile_enable(True)
        up.profile_read()
        _, sf, sb = _step(up, d, s, b)
        pk = up.profile_read()
        up.profile_enable(False)
    finally:
        up.graphs_enable(False)
    assert sum(v[1] for v in pk.values()) == sf["launches"] + sb["launches"]
