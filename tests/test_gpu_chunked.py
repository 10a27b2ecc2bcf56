"""Parity of the layer run on sequence chunks inside the head stages.

The oracle is the plain fp64 layer (the chunked oracle equals it, see the
oracle pins): chunking the sequence only regroups the work, so every chunk
count, U and C, with the offload store in device memory or in page-locked
host memory, must reproduce it within the layer tolerance (relative Frobenius
error <= 1e-2 per output).  Also checked: the guard bands around every output
and the workspace, the memory the plan reports, and the argument errors.
"""
import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import SHAPES, layer_inputs, bf16_bits_to_f64
from tests.helpers import to_dev, f64_of, rel

pytestmark = pytest.mark.gpu
TOL = 1e-2
LSE_TOL = 3e-2


@pytest.fixture(scope="module")
def up():
    import headwise_chunked_ulysses_gb300 as u
    u.lib()
    return u


class Ref:
    def __init__(self, sh, seed=0):
        self.sh = sh
        self.bits = layer_inputs(sh, seed)
        f = {k: bf16_bits_to_f64(v) for k, v in self.bits.items()}
        self.Y, self.O, self.lse = orc.layer_forward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head)
        self.dX, self.dW_qkv, self.dW_o = orc.layer_backward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head,
                                                             f["dY"])
        self.dev = {k: to_dev(v) for k, v in self.bits.items()}


@pytest.fixture(scope="module")
def tiny():
    return Ref(SHAPES["tiny"])


def _store(up, s, n_chunks, where):
    import torch
    n = up.chunked_store_bytes(s, n_chunks, True)
    assert n > 0
    t = torch.empty(n, dtype=torch.uint8)
    return t.pin_memory() if where == "host" else t.cuda()


def _run(up, ref, U, C, n_chunks, where, guard=4096):
    import torch
    sh = ref.sh
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, U, C, 0)
    d = ref.dev
    bf, f32 = torch.bfloat16, torch.float32
    specs = {"Y": ((sh.S, sh.d_model), bf), "O": ((sh.S, sh.H * sh.d_head), bf), "lse": ((sh.H, sh.S), f32),
             "dX": ((sh.S, sh.d_model), bf), "dW_qkv": ((sh.d_model, sh.qkv_cols), f32),
             "dW_o": ((sh.H * sh.d_head, sh.d_model), f32)}
    bufs, views = {}, {}
    for k, (shape, dt) in specs.items():
        n = int(np.prod(shape))
        bufs[k] = torch.empty(n + 2 * guard, dtype=dt, device="cuda")
        bufs[k].view(torch.uint8).fill_(0x5A)
        views[k] = bufs[k][guard:guard + n].view(*shape)
    nf = up.chunked_workspace_bytes(s, n_chunks, False)
    nb = up.chunked_workspace_bytes(s, n_chunks, True)
    extra = 1 << 16
    wsf = torch.full((nf + extra,), 0xA5, dtype=torch.uint8, device="cuda")
    wsb = torch.full((nb + extra,), 0xA5, dtype=torch.uint8, device="cuda")
    store = _store(up, s, n_chunks, where)
    Y, O, lse, stf = up.attn_fwd_chunked(d["X"], d["W_qkv"], d["W_o"], s, n_chunks, store, Y=views["Y"],
                                         O_saved=views["O"], lse=views["lse"], ws=wsf[:nf])
    dX, dWq, dWo, stb = up.attn_bwd_chunked(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s, n_chunks, store,
                                            dX=views["dX"], dW_qkv=views["dW_qkv"], dW_o=views["dW_o"],
                                            ws=wsb[:nb])
    torch.cuda.synchronize()
    up.sync_status()
    for k, buf in bufs.items():
        raw = buf.view(torch.uint8)
        per = buf.element_size()
        assert bool((raw[:guard * per] == 0x5A).all()) and bool((raw[-guard * per:] == 0x5A).all()), k
    assert bool((wsf[nf:] == 0xA5).all()) and bool((wsb[nb:] == 0xA5).all()), "workspace overrun"
    out = {"Y": f64_of(Y), "O": f64_of(O), "lse": f64_of(lse), "dX": f64_of(dX), "dW_qkv": f64_of(dWq),
           "dW_o": f64_of(dWo)}
    return out, stf, stb, s


def _check(ref, out):
    e = {"Y": rel(out["Y"], ref.Y), "O": rel(out["O"], ref.O), "dX": rel(out["dX"], ref.dX),
         "dW_qkv": rel(out["dW_qkv"], ref.dW_qkv), "dW_o": rel(out["dW_o"], ref.dW_o)}
    assert max(e.values()) <= TOL, e
    assert float(np.abs(out["lse"] - ref.lse).max()) < LSE_TOL


@pytest.mark.parametrize("U,C,n_chunks,where", [(2, 2, 2, "device"), (2, 2, 4, "host"), (4, 2, 8, "device"),
                                                (8, 4, 4, "host"), (8, 8, 1, "device"), (1, 1, 4, "device"),
                                                (2, 1, 2, "host"), (4, 4, 2, "device")])
def test_tiny_chunked_layer_matches_oracle(up, tiny, U, C, n_chunks, where):
    out, stf, stb, s = _run(up, tiny, U, C, n_chunks, where)
    _check(tiny, out)
    sh = tiny.sh
    Sc = sh.S // n_chunks
    assert stf["offload_bytes"] == 2 * sh.G * sh.S * sh.d_head * 2
    assert stb["offload_bytes"] == 2 * sh.G * sh.S * sh.d_head * 6
    # forward: every chunk's K/V goes out once per stage that projects it and
    # comes back once per later query chunk
    stages = sh.H // U
    kv_per_stage = max(1, U * sh.G // sh.H)
    unit = kv_per_stage * Sc * sh.d_head * 2 * 2  # K and V of one stage, one chunk
    assert stf["offload_copy_bytes"] == stages * unit * (n_chunks + n_chunks * (n_chunks - 1) // 2)
    assert stf["arena_peak_bytes"] < up.fwd_workspace_bytes(s) or n_chunks == 1


def test_llama_widths_4k_chunked(up):
    """Llama3-8B widths at S=4096: 4 chunks of 1024 with a host store, against
    the oracle."""
    ref = Ref(SHAPES["llama3_8b_4k"])
    out, stf, stb, s = _run(up, ref, 8, 8, 4, "host")
    _check(ref, out)


def test_chunked_memory_is_o_of_the_chunk(up):
    """The device workspace follows the chunk length, not S: at fixed Sc it
    stays put as S grows (only the fp32 chunk accumulator and the stage
    buffers, all Sc-sized), while the store grows with S."""
    sh = SHAPES["llama3_8b_32k"]
    sizes = []
    for S, n in ((32768, 4), (65536, 8), (131072, 16)):
        s = up.Shape(S, sh.d_model, sh.H, sh.G, sh.d_head, 8, 8, 0)
        sizes.append((up.chunked_workspace_bytes(s, n, False), up.chunked_workspace_bytes(s, n, True),
                      up.chunked_store_bytes(s, n, True)))
    assert sizes[0][0] == sizes[1][0] == sizes[2][0]
    assert sizes[0][1] == sizes[1][1] == sizes[2][1]
    assert sizes[2][2] == 4 * sizes[0][2]


def test_chunked_argument_errors(up, tiny):
    import torch
    sh = tiny.sh
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, 2, 2, 0)
    d = tiny.dev
    assert up.chunked_workspace_bytes(s, 3, False) == 0      # 3 does not divide S
    assert up.chunked_workspace_bytes(s, 16, False) == 0     # 64-token chunks
    store = _store(up, s, 2, "device")
    with pytest.raises(up.UpipeError) as e:
        up.attn_fwd_chunked(d["X"], d["W_qkv"], d["W_o"], s, 2, store[:1024])
    assert e.value.code == up.ENOSPC
    with pytest.raises(up.UpipeError) as e:
        up.attn_fwd_chunked(d["X"], d["W_qkv"], d["W_o"], s, 2, store, ws=torch.empty(1024, dtype=torch.uint8,
                                                                                      device="cuda"))
    assert e.value.code == up.ENOSPC
    with pytest.raises(up.UpipeError):
        up.attn_fwd_chunked(d["X"], d["W_qkv"], d["W_o"], s, 3, store)
