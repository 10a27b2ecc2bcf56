"""End-to-end parity of the layer (forward and backward) through the C ABI.

The oracle is the plain fp64 layer: the method only regroups the work, so
every U (including U = H, plain Ulysses), every C and both schedules must
reproduce it.  Tolerance: relative Frobenius error <= 1e-2 on each of Y, dX,
dW_qkv and dW_o (bf16 inputs, fp32 accumulation).  Also checked: the output
guards and the workspace tail stay untouched, and the plan's statistics.
"""
import numpy as np
import pytest

from oracle import upipe_oracle as orc
from synthetic import SHAPES, LayerShape, layer_inputs, bf16_bits_to_f64
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
    def __init__(self, sh: LayerShape, seed=0, backward=True):
        self.sh = sh
        self.bits = layer_inputs(sh, seed)
        f = {k: bf16_bits_to_f64(v) for k, v in self.bits.items()}
        self.Y, self.O, self.lse = orc.layer_forward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head)
        if backward:
            self.dX, self.dW_qkv, self.dW_o = orc.layer_backward(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G,
                                                                 sh.d_head, f["dY"])
        self.dev = {k: to_dev(v) for k, v in self.bits.items()}


@pytest.fixture(scope="module")
def tiny():
    return Ref(SHAPES["tiny"])


def _guarded(shape, dtype, guard=4096):
    """A tensor inside a larger buffer whose guard bands hold a sentinel."""
    import torch
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), 0, dtype=dtype, device="cuda")
    buf.view(torch.uint8 if dtype != torch.float32 else torch.int32).fill_(0x5A if dtype != torch.float32 else 0x5A5A5A5A)
    return buf, buf[guard:guard + n].view(*shape), guard


def _guard_ok(buf, guard, n):
    import torch
    raw = buf.view(torch.uint8)
    per = buf.element_size()
    head = raw[:guard * per]
    tail = raw[(guard + n) * per:]
    return bool((head == 0x5A).all()) and bool((tail == 0x5A).all())


def _run(up, ref, U, C, sched, check_guards=False, prefetch=False):
    import torch
    sh = ref.sh
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, U, C, sched)
    d = ref.dev
    bf, f32 = torch.bfloat16, torch.float32
    outs = {}
    if check_guards:
        shapes = {"Y": ((sh.S, sh.d_model), bf), "O": ((sh.S, sh.H * sh.d_head), bf), "lse": ((sh.H, sh.S), f32),
                  "dX": ((sh.S, sh.d_model), bf), "dW_qkv": ((sh.d_model, sh.qkv_cols), f32),
                  "dW_o": ((sh.H * sh.d_head, sh.d_model), f32)}
        for k, (shape, dt) in shapes.items():
            outs[k] = _guarded(shape, dt)
        # the library may use every byte it is given (a larger forward workspace
        # turns on stage prefetch), so it gets exactly the size, guard after it
        extra = 1 << 20
        nf = up.fwd_workspace_bytes_prefetch(s) if prefetch else up.fwd_workspace_bytes(s)
        nb = up.bwd_workspace_bytes(s)
        wsf = torch.full((nf + extra,), 0xA5, dtype=torch.uint8, device="cuda")
        wsb = torch.full((nb + extra,), 0xA5, dtype=torch.uint8, device="cuda")
        Y, O, lse, stf = up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], s, Y=outs["Y"][1], O_saved=outs["O"][1],
                                     lse=outs["lse"][1], ws=wsf[:nf])
        dX, dWqkv, dWo, stb = up.attn_bwd(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s, dX=outs["dX"][1],
                                          dW_qkv=outs["dW_qkv"][1], dW_o=outs["dW_o"][1], ws=wsb[:nb])
        torch.cuda.synchronize()
        for k, (buf, view, guard) in outs.items():
            assert _guard_ok(buf, guard, view.numel()), f"guard band of {k} overwritten"
        assert bool((wsf[nf:] == 0xA5).all()) and bool((wsb[nb:] == 0xA5).all()), "workspace overrun"
    else:
        Y, O, lse, stf = up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], s)
        dX, dWqkv, dWo, stb = up.attn_bwd(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s)
    up.sync_status()
    return {"Y": f64_of(Y), "O": f64_of(O), "lse": f64_of(lse), "dX": f64_of(dX), "dW_qkv": f64_of(dWqkv),
            "dW_o": f64_of(dWo), "stf": stf, "stb": stb}


def _errors(ref, out):
    return {"Y": rel(out["Y"], ref.Y), "O": rel(out["O"], ref.O), "dX": rel(out["dX"], ref.dX),
            "dW_qkv": rel(out["dW_qkv"], ref.dW_qkv), "dW_o": rel(out["dW_o"], ref.dW_o),
            "lse_abs": float(np.abs(out["lse"] - ref.lse).max())}


def _tiny_cases():
    H, G, S = 8, 2, 1024
    for U in (1, 2, 4, 8):
        for C in range(1, U + 1):
            if U % C or S % C:
                continue
            for sched in (0, 1):
                if sched == 1 and not (G % C == 0 or C % G == 0):
                    continue
                yield U, C, sched


@pytest.mark.parametrize("U,C,sched", list(_tiny_cases()))
def test_tiny_layer_matches_oracle_for_every_u(up, tiny, U, C, sched):
    out = _run(up, tiny, U, C, sched, check_guards=(U == 2 and C == 2), prefetch=(U == 2 and sched == 1))
    e = _errors(tiny, out)
    assert max(e["Y"], e["O"], e["dX"], e["dW_qkv"], e["dW_o"]) <= TOL, e
    # lse is a score-scale quantity: the scores use bf16-rounded projections
    # (relative error ~2^-8 per product), so |lse error| ~ 2^-8 * |typical score|
    assert e["lse_abs"] < LSE_TOL, e
    st = out["stf"]
    assert st["stages"] == 8 // U
    sh = tiny.sh
    if sched == 0:
        assert st["arena_peak_bytes"] <= 12 * sh.S * U * sh.d_head + 1024
    assert st["stage_closed_form_bytes"] == 12 * sh.S * U * sh.d_head


def test_u_invariance_across_stages(up, tiny):
    """Different U regroup the same sums: outputs agree with each other as
    closely as each agrees with the oracle."""
    outs = {U: _run(up, tiny, U, 2 if U >= 2 else 1, 0) for U in (2, 4, 8)}
    for U in (2, 4):
        for k in ("Y", "dX", "dW_qkv", "dW_o"):
            assert rel(outs[U][k], outs[8][k]) <= TOL, (U, k)


@pytest.mark.parametrize("shape,U,C,sched", [
    (LayerShape(S=512, d_model=192, H=4, G=2, d_head=64, U=2, C=2), 2, 2, 0),
    (LayerShape(S=512, d_model=192, H=4, G=2, d_head=64, U=2, C=2), 2, 2, 1),
    (LayerShape(S=384, d_model=320, H=4, G=1, d_head=128, U=4, C=2), 4, 2, 0),
    (LayerShape(S=256, d_model=64, H=2, G=2, d_head=64, U=1, C=1), 1, 1, 0)])
def test_d_model_a_multiple_of_64(up, shape, U, C, sched):
    """Model widths that are multiples of 64 but not of 128: the contractions
    with d_model as their row count (dW_qkv = X^T dQKV) end in a 64-row tile."""
    ref = Ref(shape, seed=5)
    out = _run(up, ref, U, C, sched, check_guards=True)
    e = _errors(ref, out)
    assert max(e["Y"], e["O"], e["dX"], e["dW_qkv"], e["dW_o"]) <= TOL, e
    assert e["lse_abs"] < LSE_TOL, e


@pytest.mark.parametrize("sched", [0, 1])
def test_llama_widths_4k(up, sched):
    ref = Ref(SHAPES["llama3_8b_4k"])
    out = _run(up, ref, 8, 8, sched)
    e = _errors(ref, out)
    assert max(e["Y"], e["O"], e["dX"], e["dW_qkv"], e["dW_o"]) <= TOL, e


def test_llama_32k_sampled_rows(up):
    """Full-size forward (the benchmarked launch configuration) against the
    oracle on sampled query rows, each computed from its exact key prefix."""
    import torch
    sh = SHAPES["llama3_8b_32k"]
    bits = layer_inputs(sh, 0)
    dev = {k: to_dev(v) for k, v in bits.items() if k != "dY"}
    for sched in (0, 1):
        s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, sched)
        Y, O, lse, st = up.attn_fwd(dev["X"], dev["W_qkv"], dev["W_o"], s)
        torch.cuda.synchronize()
        up.sync_status()
        rows = np.array([0, 1, 127, 128, 4095, 8191, 16384, 20000, 32766, 32767])
        f = {k: bf16_bits_to_f64(bits[k]) for k in ("X", "W_qkv", "W_o")}
        if sched == 0:
            Yr, Or, lser = orc.layer_forward_rows(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, rows)
        got = f64_of(Y[torch.as_tensor(rows, device="cuda")])
        assert rel(got, Yr) <= TOL
        assert np.abs(f64_of(lse)[:, rows] - lser).max() < LSE_TOL


def test_llama_32k_backward_full_size(up):
    """Full-size backward (the benchmarked configuration), both schedules,
    with the dense upstream gradient the bench uses: dW_o is O_saved^T dY by
    definition, at any size, so the library's split-K GEMM over K = S = 32768
    must match an fp32 product of the same bf16 operands; dX on the last rows
    matches the row-wise oracle (exact there: the K/V gradients of those rows
    come only from the queries after them).  dW_qkv and the other rows of dX
    are compared with the oracle in full by the sparse-gradient tests below."""
    import torch
    sh = SHAPES["llama3_8b_32k"]
    bits = layer_inputs(sh, 0)
    dev = {k: to_dev(v) for k, v in bits.items()}
    rows = np.array([sh.S - 40, sh.S - 2, sh.S - 1])
    got = {}
    for sched in (0, 1):
        s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, sched)
        Y, O, lse, _ = up.attn_fwd(dev["X"], dev["W_qkv"], dev["W_o"], s)
        dX, dWq, dWo, _ = up.attn_bwd(dev["X"], dev["W_qkv"], dev["W_o"], O, lse, dev["dY"], s)
        torch.cuda.synchronize()
        up.sync_status()
        ref = O.float().t() @ dev["dY"].float()
        assert float((dWo - ref).norm() / ref.norm()) < 1e-4, sched
        assert bool(torch.isfinite(dX.float()).all()) and bool(torch.isfinite(dWq).all()), sched
        got[sched] = f64_of(dX[torch.as_tensor(rows, device="cuda")])
        del Y, O, lse, dX, dWq, dWo, ref
    del dev
    torch.cuda.empty_cache()
    f = {k: bf16_bits_to_f64(bits[k]) for k in ("X", "W_qkv", "W_o", "dY")}
    want = orc.layer_backward_rows(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, f["dY"], rows)
    for sched in (0, 1):
        assert rel(got[sched], want) <= TOL, sched


# ---------------------------------------------------------------------------
# full-size backward parity with an upstream gradient on sampled rows
# ---------------------------------------------------------------------------
#
# With dY zero outside a set of query rows R, the oracle computes EVERY
# gradient exactly at |R| x S cost per head (layer_backward_sparse_dy, pinned
# to the whole-layer oracle): dX on all S rows, all of dW_qkv and dW_o.  The
# GPU runs its ordinary layer backward (same kernels and launch shapes as the
# bench; they do not look at the values).  R holds one row in each of 64
# randomly chosen query blocks plus the first and the last row, so every KV
# block receives gradient from many query blocks (the last row sees every
# key) and the work of 64 query blocks against every KV block before them is
# checked element by element.

_SPARSE_REF = {}


def _sparse_rows(S, n_blocks=64, seed=7):
    rng = np.random.default_rng(seed + S)
    blocks = np.sort(rng.choice(S // 128, size=min(n_blocks, S // 128), replace=False))
    rows = blocks * 128 + rng.integers(0, 128, size=len(blocks))
    return np.unique(np.concatenate([[0, S - 1], rows]))


def _sparse_reference(name):
    """Oracle gradients for the workload's inputs with dY kept only on the
    sampled rows (cached: the oracle does not depend on U or the schedule)."""
    if name not in _SPARSE_REF:
        _SPARSE_REF.clear()
        sh = SHAPES[name]
        bits = layer_inputs(sh, 0)
        rows = _sparse_rows(sh.S)
        f = {k: bf16_bits_to_f64(bits[k]) for k in ("X", "W_qkv", "W_o")}
        dX, dWq, dWo = orc.layer_backward_sparse_dy(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head,
                                                    bf16_bits_to_f64(bits["dY"][rows]), rows)
        del f
        _SPARSE_REF[name] = (bits, rows, dX.astype(np.float32), dWq, dWo)
    return _SPARSE_REF[name]


def _block_rel(got, want, block=128):
    """Largest relative error over blocks of `block` rows (rows whose reference
    is exactly zero excluded)."""
    worst = 0.0
    for b in range(0, want.shape[0], block):
        w = want[b:b + block]
        n = np.linalg.norm(w)
        if n > 0:
            worst = max(worst, float(np.linalg.norm(got[b:b + block] - w) / n))
    return worst


@pytest.mark.parametrize("name,U,sched", [("llama3_8b_32k", 8, 0), ("llama3_8b_32k", 8, 1),
                                          ("qwen3_32b_128k", 8, 0),
                                          ("llama3_8b_256k_usweep", 16, 0), ("llama3_8b_256k_usweep", 32, 0),
                                          ("llama3_8b_512k_gqa", 8, 1)])
def test_full_size_backward_on_sampled_gradient_rows(up, name, U, sched):
    """Every output of the full-size backward against the oracle: the Llama3-8B
    layer at 32K (both schedules), the Qwen3-32B layer at 128K, the 256K layer
    at U = 16 and U = 32, and the GQA out-of-order schedule at 512K."""
    import torch
    bits, rows, dX_ref, dWq_ref, dWo_ref = _sparse_reference(name)
    sh = SHAPES[name].replace(U=U)
    dY = np.zeros_like(bits["dY"])
    dY[rows] = bits["dY"][rows]
    dev = {k: to_dev(v) for k, v in bits.items() if k != "dY"}
    dev["dY"] = to_dev(dY)
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, sched)
    Y, O, lse, _ = up.attn_fwd(dev["X"], dev["W_qkv"], dev["W_o"], s)
    dX, dWq, dWo, _ = up.attn_bwd(dev["X"], dev["W_qkv"], dev["W_o"], O, lse, dev["dY"], s)
    torch.cuda.synchronize()
    up.sync_status()
    got = {"dX": f64_of(dX), "dW_qkv": f64_of(dWq), "dW_o": f64_of(dWo)}
    del Y, O, lse, dX, dWq, dWo, dev
    torch.cuda.empty_cache()
    errs = {"dX": rel(got["dX"], dX_ref), "dW_qkv": rel(got["dW_qkv"], dWq_ref), "dW_o": rel(got["dW_o"], dWo_ref)}
    assert max(errs.values()) <= TOL, errs
    # localised errors (one KV block, one head's columns) would hide in the
    # whole-tensor norm: per 128-row block of dX and per head block of dW_qkv
    d = sh.d_head
    blk = {"dX": _block_rel(got["dX"], dX_ref),
           "dW_qkv": _block_rel(got["dW_qkv"].T, dWq_ref.T, block=d)}
    assert max(blk.values()) <= 3 * TOL, blk


def _sampled_rows_check(up, name, sched, rows):
    import torch
    sh = SHAPES[name]
    bits = layer_inputs(sh, 0)
    dev = {k: to_dev(v) for k, v in bits.items() if k != "dY"}
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, sched)
    Y, O, lse, st = up.attn_fwd(dev["X"], dev["W_qkv"], dev["W_o"], s)
    torch.cuda.synchronize()
    up.sync_status()
    got = f64_of(Y[torch.as_tensor(rows, device="cuda")])
    got_lse = f64_of(lse)[:, rows]
    del Y, O, lse, dev
    torch.cuda.empty_cache()
    f = {k: bf16_bits_to_f64(bits[k]) for k in ("X", "W_qkv", "W_o")}
    Yr, _, lser = orc.layer_forward_rows(f["X"], f["W_qkv"], f["W_o"], sh.H, sh.G, sh.d_head, rows)
    assert rel(got, Yr) <= TOL
    assert np.abs(got_lse - lser).max() < LSE_TOL


def test_qwen3_32b_128k_sampled_rows(up):
    """Qwen3-32B-shaped layer (S=131072, H=64, G=8, d_model=5120, U=8, C=8)."""
    _sampled_rows_check(up, "qwen3_32b_128k", 0, np.array([0, 77, 4096, 65535, 100000, 131071]))


def test_gqa_schedule_512k_sampled_rows(up):
    """The GQA out-of-order schedule at S=524288 (Llama3-8B widths)."""
    _sampled_rows_check(up, "llama3_8b_512k_gqa", 1, np.array([5, 262143, 524287]))


@pytest.mark.parametrize("name,U,C,sched", [("tiny", 2, 2, 0), ("tiny", 2, 2, 1), ("tiny", 4, 2, 1),
                                            ("llama3_8b_4k", 8, 8, 0), ("llama3_8b_4k", 8, 8, 1)])
def test_prefetching_forward_is_bit_identical(up, tiny, name, U, C, sched):
    """With the larger workspace the next stage's projection and exchange run
    on a second stream during the current stage's attention; the same kernels
    run on the same data in the same per-stage order, so Y, O and lse are
    bit-identical to the single-stream forward (and the oracle still holds)."""
    import torch
    ref = tiny if name == "tiny" else Ref(SHAPES[name], backward=False)
    sh = ref.sh
    s = up.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, U, C, sched)
    d = ref.dev
    outs = []
    for prefetch in (False, True):
        Y, O, lse, st = up.attn_fwd(d["X"], d["W_qkv"], d["W_o"], s, prefetch=prefetch)
        torch.cuda.synchronize()
        up.sync_status()
        outs.append((Y.view(torch.int16).clone(), O.view(torch.int16).clone(), lse.clone(), st))
    for a, b in zip(outs[0][:3], outs[1][:3]):
        assert torch.equal(a, b)
    assert outs[1][3]["arena_peak_bytes"] > outs[0][3]["arena_peak_bytes"]
    assert outs[1][3]["launches"] == outs[0][3]["launches"]
    assert rel(f64_of(outs[1][0].view(torch.bfloat16)), ref.Y) <= TOL
