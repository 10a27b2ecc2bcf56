"""Headwise-chunked (UPipe) causal GQA attention layer on one GB300.

A thin ctypes binding over the C ABI in include/upipe.h (libupipe.so, built
in-tree by ``_build.build()``).  Argument marshalling only: PyTorch provides
device memory and the current stream; every step of the layer runs in the
library's CUDA kernels.  There is no CPU or PyTorch fallback: without the
built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libupipe.so")

IN_ORDER = 0
GQA_OUT_OF_ORDER = 1

OK, EINVAL, ENOSPC, EUNSUPPORTED, ECUDA, ETIMEOUT = range(6)

# Entry points declared in include/upipe.h
EXPORTS = (
    "upipe_fwd_workspace_bytes", "upipe_fwd_workspace_bytes_prefetch", "upipe_bwd_workspace_bytes",
    "upipe_attn_fwd", "upipe_attn_bwd",
    "upipe_layout_seq2head", "upipe_layout_head2seq", "upipe_schedule_table", "upipe_choose_u",
    "upipe_attention_fwd", "upipe_attention_bwd", "upipe_attention_bwd_noalloc", "upipe_gemm_bf16",
    "upipe_sync_status", "upipe_status_str", "upipe_version", "upipe_profile_enable", "upipe_profile_read",
    "upipe_graphs_enable", "upipe_chunked_workspace_bytes", "upipe_chunked_store_bytes",
    "upipe_attn_fwd_chunked", "upipe_attn_bwd_chunked",
    "upipe_quantize_e4m3", "upipe_attention_fwd_fp8", "upipe_attn_fwd_fp8", "upipe_choose_chunks",
    "upipe_layout_head2seq_sum", "upipe_watchdog_selftest",
    "upipe_attention_bwd_fp8", "upipe_attn_bwd_fp8", "upipe_bwd_workspace_bytes_fp8",
)


class UpipeError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


KERNEL_KINDS = ("gemm", "attn_fwd", "attn_bwd", "seq2head", "head2seq", "bwd_prep")


class Stats(ctypes.Structure):
    _fields_ = [("arena_peak_bytes", ctypes.c_size_t), ("stage_closed_form_bytes", ctypes.c_size_t),
                ("persistent_bytes", ctypes.c_size_t), ("permute_bytes", ctypes.c_size_t),
                ("launches", ctypes.c_int), ("stages", ctypes.c_int),
                ("launches_by_kind", ctypes.c_int * len(KERNEL_KINDS)),
                ("flops_by_kind", ctypes.c_double * len(KERNEL_KINDS)),
                ("bytes_by_kind", ctypes.c_double * len(KERNEL_KINDS)),
                ("offload_bytes", ctypes.c_size_t), ("offload_copy_bytes", ctypes.c_size_t)]

    def as_dict(self):
        d = {}
        for k, _ in self._fields_:
            v = getattr(self, k)
            d[k] = {n: v[i] for i, n in enumerate(KERNEL_KINDS)} if k.endswith("_by_kind") else v
        return d


_lib = None


def _sig(lib):
    P, I, Z, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
    i32p = ctypes.POINTER(ctypes.c_int32)
    spec = {
        "upipe_fwd_workspace_bytes": (Z, [I] * 8),
        "upipe_fwd_workspace_bytes_prefetch": (Z, [I] * 8),
        "upipe_bwd_workspace_bytes": (Z, [I] * 8),
        "upipe_attn_fwd": (I, [P, P, P] + [I] * 8 + [P, P, P, P, Z, P, ctypes.POINTER(Stats)]),
        "upipe_attn_bwd": (I, [P, P, P] + [I] * 8 + [P, P, P, P, P, P, P, Z, P, ctypes.POINTER(Stats)]),
        "upipe_layout_seq2head": (I, [P, P, I, I, I, I, I, P]),
        "upipe_layout_head2seq": (I, [P, P, I, I, I, I, I, P]),
        "upipe_layout_head2seq_sum": (I, [P, I, i32p, P, I, I, I, I, P]),
        "upipe_watchdog_selftest": (I, [LL, I, P]),
        "upipe_schedule_table": (I, [I, I, I, I, I, i32p]),
        "upipe_choose_u": (I, [I, I, I, I, I, I, I, Z]),
        "upipe_attention_fwd": (I, [P, P, P, I, I, I, I, i32p, P, P, P]),
        "upipe_attention_bwd": (I, [P, P, P, P, P, P, I, I, I, I, i32p, P, P, P, P, Z, P]),
        "upipe_attention_bwd_noalloc": (I, [P, P, P, P, P, P, I, I, I, I, i32p, P, P, P, P]),
        "upipe_gemm_bf16": (I, [P, P, P, I, I, I, I, I, LL, LL, LL, I, P]),
        "upipe_sync_status": (I, [P]),
        "upipe_status_str": (ctypes.c_char_p, [I]),
        "upipe_version": (I, []),
        "upipe_profile_enable": (I, [I]),
        "upipe_graphs_enable": (I, [I]),
        "upipe_quantize_e4m3": (I, [P, I, I, I, LL, I, P, P, P]),
        "upipe_attention_fwd_fp8": (I, [P, P, P, P, P, I, I, I, I, i32p, P, P, P]),
        "upipe_attn_fwd_fp8": (I, [P, P, P] + [I] * 7 + [ctypes.c_char_p, P, P, P, P, Z, P, P]),
        "upipe_attention_bwd_fp8": (I, [P, P, P, P, P, P, P, P, I, I, I, I, i32p, P, P, P, P, Z, P]),
        "upipe_attn_bwd_fp8": (I, [P, P, P] + [I] * 7 + [ctypes.c_char_p, P, P, P, P, P, P, P, Z, P,
                                                          ctypes.POINTER(Stats)]),
        "upipe_bwd_workspace_bytes_fp8": (Z, [I] * 7 + [ctypes.c_char_p]),
        "upipe_chunked_workspace_bytes": (Z, [I] * 9),
        "upipe_choose_chunks": (I, [I] * 7 + [Z]),
        "upipe_chunked_store_bytes": (Z, [I] * 9),
        "upipe_attn_fwd_chunked": (I, [P, P, P] + [I] * 8 + [P, P, P, P, Z, P, Z, P, P]),
        "upipe_attn_bwd_chunked": (I, [P, P, P] + [I] * 8 + [P, P, P, P, P, P, P, Z, P, Z, P, P]),
        "upipe_profile_read": (I, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
    }
    for name, (res, args) in spec.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libupipe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        _sig(l)
        _lib = l
    return _lib


def _check(fn, rc):
    if rc != OK:
        raise UpipeError(fn, rc, lib().upipe_status_str(rc).decode())


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t, dtype=None, name="tensor"):
    torch = _torch()
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


@dataclass
class Shape:
    S: int
    d_model: int
    H: int
    G: int
    d_head: int
    U: int
    C: int
    sched: int = IN_ORDER

    def args(self):
        return (self.S, self.d_model, self.H, self.G, self.d_head, self.U, self.C, self.sched)


def fwd_workspace_bytes(sh: Shape) -> int:
    return int(lib().upipe_fwd_workspace_bytes(*sh.args()))


def fwd_workspace_bytes_prefetch(sh: Shape) -> int:
    """Forward workspace that lets the next stage's projection and exchange
    overlap the current stage's attention (see upipe_fwd_workspace_bytes_prefetch)."""
    return int(lib().upipe_fwd_workspace_bytes_prefetch(*sh.args()))


def bwd_workspace_bytes(sh: Shape) -> int:
    return int(lib().upipe_bwd_workspace_bytes(*sh.args()))


def schedule_table(H, G, U, C, sched=IN_ORDER):
    """Query head of (stage, rank, slot), shape [H/U][C][U/C] (host ints)."""
    import numpy as np
    out = np.zeros(H, dtype=np.int32)
    _check("upipe_schedule_table", lib().upipe_schedule_table(
        H, G, U, C, sched, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
    return out.reshape(H // U, C, U // C)


def choose_u(S, d_model, H, G, d_head, C, sched, budget_bytes):
    """Largest stage width U whose forward and backward workspaces fit in
    budget_bytes (0 if none does); see upipe_choose_u."""
    return int(lib().upipe_choose_u(S, d_model, H, G, d_head, C, sched, int(budget_bytes)))


def _workspace(nbytes, device):
    torch = _torch()
    # 256-byte aligned (the caching allocator returns 512-byte aligned blocks)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def attn_fwd(X, W_qkv, W_o, sh: Shape, Y=None, O_saved=None, lse=None, ws=None, stream=None, prefetch=False):
    """Layer forward.  Returns (Y, O_saved, lse, stats).  prefetch=True sizes the
    workspace (when none is given) so that the next stage is fetched while the
    current one computes."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    dev = X.device
    S, dm, H, d = sh.S, sh.d_model, sh.H, sh.d_head
    Y = torch.empty(S, dm, dtype=bf, device=dev) if Y is None else Y
    O_saved = torch.empty(S, H * d, dtype=bf, device=dev) if O_saved is None else O_saved
    lse = torch.empty(H, S, dtype=f32, device=dev) if lse is None else lse
    need = fwd_workspace_bytes(sh)
    if need == 0:
        raise UpipeError("upipe_fwd_workspace_bytes", EINVAL, "invalid shape")
    if prefetch:
        need = max(need, fwd_workspace_bytes_prefetch(sh))
    ws = _workspace(need, dev) if ws is None else ws
    st = Stats()
    _check("upipe_attn_fwd", lib().upipe_attn_fwd(
        _ptr(X, bf, "X"), _ptr(W_qkv, bf, "W_qkv"), _ptr(W_o, bf, "W_o"), *sh.args(),
        _ptr(Y, bf, "Y"), _ptr(O_saved, bf, "O_saved"), _ptr(lse, f32, "lse"),
        _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(st)))
    return Y, O_saved, lse, st.as_dict()


def attn_bwd(X, W_qkv, W_o, O_saved, lse, dY, sh: Shape, dX=None, dW_qkv=None, dW_o=None, ws=None,
             stream=None):
    """Layer backward.  Returns (dX, dW_qkv, dW_o, stats)."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    dev = X.device
    S, dm, H, G, d = sh.S, sh.d_model, sh.H, sh.G, sh.d_head
    dX = torch.empty(S, dm, dtype=bf, device=dev) if dX is None else dX
    dW_qkv = torch.empty(dm, (H + 2 * G) * d, dtype=f32, device=dev) if dW_qkv is None else dW_qkv
    dW_o = torch.empty(H * d, dm, dtype=f32, device=dev) if dW_o is None else dW_o
    need = bwd_workspace_bytes(sh)
    if need == 0:
        raise UpipeError("upipe_bwd_workspace_bytes", EINVAL, "invalid shape")
    ws = _workspace(need, dev) if ws is None else ws
    st = Stats()
    _check("upipe_attn_bwd", lib().upipe_attn_bwd(
        _ptr(X, bf, "X"), _ptr(W_qkv, bf, "W_qkv"), _ptr(W_o, bf, "W_o"), *sh.args(),
        _ptr(O_saved, bf, "O_saved"), _ptr(lse, f32, "lse"), _ptr(dY, bf, "dY"),
        _ptr(dX, bf, "dX"), _ptr(dW_qkv, f32, "dW_qkv"), _ptr(dW_o, f32, "dW_o"),
        _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(st)))
    return dX, dW_qkv, dW_o, st.as_dict()


def quantize_e4m3(src, S, n_heads, d_head, src_row_stride, per_row, dst=None, scales=None, stream=None):
    """E4M3 codes [n_heads, S, d_head] (uint8) and fp32 scales of bf16 rows in
    sequence layout (see upipe_quantize_e4m3).  Returns (codes, scales)."""
    torch = _torch()
    dev = src.device
    dst = torch.empty(n_heads, S, d_head, dtype=torch.uint8, device=dev) if dst is None else dst
    n_sc = S if per_row else S // 128
    scales = torch.empty(n_heads, n_sc, dtype=torch.float32, device=dev) if scales is None else scales
    _check("upipe_quantize_e4m3", lib().upipe_quantize_e4m3(
        _ptr(src, torch.bfloat16, "src"), S, n_heads, d_head, src_row_stride, 1 if per_row else 0,
        _ptr(dst, torch.uint8, "dst"), _ptr(scales, torch.float32, "scales"), _stream(stream)))
    return dst, scales


def attention_fwd_fp8(Q8, q_scale, K8, k_scale, V, kv_of_q, O=None, lse=None, stream=None):
    """Attention with FP8 scores (see upipe_attention_fwd_fp8).  Returns (O, lse)."""
    torch = _torch()
    n_q, S, d = Q8.shape
    n_kv = K8.shape[0]
    O = torch.empty(n_q, S, d, dtype=torch.bfloat16, device=Q8.device) if O is None else O
    lse = torch.empty(n_q, S, dtype=torch.float32, device=Q8.device) if lse is None else lse
    kv = (ctypes.c_int32 * n_q)(*kv_of_q)
    _check("upipe_attention_fwd_fp8", lib().upipe_attention_fwd_fp8(
        _ptr(Q8, torch.uint8, "Q"), _ptr(q_scale, torch.float32, "q_scale"), _ptr(K8, torch.uint8, "K"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(V, torch.bfloat16, "V"), n_q, n_kv, S, d, kv,
        _ptr(O, torch.bfloat16, "O"), _ptr(lse, torch.float32, "lse"), _stream(stream)))
    return O, lse


def attn_fwd_fp8(X, W_qkv, W_o, sh: Shape, fp8_heads, Y=None, O_saved=None, lse=None, ws=None, stream=None):
    """Layer forward (in-order stages) with FP8 scores for the heads in
    fp8_heads (a set of head indices; whole stages).  Returns (Y, O_saved,
    lse, stats)."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    dev = X.device
    S, dm, H, d = sh.S, sh.d_model, sh.H, sh.d_head
    Y = torch.empty(S, dm, dtype=bf, device=dev) if Y is None else Y
    O_saved = torch.empty(S, H * d, dtype=bf, device=dev) if O_saved is None else O_saved
    lse = torch.empty(H, S, dtype=f32, device=dev) if lse is None else lse
    s0 = Shape(*sh.args()[:7], IN_ORDER)
    need = fwd_workspace_bytes(s0)
    if need == 0:
        raise UpipeError("upipe_fwd_workspace_bytes", EINVAL, "invalid shape")
    ws = _workspace(need, dev) if ws is None else ws
    flags = bytes(1 if h in fp8_heads else 0 for h in range(H))
    st = Stats()
    _check("upipe_attn_fwd_fp8", lib().upipe_attn_fwd_fp8(
        _ptr(X, bf, "X"), _ptr(W_qkv, bf, "W_qkv"), _ptr(W_o, bf, "W_o"), *sh.args()[:7], flags,
        _ptr(Y, bf, "Y"), _ptr(O_saved, bf, "O_saved"), _ptr(lse, f32, "lse"), _ptr(ws), ws.numel(),
        _stream(stream), ctypes.byref(st)))
    return Y, O_saved, lse, st.as_dict()


def bwd_workspace_bytes_fp8(sh: Shape, fp8_heads) -> int:
    """Workspace of attn_bwd_fp8 (smaller when every stage is FP8)."""
    flags = bytes(1 if h in fp8_heads else 0 for h in range(sh.H))
    return int(lib().upipe_bwd_workspace_bytes_fp8(*sh.args()[:7], flags))


def attn_bwd_fp8(X, W_qkv, W_o, O_saved, lse, dY, sh: Shape, fp8_heads, dX=None, dW_qkv=None, dW_o=None, ws=None,
                 stream=None):
    """Layer backward of attn_fwd_fp8 (in-order stages; the flagged stages'
    attention on the FP8 codes).  Returns (dX, dW_qkv, dW_o, stats)."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    dev = X.device
    S, dm, H, G, d = sh.S, sh.d_model, sh.H, sh.G, sh.d_head
    dX = torch.empty(S, dm, dtype=bf, device=dev) if dX is None else dX
    dW_qkv = torch.empty(dm, (H + 2 * G) * d, dtype=f32, device=dev) if dW_qkv is None else dW_qkv
    dW_o = torch.empty(H * d, dm, dtype=f32, device=dev) if dW_o is None else dW_o
    need = bwd_workspace_bytes_fp8(sh, fp8_heads)
    if need == 0:
        raise UpipeError("upipe_bwd_workspace_bytes_fp8", EINVAL, "invalid shape")
    ws = _workspace(need, dev) if ws is None else ws
    flags = bytes(1 if h in fp8_heads else 0 for h in range(H))
    st = Stats()
    _check("upipe_attn_bwd_fp8", lib().upipe_attn_bwd_fp8(
        _ptr(X, bf, "X"), _ptr(W_qkv, bf, "W_qkv"), _ptr(W_o, bf, "W_o"), *sh.args()[:7], flags,
        _ptr(O_saved, bf, "O_saved"), _ptr(lse, f32, "lse"), _ptr(dY, bf, "dY"), _ptr(dX, bf, "dX"),
        _ptr(dW_qkv, f32, "dW_qkv"), _ptr(dW_o, f32, "dW_o"), _ptr(ws), ws.numel(), _stream(stream),
        ctypes.byref(st)))
    return dX, dW_qkv, dW_o, st.as_dict()


def attention_bwd_fp8(Q8, q_scale, K8, k_scale, V, O, dO, lse, kv_of_q, stream=None):
    """Backward of attention_fwd_fp8: returns fp32 (dQ, dK, dV), the gradients
    in the dequantized Q and K."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    n_q, S, d = Q8.shape
    n_kv = K8.shape[0]
    dQ = torch.empty(n_q, S, d, dtype=f32, device=Q8.device)
    dK = torch.empty(n_kv, S, d, dtype=f32, device=Q8.device)
    dV = torch.empty(n_kv, S, d, dtype=f32, device=Q8.device)
    ws = torch.empty(8 * n_q * S, dtype=torch.uint8, device=Q8.device)
    _check("upipe_attention_bwd_fp8", lib().upipe_attention_bwd_fp8(
        _ptr(Q8, torch.uint8, "Q"), _ptr(q_scale, f32, "q_scale"), _ptr(K8, torch.uint8, "K"),
        _ptr(k_scale, f32, "k_scale"), _ptr(V, bf, "V"), _ptr(O, bf, "O"), _ptr(dO, bf, "dO"), _ptr(lse, f32, "lse"),
        n_q, n_kv, S, d, _i32(kv_of_q), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), _stream(stream)))
    return dQ, dK, dV


def chunked_workspace_bytes(sh: Shape, n_chunks, backward) -> int:
    return int(lib().upipe_chunked_workspace_bytes(*sh.args()[:7], n_chunks, 1 if backward else 0))


def choose_chunks(sh: Shape, budget_bytes) -> int:
    """Fewest sequence chunks whose chunked workspaces fit budget_bytes (0 if
    none); see upipe_choose_chunks."""
    return int(lib().upipe_choose_chunks(*sh.args()[:7], int(budget_bytes)))


def chunked_store_bytes(sh: Shape, n_chunks, backward) -> int:
    return int(lib().upipe_chunked_store_bytes(*sh.args()[:7], n_chunks, 1 if backward else 0))


def _store_ptr(store):
    """The offload store: a CUDA tensor, or a page-locked CPU tensor."""
    if store.is_cuda:
        return _ptr(store, None, "store")
    if not store.is_pinned():
        raise ValueError("a host store must be page-locked (pin_memory)")
    if not store.is_contiguous():
        raise ValueError("store must be contiguous")
    return ctypes.c_void_p(store.data_ptr())


def attn_fwd_chunked(X, W_qkv, W_o, sh: Shape, n_chunks, store, Y=None, O_saved=None, lse=None, ws=None,
                     stream=None):
    """Layer forward on sequence chunks (in-order stages); store is the K/V
    offload store (device or pinned host tensor of chunked_store_bytes()).
    Returns (Y, O_saved, lse, stats)."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    dev = X.device
    S, dm, H, d = sh.S, sh.d_model, sh.H, sh.d_head
    Y = torch.empty(S, dm, dtype=bf, device=dev) if Y is None else Y
    O_saved = torch.empty(S, H * d, dtype=bf, device=dev) if O_saved is None else O_saved
    lse = torch.empty(H, S, dtype=f32, device=dev) if lse is None else lse
    need = chunked_workspace_bytes(sh, n_chunks, False)
    if need == 0:
        raise UpipeError("upipe_chunked_workspace_bytes", EINVAL, "invalid shape or chunk count")
    ws = _workspace(need, dev) if ws is None else ws
    st = Stats()
    _check("upipe_attn_fwd_chunked", lib().upipe_attn_fwd_chunked(
        _ptr(X, bf, "X"), _ptr(W_qkv, bf, "W_qkv"), _ptr(W_o, bf, "W_o"), *sh.args()[:7], n_chunks,
        _ptr(Y, bf, "Y"), _ptr(O_saved, bf, "O_saved"), _ptr(lse, f32, "lse"),
        _ptr(ws), ws.numel(), _store_ptr(store), store.numel() * store.element_size(), _stream(stream),
        ctypes.byref(st)))
    return Y, O_saved, lse, st.as_dict()


def attn_bwd_chunked(X, W_qkv, W_o, O_saved, lse, dY, sh: Shape, n_chunks, store, dX=None, dW_qkv=None,
                     dW_o=None, ws=None, stream=None):
    """Layer backward on sequence chunks.  Returns (dX, dW_qkv, dW_o, stats)."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    dev = X.device
    S, dm, H, G, d = sh.S, sh.d_model, sh.H, sh.G, sh.d_head
    dX = torch.empty(S, dm, dtype=bf, device=dev) if dX is None else dX
    dW_qkv = torch.empty(dm, (H + 2 * G) * d, dtype=f32, device=dev) if dW_qkv is None else dW_qkv
    dW_o = torch.empty(H * d, dm, dtype=f32, device=dev) if dW_o is None else dW_o
    need = chunked_workspace_bytes(sh, n_chunks, True)
    if need == 0:
        raise UpipeError("upipe_chunked_workspace_bytes", EINVAL, "invalid shape or chunk count")
    ws = _workspace(need, dev) if ws is None else ws
    st = Stats()
    _check("upipe_attn_bwd_chunked", lib().upipe_attn_bwd_chunked(
        _ptr(X, bf, "X"), _ptr(W_qkv, bf, "W_qkv"), _ptr(W_o, bf, "W_o"), *sh.args()[:7], n_chunks,
        _ptr(O_saved, bf, "O_saved"), _ptr(lse, f32, "lse"), _ptr(dY, bf, "dY"),
        _ptr(dX, bf, "dX"), _ptr(dW_qkv, f32, "dW_qkv"), _ptr(dW_o, f32, "dW_o"),
        _ptr(ws), ws.numel(), _store_ptr(store), store.numel() * store.element_size(), _stream(stream),
        ctypes.byref(st)))
    return dX, dW_qkv, dW_o, st.as_dict()


def layout_seq2head(src, dst, S, n_heads, d_head, C, src_row_stride, stream=None):
    bf = _torch().bfloat16
    _check("upipe_layout_seq2head", lib().upipe_layout_seq2head(
        _ptr(src, bf, "src"), _ptr(dst, bf, "dst"), S, n_heads, d_head, C, src_row_stride, _stream(stream)))
    return dst


def layout_head2seq(src, dst, S, n_heads, d_head, C, dst_row_stride, stream=None):
    bf = _torch().bfloat16
    _check("upipe_layout_head2seq", lib().upipe_layout_head2seq(
        _ptr(src, bf, "src"), _ptr(dst, bf, "dst"), S, n_heads, d_head, C, dst_row_stride, _stream(stream)))
    return dst


def layout_head2seq_sum(src, head_of_src, dst, n_heads, dst_row_stride, stream=None):
    """Gradients in head layout (fp32 [n_src, S, d]) back to bf16 sequence
    rows, the copies of each head summed in ascending slot order
    (see upipe_layout_head2seq_sum)."""
    torch = _torch()
    n_src, S, d = src.shape
    _check("upipe_layout_head2seq_sum", lib().upipe_layout_head2seq_sum(
        _ptr(src, torch.float32, "src"), n_src, _i32(head_of_src), _ptr(dst, torch.bfloat16, "dst"), S, n_heads, d,
        dst_row_stride, _stream(stream)))
    return dst


def watchdog_selftest(limit_cycles, warp_form=0, stream=None):
    """Launch the bounded-wait self-test (see upipe_watchdog_selftest); the
    next sync_status() raises with UPIPE_ETIMEOUT."""
    _check("upipe_watchdog_selftest", lib().upipe_watchdog_selftest(int(limit_cycles), int(warp_form),
                                                                    _stream(stream)))


def _i32(seq):
    arr = (ctypes.c_int32 * len(seq))(*[int(x) for x in seq])
    return arr


def attention_fwd(Q, K, V, kv_of_q, O=None, lse=None, stream=None):
    """Causal GQA attention in head layout: Q [n_q, S, d], K/V [n_kv, S, d]."""
    torch = _torch()
    bf = torch.bfloat16
    n_q, S, d = Q.shape
    n_kv = K.shape[0]
    O = torch.empty_like(Q) if O is None else O
    lse = torch.empty(n_q, S, dtype=torch.float32, device=Q.device) if lse is None else lse
    _check("upipe_attention_fwd", lib().upipe_attention_fwd(
        _ptr(Q, bf, "Q"), _ptr(K, bf, "K"), _ptr(V, bf, "V"), n_q, n_kv, S, d, _i32(kv_of_q),
        _ptr(O, bf, "O"), _ptr(lse, torch.float32, "lse"), _stream(stream)))
    return O, lse


def attention_bwd(Q, K, V, O, dO, lse, kv_of_q, stream=None):
    """Backward of ``attention_fwd``: returns fp32 (dQ, dK, dV)."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    n_q, S, d = Q.shape
    n_kv = K.shape[0]
    dQ = torch.empty(n_q, S, d, dtype=f32, device=Q.device)
    dK = torch.empty(n_kv, S, d, dtype=f32, device=Q.device)
    dV = torch.empty(n_kv, S, d, dtype=f32, device=Q.device)
    ws = torch.empty(8 * n_q * S, dtype=torch.uint8, device=Q.device)
    _check("upipe_attention_bwd", lib().upipe_attention_bwd(
        _ptr(Q, bf, "Q"), _ptr(K, bf, "K"), _ptr(V, bf, "V"), _ptr(O, bf, "O"), _ptr(dO, bf, "dO"),
        _ptr(lse, f32, "lse"), n_q, n_kv, S, d, _i32(kv_of_q), _ptr(dQ), _ptr(dK), _ptr(dV),
        _ptr(ws), ws.numel(), _stream(stream)))
    return dQ, dK, dV


def attention_bwd_noalloc(Q, K, V, O, dO, lse, kv_of_q, dQ, dK, dV, stream=None):
    """``attention_bwd`` for callers that cannot allocate: no workspace, the
    scratch is a fixed 8 MiB array inside the library (n_q * S <= 1,048,576).
    Outputs are written into the caller's dQ, dK, dV."""
    torch = _torch()
    bf, f32 = torch.bfloat16, torch.float32
    n_q, S, d = Q.shape
    _check("upipe_attention_bwd_noalloc", lib().upipe_attention_bwd_noalloc(
        _ptr(Q, bf, "Q"), _ptr(K, bf, "K"), _ptr(V, bf, "V"), _ptr(O, bf, "O"), _ptr(dO, bf, "dO"),
        _ptr(lse, f32, "lse"), n_q, K.shape[0], S, d, _i32(kv_of_q), _ptr(dQ, f32, "dQ"), _ptr(dK, f32, "dK"),
        _ptr(dV, f32, "dV"), _stream(stream)))
    return dQ, dK, dV


def gemm(A, B, M, N, K, a_trans, b_trans, out_mode=1, D=None, stream=None):
    """D = A B on the tensor cores (see upipe_gemm_bf16).  out_mode 0 bf16, 1 fp32, 2 fp32 +=,
    3 fp32 += with split-K partial sums added atomically."""
    torch = _torch()
    bf = torch.bfloat16
    if D is None:
        D = torch.empty(M, N, dtype=bf if out_mode == 0 else torch.float32, device=A.device)
    _check("upipe_gemm_bf16", lib().upipe_gemm_bf16(
        _ptr(A, bf, "A"), _ptr(B, bf, "B"), _ptr(D), M, N, K, a_trans, b_trans,
        A.shape[1], B.shape[1], D.shape[1], out_mode, _stream(stream)))
    return D


def profile_enable(on=True):
    _check("upipe_profile_enable", lib().upipe_profile_enable(1 if on else 0))


def graphs_enable(on=True):
    """Replay layer calls with unchanged arguments as captured CUDA graphs (off clears the cache)."""
    _check("upipe_graphs_enable", lib().upipe_graphs_enable(1 if on else 0))


def profile_read():
    """{kind: (milliseconds, launches)} since the last read; waits for the events."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    _check("upipe_profile_read", lib().upipe_profile_read(ms, cnt))
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def sync_status(stream=None):
    _check("upipe_sync_status", lib().upipe_sync_status(_stream(stream)))
