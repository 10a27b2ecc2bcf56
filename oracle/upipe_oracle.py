"""fp64 oracle of the UPipe headwise-chunked causal GQA self-attention layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and ``bench.py``'s cpu baseline / reference arm may import or run this
module.  The CUDA library never calls it, and it imports nothing from the
library: the two share no code.  Inputs arrive as float64 arrays upcast
exactly from the bf16 bits made by ``synthetic``.

Plain and slow on purpose: materialised score matrices, one head at a time,
numpy matmul as the only library primitive.

Sources (page title and section):

[U1] "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise
     Chunking", summary page (paper.rainbus.top):
       - Background / DeepSpeed Ulysses: an all-to-all turns S/C-token
         sequence shards into all-token head shards and back.
       - Background / GQA: H query heads share G key/value heads, each KV
         head serving H/G query heads.
       - Motivation: Ulysses attention memory 12*(S/C)*H*d_head bytes.
       - Core method: H/U stages of U heads; buffers reused across stages;
         at U = C the peak is 12*S*d_head; Qwen3-32B (H=64, C=8) 96 vs 12.
       - Method steps (1)-(4): project X onto heads iU..(i+1)U-1 (QKV
         6*(S/C)*U*d_head bytes), all-to-all to U/C heads per rank (buffer
         6*(S/C)*U*d_head), attention, all-to-all back.
       - Novelty: GQA schedule processes heads out of order so every unique
         KV head is communicated in the first stage and later stages move
         query heads only.
       - Limitations: U must be divisible by C.
[U3] Same title, arXiv abstract (fugumt.com): chunking at the attention
     head level; up to 87.5% less intermediate memory for 32B models.

Readings where the pages are silent or garbled:
  * attention is softmax(Q K^T / sqrt(d_head) + causal mask) V with key j
    visible to query i iff j <= i; no bias, positional rotation or dropout;
  * query head h uses KV head h // (H/G) (contiguous groups);
  * in-order stage i holds heads iU..(i+1)U-1, rank r the r-th block of U/C;
    every query slot receives its own copy of its KV head, which is what
    makes the QKV exchange buffer exactly 6*(S/C)*U*d_head bytes;
  * out-of-order: rank r owns query heads r*H/C..(r+1)*H/C-1 over all
    stages, U/C of them per stage; the KV heads those use move once, in
    stage 0, and stay resident;
  * each stage adds its heads' share O_s W_o[rows of s] to Y;
  * the backward pass (absent from the pages) is the analytic gradient of
    L = <Y, dY>; only O and the log-sum-exp are kept from the forward pass.
"""
from __future__ import annotations

import numpy as np

IN_ORDER = 0
GQA_OUT_OF_ORDER = 1


# ---------------------------------------------------------------------------
# shapes, head grouping and schedules
# ---------------------------------------------------------------------------

def kv_head(h: int, H: int, G: int) -> int:
    """[U1] Background/GQA: each run of H/G consecutive query heads shares one KV head."""
    return h // (H // G)


def check_shape(S, d_model, H, G, d_head, U, C, order=IN_ORDER):
    """Divisibility the method needs: [U1] Limitations (C | U), Method steps
    (H/U stages of U heads, S/C tokens per rank), Background/GQA (G | H)."""
    if min(S, d_model, H, G, d_head, U, C) <= 0:
        raise ValueError("all sizes must be positive")
    if H % U:
        raise ValueError("U must divide H")
    if U % C:
        raise ValueError("C must divide U")
    if S % C:
        raise ValueError("C must divide S")
    if H % G:
        raise ValueError("G must divide H")
    if order == GQA_OUT_OF_ORDER and not (G % C == 0 or C % G == 0):
        raise ValueError("out-of-order schedule needs C | G or G | C")


def stage_heads(H: int, G: int, U: int, C: int, order: int = IN_ORDER) -> np.ndarray:
    """Query head held by (stage i, rank r, slot j): array [H/U, C, U/C].

    In order ([U1] Method steps (1)-(2)): stage i covers heads iU..(i+1)U-1
    and rank r receives the r-th run of U/C of them.
    Out of order ([U1] Novelty): rank r keeps the query heads of one block of
    H/C heads for every stage and works through them U/C at a time, so the KV
    heads it needs never change after stage 0.
    """
    n_stages, per_rank = H // U, U // C
    out = np.empty((n_stages, C, per_rank), dtype=np.int64)
    for i in range(n_stages):
        for r in range(C):
            for j in range(per_rank):
                if order == IN_ORDER:
                    out[i, r, j] = i * U + r * per_rank + j
                else:
                    out[i, r, j] = r * (H // C) + i * per_rank + j
    return out


def rank_kv_heads(H: int, G: int, U: int, C: int, r: int, order: int) -> list:
    """KV heads rank r holds resident under the out-of-order schedule: the set
    of KV heads its query heads use, over all stages ([U1] Novelty)."""
    sched = stage_heads(H, G, U, C, order)
    return sorted({kv_head(int(h), H, G) for h in sched[:, r, :].ravel()})


def kv_moves(H, G, U, C, order):
    """(stage, rank, kv head) triples for every KV head sent to a rank.

    In order, every query slot receives the KV head it uses, in every stage.
    Out of order, rank r receives its resident KV heads once, in stage 0.
    """
    sched = stage_heads(H, G, U, C, order)
    moves = []
    for i in range(H // U):
        for r in range(C):
            if order == IN_ORDER:
                for j in range(U // C):
                    moves.append((i, r, kv_head(int(sched[i, r, j]), H, G)))
            elif i == 0:
                for g in rank_kv_heads(H, G, U, C, r, order):
                    moves.append((0, r, g))
    return moves


# ---------------------------------------------------------------------------
# memory closed forms ([U1] Motivation, Core method, Method steps)
# ---------------------------------------------------------------------------

def ulysses_attention_bytes_per_rank(S, C, H, d_head):
    """[U1] Motivation: Ulysses keeps QKV and the all-to-all buffers of all H
    heads: 12*(S/C)*H*d_head bytes per device (16-bit elements)."""
    return 12 * (S // C) * H * d_head


def upipe_stage_bytes_per_rank(S, C, U, d_head):
    """[U1] Method steps (1)+(2): projected QKV 6*(S/C)*U*d_head bytes plus the
    exchange buffer of the same size; reused by every stage."""
    qkv = 6 * (S // C) * U * d_head
    exchange = 6 * (S // C) * U * d_head
    return qkv + exchange


def upipe_output_bytes_per_rank(S, C, U, d_head):
    """[U1] Method steps (3)+(4), with the printed d_model read as d_head (an
    output of U heads has U*d_head values per token): 2*(S/C)*U*d_head for the
    attention output and the same for its exchange buffer."""
    return 2 * (S // C) * U * d_head + 2 * (S // C) * U * d_head


# ---------------------------------------------------------------------------
# attention core (one query head against its KV head)
# ---------------------------------------------------------------------------

def causal_scores(q, k):
    """A = q k^T / sqrt(d_head) with -inf where key j comes after query i."""
    d = q.shape[1]
    A = (q @ k.T) / np.sqrt(d)
    n = q.shape[0]
    A[np.triu_indices(n, k=1)] = -np.inf
    return A


def attention_head_forward(q, k, v):
    """O = softmax(A) v per row; lse_i = ln sum_{j<=i} exp(A_ij).  Returns (O, lse, P)."""
    A = causal_scores(q, k)
    m = A.max(axis=1, keepdims=True)
    E = np.exp(A - m)
    l = E.sum(axis=1, keepdims=True)
    P = E / l
    return P @ v, (m + np.log(l))[:, 0], P


def attention_head_backward(q, k, v, P, o, do):
    """Analytic gradients of <O, dO> for one head: (dq, dk, dv).

    dv = P^T dO;  dP = dO v^T;  dA = P * (dP - rowsum(dO * O));
    dq = dA k / sqrt(d);  dk = dA^T q / sqrt(d).
    """
    d = q.shape[1]
    dv = P.T @ do
    dP = do @ v.T
    D = (do * o).sum(axis=1, keepdims=True)
    dA = P * (dP - D)
    dq = dA @ k / np.sqrt(d)
    dk = dA.T @ q / np.sqrt(d)
    return dq, dk, dv


def attention_rows(q, k, v, do, rows):
    """Forward and dQ of one head at the given query rows only (exact: row i
    needs keys 0..i).  Returns (O [n, d], lse [n], dQ [n, d]) for those rows."""
    d = q.shape[1]
    O, L, dQ = [], [], []
    for i in np.asarray(rows, dtype=np.int64):
        s = k[:i + 1] @ q[i] / np.sqrt(d)
        m = s.max()
        e = np.exp(s - m)
        p = e / e.sum()
        o = p @ v[:i + 1]
        dP = v[:i + 1] @ do[i]
        dA = p * (dP - do[i] @ o)
        O.append(o)
        L.append(m + np.log(e.sum()))
        dQ.append(dA @ k[:i + 1] / np.sqrt(d))
    return np.array(O), np.array(L), np.array(dQ)


# ---------------------------------------------------------------------------
# the layer, all heads at once (the definition)
# ---------------------------------------------------------------------------

def split_w_qkv(W_qkv, H, G, d_head):
    """W_qkv [d_model, (H+2G)*d_head] -> per-head column blocks (Wq[h], Wk[g], Wv[g])."""
    d = d_head
    Wq = [W_qkv[:, h * d:(h + 1) * d] for h in range(H)]
    Wk = [W_qkv[:, (H + g) * d:(H + g + 1) * d] for g in range(G)]
    Wv = [W_qkv[:, (H + G + g) * d:(H + G + g + 1) * d] for g in range(G)]
    return Wq, Wk, Wv


def layer_forward(X, W_qkv, W_o, H, G, d_head):
    """Y = [O_0 ... O_{H-1}] W_o with O_h = causal attention of head h.

    Returns (Y [S, d_model], O [S, H*d_head], lse [H, S]).
    """
    S = X.shape[0]
    d = d_head
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    K = [X @ Wk[g] for g in range(G)]
    V = [X @ Wv[g] for g in range(G)]
    O = np.zeros((S, H * d))
    lse = np.zeros((H, S))
    for h in range(H):
        g = kv_head(h, H, G)
        o, l, _ = attention_head_forward(X @ Wq[h], K[g], V[g])
        O[:, h * d:(h + 1) * d] = o
        lse[h] = l
    return O @ W_o, O, lse


def layer_backward(X, W_qkv, W_o, H, G, d_head, dY):
    """Gradients of L = <Y, dY>: returns (dX, dW_qkv, dW_o)."""
    S, d_model = X.shape
    d = d_head
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    K = [X @ Wk[g] for g in range(G)]
    V = [X @ Wv[g] for g in range(G)]
    dK = [np.zeros((S, d)) for _ in range(G)]
    dV = [np.zeros((S, d)) for _ in range(G)]
    O = np.zeros((S, H * d))
    dW_qkv = np.zeros_like(W_qkv)
    dX = np.zeros_like(X)
    for h in range(H):
        g = kv_head(h, H, G)
        q = X @ Wq[h]
        o, _, P = attention_head_forward(q, K[g], V[g])
        O[:, h * d:(h + 1) * d] = o
        do = dY @ W_o[h * d:(h + 1) * d, :].T
        dq, dk, dv = attention_head_backward(q, K[g], V[g], P, o, do)
        dK[g] += dk
        dV[g] += dv
        dW_qkv[:, h * d:(h + 1) * d] = X.T @ dq
        dX += dq @ Wq[h].T
    for g in range(G):
        dW_qkv[:, (H + g) * d:(H + g + 1) * d] = X.T @ dK[g]
        dW_qkv[:, (H + G + g) * d:(H + G + g + 1) * d] = X.T @ dV[g]
        dX += dK[g] @ Wk[g].T + dV[g] @ Wv[g].T
    dW_o = O.T @ dY
    return dX, dW_qkv, dW_o


def layer_backward_rows(X, W_qkv, W_o, H, G, d_head, dY, rows):
    """dX at the given rows only (exact).  Row t of dX needs dQ of query t
    (keys 0..t) and dK, dV of key t, which only the queries i >= t reach, so
    rows near the end of the sequence are cheap: each query i >= min(rows) is
    processed once, with its softmax row over keys 0..i."""
    rows = np.asarray(rows, dtype=np.int64)
    S = X.shape[0]
    d = d_head
    t0 = int(rows.min())
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    K = [X @ Wk[g] for g in range(G)]
    V = [X @ Wv[g] for g in range(G)]
    dX = np.zeros((len(rows), X.shape[1]))
    dK = np.zeros((G, len(rows), d))
    dV = np.zeros((G, len(rows), d))
    for h in range(H):
        g = kv_head(h, H, G)
        Wo_h = W_o[h * d:(h + 1) * d, :]
        for i in range(t0, S):
            q = X[i] @ Wq[h]
            s = K[g][:i + 1] @ q / np.sqrt(d)
            e = np.exp(s - s.max())
            p = e / e.sum()
            o = p @ V[g][:i + 1]
            do = dY[i] @ Wo_h.T
            dA = p * (V[g][:i + 1] @ do - do @ o)
            for r, t in enumerate(rows):
                if t <= i:  # key t is visible to query i
                    dK[g, r] += dA[t] * q / np.sqrt(d)
                    dV[g, r] += p[t] * do
                if t == i:
                    dX[r] += (dA @ K[g][:i + 1] / np.sqrt(d)) @ Wq[h].T
    for g in range(G):
        dX += dK[g] @ Wk[g].T + dV[g] @ Wv[g].T
    return dX


def layer_backward_sparse_dy(X, W_qkv, W_o, H, G, d_head, dY_rows, rows):
    """Every gradient (dX, dW_qkv, dW_o) of L = <Y, dY> for an upstream
    gradient dY that is zero outside the given query rows, dY[rows] = dY_rows.

    This is ``layer_backward`` with the zero rows left out, not an
    approximation: a row i with dY[i] = 0 has dO_h[i] = 0 for every head, so
    its dP row and its D are zero, its dA row is zero, and it adds nothing to
    dV = P^T dO, dK = dA^T q, dQ or dW_o = O^T dY.  Only the softmax rows of
    the listed queries are formed (each over keys 0..i), so the cost is
    |rows| x S per head instead of S x S, and the full-length K/V gradients,
    dW_qkv and every row of dX still come out exact."""
    rows = np.asarray(rows, dtype=np.int64)
    S = X.shape[0]
    d = d_head
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    Xr = X[rows]
    visible = np.arange(S)[None, :] <= rows[:, None]  # key j visible to query rows[r]
    dX = np.zeros_like(X)
    dW_qkv = np.zeros_like(W_qkv)
    O_rows = np.zeros((len(rows), H * d))
    for g in range(G):
        K = X @ Wk[g]
        V = X @ Wv[g]
        dK = np.zeros((S, d))
        dV = np.zeros((S, d))
        for h in range(H):
            if kv_head(h, H, G) != g:
                continue
            q = Xr @ Wq[h]
            A = np.where(visible, (q @ K.T) / np.sqrt(d), -np.inf)
            m = A.max(axis=1, keepdims=True)
            E = np.exp(A - m)
            P = E / E.sum(axis=1, keepdims=True)
            o = P @ V
            O_rows[:, h * d:(h + 1) * d] = o
            do = dY_rows @ W_o[h * d:(h + 1) * d, :].T
            dA = P * (do @ V.T - (do * o).sum(axis=1, keepdims=True))
            dq = dA @ K / np.sqrt(d)
            dK += dA.T @ q / np.sqrt(d)
            dV += P.T @ do
            dW_qkv[:, h * d:(h + 1) * d] = Xr.T @ dq
            dX[rows] += dq @ Wq[h].T
        dW_qkv[:, (H + g) * d:(H + g + 1) * d] = X.T @ dK
        dW_qkv[:, (H + G + g) * d:(H + G + g + 1) * d] = X.T @ dV
        dX += dK @ Wk[g].T + dV @ Wv[g].T
    return dX, dW_qkv, O_rows.T @ dY_rows


def layer_forward_rows(X, W_qkv, W_o, H, G, d_head, rows):
    """Y at the given query positions only (exact: each row needs keys 0..row)."""
    rows = np.asarray(rows, dtype=np.int64)
    d = d_head
    n = int(rows.max()) + 1
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    Xp = X[:n]
    K = [Xp @ Wk[g] for g in range(G)]
    V = [Xp @ Wv[g] for g in range(G)]
    O = np.zeros((len(rows), H * d))
    lse = np.zeros((H, len(rows)))
    for h in range(H):
        g = kv_head(h, H, G)
        q = X[rows] @ Wq[h]
        for t, i in enumerate(rows):
            a = (K[g][:i + 1] @ q[t]) / np.sqrt(d)
            m = a.max()
            e = np.exp(a - m)
            O[t, h * d:(h + 1) * d] = (e @ V[g][:i + 1]) / e.sum()
            lse[h, t] = m + np.log(e.sum())
    return O @ W_o, O, lse


# ---------------------------------------------------------------------------
# the all-to-all on C virtual ranks
# ---------------------------------------------------------------------------

def all_to_all(send):
    """send[c][r] is what rank c sends to rank r; returns recv with recv[r][c] = send[c][r]."""
    C = len(send)
    return [[send[c][r] for c in range(C)] for r in range(C)]


def seq_to_head(shards, wanted):
    """Ulysses input exchange ([U1] Background, Method steps (2)).

    shards[c]: dict head -> [S/C, d] block rank c computed for its tokens.
    wanted[r]: list of heads rank r must hold after the exchange.
    Returns per rank r an array [len(wanted[r]), S, d]: every wanted head over
    all S tokens, token blocks in rank order.
    """
    C = len(shards)
    send = [[np.stack([shards[c][h] for h in wanted[r]]) if wanted[r] else None
             for r in range(C)] for c in range(C)]
    recv = all_to_all(send)
    return [np.concatenate(recv[r], axis=1) if wanted[r] else None for r in range(C)]


def head_to_seq(held, heads_of, S):
    """Ulysses output exchange ([U1] Method steps (4)).

    held[r]: array [n_r, S, d] of the heads heads_of[r] on rank r.
    Returns per rank c a list of (head, [S/C, d] block) pairs, in the order the
    ranks send them (ascending source rank, then slot).
    """
    C = len(held)
    Sc = S // C
    send = [[[(h, held[r][j, c * Sc:(c + 1) * Sc]) for j, h in enumerate(heads_of[r])]
             for c in range(C)] for r in range(C)]
    recv = all_to_all(send)
    return [[pair for blocks in recv[c] for pair in blocks] for c in range(C)]


def replica_gradient_sum(copies):
    """Gradient of a head whose copies several ranks held, in the in-order
    exchange's backward (reading: every query slot receives its own copy of
    its KV head, [U1] Method steps (2); the copies' gradients are added in
    ascending rank order, in fp32).

    copies: [n, S, d] fp32 values, in ascending rank order.  Returns
    (sum32, rounded): the fp32 running sum copy_0 + copy_1 + ... evaluated
    left to right with float32 rounding after every addition, and that sum
    rounded once to bfloat16 (as float64 values)."""
    c = np.asarray(copies, dtype=np.float32)
    acc = c[0].copy()
    for x in c[1:]:
        acc = (acc + x).astype(np.float32)
    return acc, bf16_round(acc)


# ---------------------------------------------------------------------------
# the staged layer: H/U stages on C virtual ranks ([U1] Method steps)
# ---------------------------------------------------------------------------

def _stage_kv_wanted(sched_i, H, G, C, order, stage, resident):
    """KV heads each rank receives in this stage (one per query slot in order;
    the resident set in stage 0 only, out of order)."""
    if order == IN_ORDER:
        return [[kv_head(int(h), H, G) for h in sched_i[r]] for r in range(C)]
    return [list(resident[r]) if stage == 0 else [] for r in range(C)]


def staged_forward(X, W_qkv, W_o, H, G, d_head, U, C, order=IN_ORDER):
    """The layer run as H/U stages of U heads on C virtual ranks.

    Stage i: (1) each rank projects its S/C tokens onto the stage's heads;
    (2) all-to-all to head shards; (3) causal attention per held head;
    (4) all-to-all of the outputs back to sequence shards; then each rank adds
    the stage's heads' share of the output projection to its Y shard.
    Returns (Y, O [S, H*d], lse [H, S]) like ``layer_forward``.
    """
    S, d_model = X.shape
    check_shape(S, d_model, H, G, d_head, U, C, order)
    d, Sc = d_head, S // C
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    sched = stage_heads(H, G, U, C, order)
    resident = [rank_kv_heads(H, G, U, C, r, order) for r in range(C)] \
        if order == GQA_OUT_OF_ORDER else None
    Xs = [X[c * Sc:(c + 1) * Sc] for c in range(C)]
    Y = [np.zeros((Sc, d_model)) for _ in range(C)]
    O_saved = np.zeros((S, H * d))
    lse = np.zeros((H, S))
    K_held = V_held = None
    for i in range(H // U):
        q_wanted = [list(map(int, sched[i, r])) for r in range(C)]
        kv_wanted = _stage_kv_wanted(sched[i], H, G, C, order, i, resident)
        kv_needed = sorted({g for r in range(C) for g in kv_wanted[r]})
        # (1) projection on every rank's sequence shard
        Qs = [{h: Xs[c] @ Wq[h] for r in range(C) for h in q_wanted[r]} for c in range(C)]
        Ks = [{g: Xs[c] @ Wk[g] for g in kv_needed} for c in range(C)]
        Vs = [{g: Xs[c] @ Wv[g] for g in kv_needed} for c in range(C)]
        # (2) exchange to head shards
        Q_held = seq_to_head(Qs, q_wanted)
        if kv_needed:
            K_new, V_new = seq_to_head(Ks, kv_wanted), seq_to_head(Vs, kv_wanted)
            K_held = [(kv_wanted[r], K_new[r]) for r in range(C)]
            V_held = [(kv_wanted[r], V_new[r]) for r in range(C)]
        # (3) attention on each rank's heads
        O_held = []
        for r in range(C):
            outs = []
            for j, h in enumerate(q_wanted[r]):
                g = kv_head(h, H, G)
                slot = j if order == IN_ORDER else K_held[r][0].index(g)
                o, l, _ = attention_head_forward(Q_held[r][j], K_held[r][1][slot],
                                                 V_held[r][1][slot])
                outs.append(o)
                lse[h] = l
            O_held.append(np.stack(outs))
        # (4) exchange back, then the stage's share of the output projection
        O_back = head_to_seq(O_held, q_wanted, S)
        for c in range(C):
            for h, blk in O_back[c]:
                O_saved[c * Sc:(c + 1) * Sc, h * d:(h + 1) * d] = blk
                Y[c] += blk @ W_o[h * d:(h + 1) * d, :]
    return np.concatenate(Y), O_saved, lse


def staged_backward(X, W_qkv, W_o, H, G, d_head, U, C, dY, O_saved, lse, order=IN_ORDER):
    """Backward of the staged layer, stage by stage.

    Per stage: recompute (1)+(2) for the stage's heads; dO = dY W_o[rows]^T on
    each sequence shard, exchanged to head shards with the saved O; attention
    backward from the saved lse; the exchange back of dQ (and of dK, dV, whose
    per-slot copies are summed per KV head); then each rank adds its shard's
    share to dX and to the weight gradients.  Out of order, dK and dV stay on
    their resident ranks and go back once, after the last stage.
    Returns (dX, dW_qkv, dW_o).
    """
    S, d_model = X.shape
    check_shape(S, d_model, H, G, d_head, U, C, order)
    d, Sc = d_head, S // C
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    sched = stage_heads(H, G, U, C, order)
    resident = [rank_kv_heads(H, G, U, C, r, order) for r in range(C)] \
        if order == GQA_OUT_OF_ORDER else None
    Xs = [X[c * Sc:(c + 1) * Sc] for c in range(C)]
    dYs = [dY[c * Sc:(c + 1) * Sc] for c in range(C)]
    Os = [O_saved[c * Sc:(c + 1) * Sc] for c in range(C)]
    dX = [np.zeros((Sc, d_model)) for _ in range(C)]
    dW_qkv = np.zeros_like(W_qkv)
    dK_res = dV_res = None
    K_held = V_held = None
    for i in range(H // U):
        q_wanted = [list(map(int, sched[i, r])) for r in range(C)]
        kv_wanted = _stage_kv_wanted(sched[i], H, G, C, order, i, resident)
        kv_needed = sorted({g for r in range(C) for g in kv_wanted[r]})
        Qs = [{h: Xs[c] @ Wq[h] for r in range(C) for h in q_wanted[r]} for c in range(C)]
        Ks = [{g: Xs[c] @ Wk[g] for g in kv_needed} for c in range(C)]
        Vs = [{g: Xs[c] @ Wv[g] for g in kv_needed} for c in range(C)]
        dOs = [{h: dYs[c] @ W_o[h * d:(h + 1) * d, :].T for r in range(C) for h in q_wanted[r]}
               for c in range(C)]
        Osv = [{h: Os[c][:, h * d:(h + 1) * d] for r in range(C) for h in q_wanted[r]}
               for c in range(C)]
        Q_held = seq_to_head(Qs, q_wanted)
        dO_held = seq_to_head(dOs, q_wanted)
        O_held = seq_to_head(Osv, q_wanted)
        if kv_needed:
            K_new, V_new = seq_to_head(Ks, kv_wanted), seq_to_head(Vs, kv_wanted)
            K_held = [(kv_wanted[r], K_new[r]) for r in range(C)]
            V_held = [(kv_wanted[r], V_new[r]) for r in range(C)]
            if order == GQA_OUT_OF_ORDER:
                dK_res = [np.zeros_like(K_new[r]) for r in range(C)]
                dV_res = [np.zeros_like(V_new[r]) for r in range(C)]
        dQ_held, dK_slot, dV_slot = [], [], []
        for r in range(C):
            dq_r, dk_r, dv_r = [], [], []
            for j, h in enumerate(q_wanted[r]):
                g = kv_head(h, H, G)
                slot = j if order == IN_ORDER else K_held[r][0].index(g)
                k, v = K_held[r][1][slot], V_held[r][1][slot]
                q, o, do = Q_held[r][j], O_held[r][j], dO_held[r][j]
                # P rebuilt from the saved log-sum-exp
                P = np.exp(causal_scores(q, k) - lse[h][:, None])
                dq, dk, dv = attention_head_backward(q, k, v, P, o, do)
                dq_r.append(dq)
                if order == IN_ORDER:
                    dk_r.append(dk)
                    dv_r.append(dv)
                else:
                    dK_res[r][slot] += dk
                    dV_res[r][slot] += dv
            dQ_held.append(np.stack(dq_r))
            if order == IN_ORDER:
                dK_slot.append(np.stack(dk_r))
                dV_slot.append(np.stack(dv_r))
        dQ_back = head_to_seq(dQ_held, q_wanted, S)
        for c in range(C):
            for h, blk in dQ_back[c]:
                dX[c] += blk @ Wq[h].T
                dW_qkv[:, h * d:(h + 1) * d] += Xs[c].T @ blk
        if order == IN_ORDER:
            _kv_back_and_project(dK_slot, dV_slot, kv_wanted, Xs, Wk, Wv, dX, dW_qkv, H, G, d, S)
    if order == GQA_OUT_OF_ORDER:
        _kv_back_and_project(dK_res, dV_res, resident, Xs, Wk, Wv, dX, dW_qkv, H, G, d, S)
    dW_o = sum(Os[c].T @ dYs[c] for c in range(C))
    return np.concatenate(dX), dW_qkv, dW_o


def _kv_back_and_project(dK_held, dV_held, heads_of, Xs, Wk, Wv, dX, dW_qkv, H, G, d, S):
    """Exchange dK, dV back to sequence shards, sum the copies of each KV head
    (ascending source rank, then slot), and add their projection gradients."""
    C = len(Xs)
    dK_back = head_to_seq(dK_held, heads_of, S)
    dV_back = head_to_seq(dV_held, heads_of, S)
    for c in range(C):
        dk_sum, dv_sum = {}, {}
        for (g, blk) in dK_back[c]:
            dk_sum[g] = dk_sum.get(g, 0.0) + blk
        for (g, blk) in dV_back[c]:
            dv_sum[g] = dv_sum.get(g, 0.0) + blk
        for g in dk_sum:
            dX[c] += dk_sum[g] @ Wk[g].T + dv_sum[g] @ Wv[g].T
            dW_qkv[:, (H + g) * d:(H + g + 1) * d] += Xs[c].T @ dk_sum[g]
            dW_qkv[:, (H + G + g) * d:(H + G + g + 1) * d] += Xs[c].T @ dv_sum[g]


# ---------------------------------------------------------------------------
# head stages combined with sequence chunks ([U1] Limitations and Future
# directions: FPDT chunks the sequence, UPipe the heads; the two are
# orthogonal and the pages suggest combining them)
# ---------------------------------------------------------------------------

def chunk_scores(q, k, q_pos, k_pos):
    """Scores of a query chunk whose first row sits at sequence position q_pos
    against a key chunk starting at k_pos: q k^T / sqrt(d), -inf where the
    key's position is after the query's."""
    A = (q @ k.T) / np.sqrt(q.shape[1])
    qi = q_pos + np.arange(q.shape[0])[:, None]
    kj = k_pos + np.arange(k.shape[0])[None, :]
    A[kj > qi] = -np.inf
    return A


def partial_attention(q, k, v, q_pos, k_pos):
    """Attention of a query chunk over one key chunk: the normalised partial
    output and its log-sum-exp (every row sees at least one key)."""
    A = chunk_scores(q, k, q_pos, k_pos)
    m = A.max(axis=1, keepdims=True)
    E = np.exp(A - m)
    l = E.sum(axis=1, keepdims=True)
    return (E / l) @ v, (m + np.log(l))[:, 0]


def merge_partials(o_a, lse_a, o_b, lse_b):
    """Softmax over the union of two disjoint key sets from the two partial
    results: weights exp(lse_x - lse) with lse = log(exp(lse_a) + exp(lse_b))."""
    lse = np.logaddexp(lse_a, lse_b)
    return o_a * np.exp(lse_a - lse)[:, None] + o_b * np.exp(lse_b - lse)[:, None], lse


def _check_chunks(S, C, n_chunks):
    if n_chunks <= 0 or S % n_chunks or (S // n_chunks) % C:
        raise ValueError("n_chunks must divide S into chunks the C ranks split evenly")


def chunked_forward(X, W_qkv, W_o, H, G, d_head, U, C, n_chunks):
    """The in-order head stages run on sequence chunks of S/n_chunks tokens.

    For chunk i (ascending) and stage s: project the chunk's rows onto the
    stage's Q heads and the KV heads they use; the chunk's K and V go to an
    offload store; each query head attends to KV chunks 0..i of the store, the
    partial results merged by log-sum-exp; the stage's share of the output
    projection is added to the chunk's rows of Y.  Returns (Y, O, lse) like
    ``layer_forward``.
    """
    S, d_model = X.shape
    check_shape(S, d_model, H, G, d_head, U, C, IN_ORDER)
    _check_chunks(S, C, n_chunks)
    d, Sc = d_head, S // n_chunks
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    sched = stage_heads(H, G, U, C, IN_ORDER)
    store_K, store_V = {}, {}
    Y = np.zeros((S, d_model))
    O = np.zeros((S, H * d))
    lse = np.zeros((H, S))
    for i in range(n_chunks):
        rows = slice(i * Sc, (i + 1) * Sc)
        Xi = X[rows]
        for st in range(H // U):
            heads = [int(h) for h in sched[st].reshape(-1)]
            for g in sorted({kv_head(h, H, G) for h in heads}):
                store_K[g, i] = Xi @ Wk[g]
                store_V[g, i] = Xi @ Wv[g]
            for h in heads:
                g = kv_head(h, H, G)
                q = Xi @ Wq[h]
                o, l = partial_attention(q, store_K[g, 0], store_V[g, 0], i * Sc, 0)
                for j in range(1, i + 1):
                    o_j, l_j = partial_attention(q, store_K[g, j], store_V[g, j], i * Sc, j * Sc)
                    o, l = merge_partials(o, l, o_j, l_j)
                O[rows, h * d:(h + 1) * d] = o
                lse[h, rows] = l
                Y[rows] += o @ W_o[h * d:(h + 1) * d, :]
    return Y, O, lse


def chunked_backward(X, W_qkv, W_o, H, G, d_head, U, C, n_chunks, dY, O_saved, lse):
    """Backward of ``chunked_forward``: query chunks in descending order.

    The K and V chunks are recomputed into the store first.  For query chunk i
    and stage s, each head's P against KV chunk j <= i is rebuilt from the
    saved log-sum-exp; dQ of the chunk sums over j, dK and dV of chunk j sum
    over the query chunks i >= j (and the query heads of the KV head).  Chunk
    i's dK, dV are complete once query chunk i is done (later chunks came
    first), and go into dX and dW_qkv then.  Returns (dX, dW_qkv, dW_o).
    """
    S, d_model = X.shape
    check_shape(S, d_model, H, G, d_head, U, C, IN_ORDER)
    _check_chunks(S, C, n_chunks)
    d, Sc = d_head, S // n_chunks
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    sched = stage_heads(H, G, U, C, IN_ORDER)
    store_K = {(g, j): X[j * Sc:(j + 1) * Sc] @ Wk[g] for g in range(G) for j in range(n_chunks)}
    store_V = {(g, j): X[j * Sc:(j + 1) * Sc] @ Wv[g] for g in range(G) for j in range(n_chunks)}
    dK = {key: np.zeros((Sc, d)) for key in store_K}
    dV = {key: np.zeros((Sc, d)) for key in store_V}
    dX = np.zeros_like(X)
    dW_qkv = np.zeros_like(W_qkv)
    for i in reversed(range(n_chunks)):
        rows = slice(i * Sc, (i + 1) * Sc)
        Xi = X[rows]
        for st in range(H // U):
            for h in [int(h) for h in sched[st].reshape(-1)]:
                g = kv_head(h, H, G)
                q = Xi @ Wq[h]
                do = dY[rows] @ W_o[h * d:(h + 1) * d, :].T
                Dsum = (do * O_saved[rows, h * d:(h + 1) * d]).sum(axis=1, keepdims=True)
                dq = np.zeros((Sc, d))
                for j in range(i + 1):
                    k, v = store_K[g, j], store_V[g, j]
                    P = np.exp(chunk_scores(q, k, i * Sc, j * Sc) - lse[h, rows][:, None])
                    dV[g, j] += P.T @ do
                    dA = P * (do @ v.T - Dsum)
                    dq += dA @ k / np.sqrt(d)
                    dK[g, j] += dA.T @ q / np.sqrt(d)
                dX[rows] += dq @ Wq[h].T
                dW_qkv[:, h * d:(h + 1) * d] += Xi.T @ dq
        for g in range(G):
            dX[rows] += dK[g, i] @ Wk[g].T + dV[g, i] @ Wv[g].T
            dW_qkv[:, (H + g) * d:(H + g + 1) * d] += Xi.T @ dK[g, i]
            dW_qkv[:, (H + G + g) * d:(H + G + g + 1) * d] += Xi.T @ dV[g, i]
    return dX, dW_qkv, O_saved.T @ dY


# ---------------------------------------------------------------------------
# lower-precision heads ([U1] weaknesses from an independent analysis: some
# heads could run in FP8 to cut memory and communication further)
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0
FP8_BLOCK = 128  # keys per K scale


def e4m3_round(x):
    """Nearest value of the FP8 E4M3 format (1 sign, 4 exponent bits with
    bias 7, 3 mantissa bits; no infinities; largest finite 448; subnormals
    m * 2^-9), ties to the even mantissa, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # spacing of the format around |x|: 2^(e-3) in binade [2^e, 2^(e+1)), e >= -6
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    q = 2.0 ** (e - 3)
    r = np.round(a / q) * q  # numpy rounds half to even, and a/q is exact
    r = np.minimum(r, E4M3_MAX)
    return np.where(a > 0, np.sign(x) * r, 0.0 * x)


def bf16_round(x):
    """Nearest bfloat16 value (8 exponent bits, 7 mantissa bits), ties to the
    even mantissa: the top 16 bits of the fp32 pattern after adding half a
    unit of the dropped 16 bits (plus the kept LSB for ties).  x is rounded to
    fp32 first."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def fp8_scale(amax):
    """Per-group scale: amax / 448 in fp32 (1 for an all-zero group)."""
    amax = np.float32(amax)
    return np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))


def quantize_e4m3(x, scale):
    """Codes of x (fp32 values) under one fp32 scale: e4m3(fl32(x / scale)),
    returned as their values (exact in fp64)."""
    return e4m3_round(np.asarray(x, dtype=np.float32) / np.float32(scale))


def fp8_rows(q):
    """Q of one head [S, d] -> (codes [S, d], scales [S]): one scale per row."""
    sc = np.array([fp8_scale(np.abs(np.float32(r)).max()) for r in np.asarray(q, dtype=np.float32)], dtype=np.float32)
    return np.stack([quantize_e4m3(r, s) for r, s in zip(np.asarray(q, dtype=np.float32), sc)]), sc


def fp8_key_blocks(k):
    """K of one head [S, d] -> (codes, scales [S / 128]): one scale per block of
    128 consecutive keys."""
    k = np.asarray(k, dtype=np.float32)
    codes, scales = np.zeros(k.shape), []
    for b in range(0, k.shape[0], FP8_BLOCK):
        s = fp8_scale(np.abs(k[b:b + FP8_BLOCK]).max())
        codes[b:b + FP8_BLOCK] = quantize_e4m3(k[b:b + FP8_BLOCK], s)
        scales.append(s)
    return codes, np.array(scales, dtype=np.float32)


def attention_head_forward_fp8(q, k, v):
    """Causal attention whose scores use FP8 Q and K: q = codes * row scale,
    k = codes * block scale, then the exact softmax and P V.  Returns (O, lse)."""
    qd, kd = fp8_dequantized(q, k)
    o, lse, _ = attention_head_forward(qd, kd, v)
    return o, lse


def fp8_dequantized(q, k):
    """The operands the FP8 score path multiplies, as values: q = codes x its
    row's scale, k = codes x its 128-key block's scale (exact in fp64)."""
    cq, sq = fp8_rows(q)
    ck, sk = fp8_key_blocks(k)
    qd = cq * sq.astype(np.float64)[:, None]
    kd = ck * np.repeat(sk.astype(np.float64), FP8_BLOCK)[:k.shape[0], None]
    return qd, kd


def attention_head_backward_fp8(q, k, v, do):
    """Gradients of <O, dO> for a head attending with FP8 scores
    (``attention_head_forward_fp8``).  O depends on q and k only through the
    dequantized operands q~, k~ (``fp8_dequantized``); the attention is
    differentiated exactly in q~, k~ and v, and the rounding to E4M3, whose
    derivative is zero almost everywhere, is passed through as the identity
    (straight-through): dq = dq~, dk = dk~.  Returns (dq, dk, dv)."""
    qd, kd = fp8_dequantized(q, k)
    o, _, P = attention_head_forward(qd, kd, v)
    return attention_head_backward(qd, kd, v, P, o, do)


def layer_forward_fp8(X, W_qkv, W_o, H, G, d_head, fp8_heads):
    """``layer_forward`` with the heads in fp8_heads attending through FP8
    Q and K (``attention_head_forward_fp8``); other heads are unchanged.  The
    codes are decided from the projections as the exchange holds them, in
    bf16: a quantised code is an integer the two sides must decide from the
    same value."""
    S = X.shape[0]
    d = d_head
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    K = [X @ Wk[g] for g in range(G)]
    V = [X @ Wv[g] for g in range(G)]
    O = np.zeros((S, H * d))
    lse = np.zeros((H, S))
    for h in range(H):
        g = kv_head(h, H, G)
        if h in fp8_heads:
            o, l = attention_head_forward_fp8(bf16_round(X @ Wq[h]), bf16_round(K[g]), V[g])
        else:
            o, l, _ = attention_head_forward(X @ Wq[h], K[g], V[g])
        O[:, h * d:(h + 1) * d] = o
        lse[h] = l
    return O @ W_o, O, lse


def layer_backward_fp8(X, W_qkv, W_o, H, G, d_head, dY, fp8_heads):
    """``layer_backward`` of ``layer_forward_fp8``: the heads in fp8_heads
    take their attention gradients from ``attention_head_backward_fp8`` on the
    bf16-rounded projections (the values their codes are decided from), the
    others from the plain attention.  The projection gradients then follow as
    in ``layer_backward``.  Returns (dX, dW_qkv, dW_o)."""
    S = X.shape[0]
    d = d_head
    Wq, Wk, Wv = split_w_qkv(W_qkv, H, G, d)
    K = [X @ Wk[g] for g in range(G)]
    V = [X @ Wv[g] for g in range(G)]
    dK = [np.zeros((S, d)) for _ in range(G)]
    dV = [np.zeros((S, d)) for _ in range(G)]
    O = np.zeros((S, H * d))
    dW_qkv = np.zeros_like(W_qkv)
    dX = np.zeros_like(X)
    for h in range(H):
        g = kv_head(h, H, G)
        q = X @ Wq[h]
        do = dY @ W_o[h * d:(h + 1) * d, :].T
        if h in fp8_heads:
            qb, kb = bf16_round(q), bf16_round(K[g])
            qd, kd = fp8_dequantized(qb, kb)
            o, _, _ = attention_head_forward(qd, kd, V[g])
            dq, dk, dv = attention_head_backward_fp8(qb, kb, V[g], do)
        else:
            o, _, P = attention_head_forward(q, K[g], V[g])
            dq, dk, dv = attention_head_backward(q, K[g], V[g], P, o, do)
        O[:, h * d:(h + 1) * d] = o
        dK[g] += dk
        dV[g] += dv
        dW_qkv[:, h * d:(h + 1) * d] = X.T @ dq
        dX += dq @ Wq[h].T
    for g in range(G):
        dW_qkv[:, (H + g) * d:(H + g + 1) * d] = X.T @ dK[g]
        dW_qkv[:, (H + G + g) * d:(H + G + g + 1) * d] = X.T @ dV[g]
        dX += dK[g] @ Wk[g].T + dV[g] @ Wv[g].T
    return dX, dW_qkv, O.T @ dY


# ---------------------------------------------------------------------------
# FLOP accounting (model FLOPs; not a method step)
# ---------------------------------------------------------------------------

def layer_model_flops(S, d_model, H, G, d_head):
    """Forward model FLOPs of the layer: projections plus causal attention
    (half of the dense QK^T and PV); fwd+bwd counts 3x this."""
    proj = 2 * S * d_model * (H + 2 * G) * d_head
    out = 2 * S * H * d_head * d_model
    attn = 2 * S * S * H * d_head  # (2 matmuls x 2 flops x S^2/2)
    return proj + out + attn
