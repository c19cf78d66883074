"""fp64 CPU oracle for block-sparse attention (backward, forward, mask compaction).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. It shares no code
with the CUDA path and imports nothing from it.

Everything is computed in float64 from exact up-conversions of the inputs.
The sources it follows (all from the ``aclnnBlockSparseAttentionGrad`` page,
"CANN/ops-transformer块稀疏注意力梯度算子", unless said otherwise):

* forward, section 计算公式 (formulas): S = scale*Q*K_sparse^T, P = Softmax(S),
  Out = P*V, with K_sparse the keys of the blocks the BlockSparseMask selects;
* backward, same section: softmax_grad = softmaxGrad(dOut, attentionOut),
  dP = dOut*V^T, dS = P*(dP - softmax_grad), dV = P^T*dOut,
  dQ = (dS*K)*scale, dK = (dS^T*Q)*scale;
* layouts BNSD / TND and actualSeqLengths(Kv), section 参数说明 (parameter
  table), rows dout/query/key/value/softmaxLse/actualSeqLengthsOptional;
* blockSparseMaskOptional [B, N, ceil(Sq/bx), ceil(Skv/by)], 1 = the block takes
  part, nullptr = every token pair takes part; blockShapeOptional [bx, by],
  default [128, 128] (same table);
* numKeyValueHeads: N1 % N2 == 0 (section 约束说明, constraints).

Readings of points the pages leave open (numbered; the same numbers are used
wherever the project refers to them):

R1  softmaxGrad(dOut, attentionOut) is the row vector D_s = sum_d dOut_sd*Out_sd
    (the softmax Jacobian-vector product that makes dS = P*(dP - D) exact).
R2  softmaxLse is the natural-log logsumexp of the *scaled* scores over the
    selected keys, so P = exp(scale*q.k - lse). The backward uses the given
    attentionOut and softmaxLse as they are (it never recomputes them).
R3  Query head h reads key/value head g = h // (N1/N2) (contiguous groups);
    dK/dV of head g sum the contributions of all query heads of the group.
R4  Only tokens below the per-batch actual lengths count; mask bits of blocks
    starting at or beyond them are ignored. Output rows at or beyond the actual
    length (BNSD padding) are 0.
R5  Inside a selected block every token pair takes part unless the sliding
    window of R18 or the token mask of R19 excludes it.
R6  A query row with no selected key has Out = 0 and lse = -inf in the forward
    and contributes nothing in the backward (its dQ row is 0).
R7  In TND, actualSeqLengths are per-batch counts; batch b starts at the
    exclusive prefix sum of the counts.
R18 preTokens / nextTokens (parameter table rows preTokens, nextTokens: how
    many earlier / later tokens a token may attend to; FlashAttentionScore
    page, 参数说明: left / right edge of the sliding window, and 约束说明: the
    two must overlap). Query s and key t of one sequence, both counted from 0
    at the start of that sequence, form a pair of the window iff
    s - preTokens <= t <= s + nextTokens; a pair takes part iff its block is
    selected AND it lies in the window. preTokens + nextTokens >= 0 (the
    window is never empty on the diagonal). 2147483647 for both (the only
    value the page's own build accepts) is no window for any sequence shorter
    than 2^31. nextTokens = 0 with preTokens = 2147483647 is the causal
    (lower-triangular, top-left aligned) mask.
R19 attenMaskOptional (parameter table: the atten_mask of the formula
    S = Mask(scale*Q*K^T, atten_mask), BOOL, 2 dimensions; FlashAttentionScore
    page, 参数说明 and 实现原理: a true entry masks the position out, a false one
    keeps it). A 2-D [maxSq, maxSkv] matrix shared by every batch and head,
    indexed like the window by the positions s, t counted from each
    sequence's start; pair (s, t) takes part iff atten_mask[s, t] == 0, on top
    of the block mask and the window. maskType 0 = no token mask (attenMask
    absent), maskType 1 = the given attenMask.
"""
from __future__ import annotations

import numpy as np

__all__ = ["token_mask", "token_mask_at", "window_mask", "head_rows", "forward",
           "forward_blockrows", "backward", "backward_blockrows", "backward_dq_rows",
           "backward_dkdv_rows", "compact_mask", "seq_offsets", "NO_WINDOW"]

NO_WINDOW = 2147483647   # preTokens / nextTokens value for "no sliding window" (R18)


# --------------------------------------------------------------------------
# layout helpers (parameter table: BNSD [B,N,S,D], TND [T,N,D])
# --------------------------------------------------------------------------
def seq_offsets(lengths):
    """Exclusive prefix sum of per-batch token counts (reading R7)."""
    off = [0]
    for n in lengths:
        off.append(off[-1] + int(n))
    return off


def head_rows(x, layout, b, h, length, offsets):
    """The [length, D] fp64 matrix of batch b, head h of a BNSD or TND tensor."""
    if layout == "BNSD":
        return np.asarray(x[b, h, :length, :], dtype=np.float64)
    o = offsets[b]
    return np.asarray(x[o:o + length, h, :], dtype=np.float64)


def _lse_rows(lse, layout, b, h, length, offsets):
    lse = np.asarray(lse)
    if layout == "BNSD":
        return np.asarray(lse.reshape(lse.shape[0], lse.shape[1], -1)[b, h, :length],
                          dtype=np.float64)
    o = offsets[b]
    return np.asarray(lse.reshape(lse.shape[0], lse.shape[1])[o:o + length, h],
                      dtype=np.float64)


def window_mask(rows, cols, pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW):
    """[len(rows), len(cols)] bool: query position s = rows[i] and key position
    t = cols[j] (both counted from the start of their sequence) satisfy
    s - preTokens <= t <= s + nextTokens (reading R18)."""
    s = np.asarray(rows, dtype=np.int64)[:, None]
    t = np.asarray(cols, dtype=np.int64)[None, :]
    # |t - s| < 2^31, so limits beyond +-2^40 act as no limit; clipping them
    # only keeps the int64 arithmetic away from overflow
    pre = max(-(1 << 40), min(1 << 40, int(pre_tokens)))
    nxt = max(-(1 << 40), min(1 << 40, int(next_tokens)))
    return (t >= s - pre) & (t <= s + nxt)


def token_mask(block_mask, bx, by, Lq, Lk, pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW,
               atten_mask=None):
    """Token-level [Lq, Lk] bool mask of one (b, h): pair (s, t) takes part iff
    the block (s // bx, t // by) is selected (parameter table,
    blockSparseMaskOptional; ``None`` = every block), (s, t) lies in the
    sliding window (R18) and atten_mask[s, t] is 0 (R19; ``None`` = no mask)."""
    return token_mask_at(block_mask, bx, by, np.arange(Lq), np.arange(Lk),
                         pre_tokens, next_tokens, atten_mask)


def token_mask_at(block_mask, bx, by, rows, cols, pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW,
                  atten_mask=None):
    """The entries [rows x cols] of :func:`token_mask` only (same definition,
    evaluated on the requested query rows and key columns)."""
    rows, cols = np.asarray(rows), np.asarray(cols)
    if block_mask is None:
        sel = np.ones((len(rows), len(cols)), dtype=bool)
    else:
        bm = np.asarray(block_mask) != 0
        sel = bm[(rows // bx)[:, None], (cols // by)[None, :]]
    sel = sel & window_mask(rows, cols, pre_tokens, next_tokens)
    if atten_mask is not None:
        sel = sel & (np.asarray(atten_mask)[rows[:, None], cols[None, :]] == 0)
    return sel


def _dims(q, k, layout):
    if layout == "BNSD":
        B, N1, _, D = q.shape
        N2 = k.shape[1]
    else:
        _, N1, D = q.shape
        N2 = k.shape[1]
        B = None
    return B, N1, N2, D


def _lengths(q, k, layout, seq_q, seq_kv):
    if layout == "BNSD":
        B, Sq, Skv = q.shape[0], q.shape[2], k.shape[2]
        lq = [Sq] * B if seq_q is None else [int(x) for x in seq_q]
        lk = [Skv] * B if seq_kv is None else [int(x) for x in seq_kv]
        return B, lq, lk
    lq = [int(x) for x in seq_q]
    lk = [int(x) for x in seq_kv]
    return len(lq), lq, lk


# --------------------------------------------------------------------------
# forward (formulas: S = scale*Q*K_sparse^T, P = Softmax(S), Out = P*V)
# --------------------------------------------------------------------------
def _head_forward(Qm, Km, Vm, M, scale):
    """One (b, h): returns out [Lq, D], lse [Lq] in fp64 (readings R2, R6)."""
    S = scale * (Qm @ Km.T)
    S = np.where(M, S, -np.inf)
    has = M.any(axis=1)
    mx = np.where(has, S.max(axis=1, initial=-np.inf), 0.0)
    E = np.where(M, np.exp(S - mx[:, None]), 0.0)
    ssum = E.sum(axis=1)
    lse = np.where(has, mx + np.log(np.where(has, ssum, 1.0)), -np.inf)
    P = np.where(has[:, None], E / np.where(has, ssum, 1.0)[:, None], 0.0)
    return P @ Vm, lse


def forward(q, k, v, mask=None, block_shape=(128, 128), seq_q=None, seq_kv=None,
            layout="BNSD", num_kv_heads=None, scale=1.0, pre_tokens=NO_WINDOW,
            next_tokens=NO_WINDOW, atten_mask=None):
    """Plain dense-with-mask forward. Returns (out, lse) in the layout's shapes
    (lse with the trailing 1), fp64. Padding rows: out 0, lse -inf (R4, R6)."""
    bx, by = int(block_shape[0]), int(block_shape[1])
    B, lq, lk = _lengths(q, k, layout, seq_q, seq_kv)
    _, N1, N2, D = _dims(q, k, layout)
    G = N1 // N2
    oq, okv = seq_offsets(lq), seq_offsets(lk)
    out = np.zeros(q.shape, dtype=np.float64)
    if layout == "BNSD":
        lse = np.full((B, N1, q.shape[2], 1), -np.inf)
    else:
        lse = np.full((q.shape[0], N1, 1), -np.inf)
    for b in range(B):
        for h in range(N1):
            g = h // G
            Qm = head_rows(q, layout, b, h, lq[b], oq)
            Km = head_rows(k, layout, b, g, lk[b], okv)
            Vm = head_rows(v, layout, b, g, lk[b], okv)
            M = token_mask(None if mask is None else mask[b, h], bx, by, lq[b], lk[b],
                           pre_tokens, next_tokens, atten_mask)
            o, l = _head_forward(Qm, Km, Vm, M, scale)
            if layout == "BNSD":
                out[b, h, :lq[b]] = o
                lse[b, h, :lq[b], 0] = l
            else:
                out[oq[b]:oq[b] + lq[b], h] = o
                lse[oq[b]:oq[b] + lq[b], h, 0] = l
    return out, lse


def forward_blockrows(q, k, v, mask=None, block_shape=(128, 128), seq_q=None,
                      seq_kv=None, layout="BNSD", num_kv_heads=None, scale=1.0,
                      pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW, atten_mask=None):
    """The same forward, evaluated per query block row over that row's selected
    key set K(s) only (every query row of a block row has the same K(s)). Used
    where the dense [Lq, Lk] score matrix would not fit in host memory; pinned
    to :func:`forward` by the tests."""
    bx, by = int(block_shape[0]), int(block_shape[1])
    B, lq, lk = _lengths(q, k, layout, seq_q, seq_kv)
    _, N1, N2, D = _dims(q, k, layout)
    G = N1 // N2
    oq, okv = seq_offsets(lq), seq_offsets(lk)
    out = np.zeros(q.shape, dtype=np.float64)
    if layout == "BNSD":
        lse = np.full((B, N1, q.shape[2], 1), -np.inf)
    else:
        lse = np.full((q.shape[0], N1, 1), -np.inf)
    for b in range(B):
        mq = -(-lq[b] // bx)
        mk = -(-lk[b] // by)
        for h in range(N1):
            g = h // G
            Qh = head_rows(q, layout, b, h, lq[b], oq)
            Kh = head_rows(k, layout, b, g, lk[b], okv)
            Vh = head_rows(v, layout, b, g, lk[b], okv)
            for i in range(mq):
                s0, s1 = i * bx, min(lq[b], (i + 1) * bx)
                if mask is None:
                    sel = np.arange(mk)
                else:
                    sel = np.nonzero(np.asarray(mask[b, h, i, :mk]) != 0)[0]
                if len(sel) == 0:
                    continue
                keys = np.concatenate([np.arange(j * by, min(lk[b], (j + 1) * by))
                                       for j in sel])
                M = window_mask(np.arange(s0, s1), keys, pre_tokens, next_tokens)
                if atten_mask is not None:
                    M = M & (np.asarray(atten_mask)[s0:s1][:, keys] == 0)
                o, l = _head_forward(Qh[s0:s1], Kh[keys], Vh[keys], M, scale)
                if layout == "BNSD":
                    out[b, h, s0:s1] = o
                    lse[b, h, s0:s1, 0] = l
                else:
                    out[oq[b] + s0:oq[b] + s1, h] = o
                    lse[oq[b] + s0:oq[b] + s1, h, 0] = l
    return out, lse


# --------------------------------------------------------------------------
# backward (formulas: dP = dOut*V^T, dS = P*(dP - softmax_grad), dV = P^T*dOut,
#                     dQ = (dS*K)*scale, dK = (dS^T*Q)*scale)
# --------------------------------------------------------------------------
def _head_backward(Qm, Km, Vm, dOm, Om, lse, M, scale):
    """One (b, h) with its token mask M [Lq, Lk]. Returns dQ [Lq, D] and this
    head's contributions dK, dV [Lk, D] (readings R1, R2, R5)."""
    Dv = (dOm * Om).sum(axis=1)                                     # R1
    S = scale * (Qm @ Km.T)
    P = np.where(M, np.exp(np.where(M, S - lse[:, None], 0.0)), 0.0)  # R2
    dP = dOm @ Vm.T
    dS = P * (dP - Dv[:, None])
    dV = P.T @ dOm
    dQ = scale * (dS @ Km)
    dK = scale * (dS.T @ Qm)
    return dQ, dK, dV


def backward(dout, q, k, v, out, lse, mask=None, block_shape=(128, 128), seq_q=None,
             seq_kv=None, layout="BNSD", num_kv_heads=None, scale=1.0, pre_tokens=NO_WINDOW,
             next_tokens=NO_WINDOW, atten_mask=None):
    """Full dQ, dK, dV (fp64, the layout's shapes) from the given Out and lse."""
    bx, by = int(block_shape[0]), int(block_shape[1])
    B, lq, lk = _lengths(q, k, layout, seq_q, seq_kv)
    _, N1, N2, D = _dims(q, k, layout)
    G = N1 // N2
    oq, okv = seq_offsets(lq), seq_offsets(lk)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for b in range(B):
        for h in range(N1):
            g = h // G                                                   # R3
            Qm = head_rows(q, layout, b, h, lq[b], oq)
            Km = head_rows(k, layout, b, g, lk[b], okv)
            Vm = head_rows(v, layout, b, g, lk[b], okv)
            dOm = head_rows(dout, layout, b, h, lq[b], oq)
            Om = head_rows(out, layout, b, h, lq[b], oq)
            L = _lse_rows(lse, layout, b, h, lq[b], oq)
            M = token_mask(None if mask is None else mask[b, h], bx, by, lq[b], lk[b],
                           pre_tokens, next_tokens, atten_mask)
            dQ, dK, dV = _head_backward(Qm, Km, Vm, dOm, Om, L, M, scale)
            if layout == "BNSD":
                dq[b, h, :lq[b]] = dQ
                dk[b, g, :lk[b]] += dK
                dv[b, g, :lk[b]] += dV
            else:
                dq[oq[b]:oq[b] + lq[b], h] = dQ
                dk[okv[b]:okv[b] + lk[b], g] += dK
                dv[okv[b]:okv[b] + lk[b], g] += dV
    return dq, dk, dv


def backward_blockrows(dout, q, k, v, out, lse, mask=None, block_shape=(128, 128), seq_q=None,
                       seq_kv=None, layout="BNSD", num_kv_heads=None, scale=1.0,
                       pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW, atten_mask=None):
    """The same full dQ, dK, dV as :func:`backward`, evaluated per query block
    row over that row's selected key set only (every query row of a block row
    has the same K(s)): the row's dQ comes out whole, and its contributions to
    dK / dV of the selected keys are added to those keys' rows (the sums over s
    of the formulas, taken block row by block row). Used where the dense
    [Lq, Lk] matrices would not fit in host memory; pinned to
    :func:`backward` by the tests."""
    bx, by = int(block_shape[0]), int(block_shape[1])
    B, lq, lk = _lengths(q, k, layout, seq_q, seq_kv)
    _, N1, N2, D = _dims(q, k, layout)
    G = N1 // N2
    oq, okv = seq_offsets(lq), seq_offsets(lk)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for b in range(B):
        mq = -(-lq[b] // bx)
        mk = -(-lk[b] // by)
        for g in range(N2):
            Kh = head_rows(k, layout, b, g, lk[b], okv)
            Vh = head_rows(v, layout, b, g, lk[b], okv)
            dKh = np.zeros((lk[b], D))
            dVh = np.zeros((lk[b], D))
            for h in range(g * G, (g + 1) * G):                          # R3
                Qh = head_rows(q, layout, b, h, lq[b], oq)
                dOh = head_rows(dout, layout, b, h, lq[b], oq)
                Oh = head_rows(out, layout, b, h, lq[b], oq)
                Lh = _lse_rows(lse, layout, b, h, lq[b], oq)
                dQh = np.zeros((lq[b], D))
                for i in range(mq):
                    s0, s1 = i * bx, min(lq[b], (i + 1) * bx)
                    if mask is None:
                        sel = np.arange(mk)
                    else:
                        sel = np.nonzero(np.asarray(mask[b, h, i, :mk]) != 0)[0]
                    if len(sel) == 0:
                        continue                                          # R6
                    keys = np.concatenate([np.arange(j * by, min(lk[b], (j + 1) * by))
                                           for j in sel])
                    M = window_mask(np.arange(s0, s1), keys, pre_tokens, next_tokens)
                    if atten_mask is not None:
                        M = M & (np.asarray(atten_mask)[s0:s1][:, keys] == 0)
                    a, c, e = _head_backward(Qh[s0:s1], Kh[keys], Vh[keys], dOh[s0:s1],
                                             Oh[s0:s1], Lh[s0:s1], M, scale)
                    dQh[s0:s1] = a
                    dKh[keys] += c          # keys are distinct within one block row
                    dVh[keys] += e
                if layout == "BNSD":
                    dq[b, h, :lq[b]] = dQh
                else:
                    dq[oq[b]:oq[b] + lq[b], h] = dQh
            if layout == "BNSD":
                dk[b, g, :lk[b]] = dKh
                dv[b, g, :lk[b]] = dVh
            else:
                dk[okv[b]:okv[b] + lk[b], g] = dKh
                dv[okv[b]:okv[b] + lk[b], g] = dVh
    return dq, dk, dv


def backward_dq_rows(dout, q, k, v, out, lse, b, h, rows, mask=None,
                     block_shape=(128, 128), seq_q=None, seq_kv=None, layout="BNSD",
                     num_kv_heads=None, scale=1.0, pre_tokens=NO_WINDOW,
                     next_tokens=NO_WINDOW, atten_mask=None):
    """dQ[b, h, rows] only (fp64 [len(rows), D]); each row needs only its own
    query, dOut, Out, lse and the keys it selects. Rows at or beyond the actual
    length are 0 (R4)."""
    bx, by = int(block_shape[0]), int(block_shape[1])
    B, lq, lk = _lengths(q, k, layout, seq_q, seq_kv)
    _, N1, N2, D = _dims(q, k, layout)
    g = h // (N1 // N2)
    oq, okv = seq_offsets(lq), seq_offsets(lk)
    rows = np.asarray(rows)
    res = np.zeros((len(rows), D))
    ok = rows < lq[b]
    r = rows[ok]
    if len(r) == 0:
        return res
    Qh = head_rows(q, layout, b, h, lq[b], oq)[r]
    dOh = head_rows(dout, layout, b, h, lq[b], oq)[r]
    Oh = head_rows(out, layout, b, h, lq[b], oq)[r]
    L = _lse_rows(lse, layout, b, h, lq[b], oq)[r]
    Km = head_rows(k, layout, b, g, lk[b], okv)
    Vm = head_rows(v, layout, b, g, lk[b], okv)
    M = token_mask_at(None if mask is None else mask[b, h], bx, by, r, np.arange(lk[b]),
                      pre_tokens, next_tokens, atten_mask)
    dQ, _, _ = _head_backward(Qh, Km, Vm, dOh, Oh, L, M, scale)
    res[ok] = dQ
    return res


def backward_dkdv_rows(dout, q, k, v, out, lse, b, g, rows, mask=None,
                       block_shape=(128, 128), seq_q=None, seq_kv=None, layout="BNSD",
                       num_kv_heads=None, scale=1.0, pre_tokens=NO_WINDOW,
                       next_tokens=NO_WINDOW, atten_mask=None):
    """dK[b, g, rows], dV[b, g, rows] only (fp64), summed over the query heads of
    group g (R3). Each key row needs all query rows that select it."""
    bx, by = int(block_shape[0]), int(block_shape[1])
    B, lq, lk = _lengths(q, k, layout, seq_q, seq_kv)
    _, N1, N2, D = _dims(q, k, layout)
    G = N1 // N2
    oq, okv = seq_offsets(lq), seq_offsets(lk)
    rows = np.asarray(rows)
    dk = np.zeros((len(rows), D))
    dv = np.zeros((len(rows), D))
    ok = rows < lk[b]
    t = rows[ok]
    if len(t) == 0:
        return dk, dv
    Kt = head_rows(k, layout, b, g, lk[b], okv)[t]
    Vt = head_rows(v, layout, b, g, lk[b], okv)[t]
    for h in range(g * G, (g + 1) * G):
        Qm = head_rows(q, layout, b, h, lq[b], oq)
        dOm = head_rows(dout, layout, b, h, lq[b], oq)
        Om = head_rows(out, layout, b, h, lq[b], oq)
        L = _lse_rows(lse, layout, b, h, lq[b], oq)
        M = token_mask_at(None if mask is None else mask[b, h], bx, by, np.arange(lq[b]), t,
                          pre_tokens, next_tokens, atten_mask)
        _, dK, dV = _head_backward(Qm, Kt, Vt, dOm, Om, L, M, scale)
        dk[ok] += dK
        dv[ok] += dV
    return dk, dv


# --------------------------------------------------------------------------
# mask compaction (parameter table, blockSparseMaskOptional; reading R4)
# --------------------------------------------------------------------------
def compact_mask(mask, bx, by, seq_q, seq_kv):
    """Per-(b, h) CSR (query block -> selected key blocks) and CSC (key block ->
    query blocks that select it), ascending, keeping only blocks that start
    inside the actual lengths. Returns int32 arrays
    row_ptr [B*N*(Mq+1)], col_idx [nnz], col_ptr [B*N*(Mk+1)], row_idx [nnz]
    where (b, h) occupies slot b*N + h and each pointer array restarts at the
    running nnz of the previous slots (one global numbering)."""
    mask = np.asarray(mask)
    B, N, Mq, Mk = mask.shape
    row_ptr, col_idx, col_ptr, row_idx = [], [], [], []
    nnz_r = nnz_c = 0
    for b in range(B):
        mq = min(Mq, -(-int(seq_q[b]) // bx))
        mk = min(Mk, -(-int(seq_kv[b]) // by))
        for h in range(N):
            sel = np.asarray(mask[b, h]) != 0
            for i in range(Mq):
                row_ptr.append(nnz_r)
                if i < mq:
                    js = np.nonzero(sel[i, :mk])[0]
                    col_idx.extend(js.tolist())
                    nnz_r += len(js)
            row_ptr.append(nnz_r)
            for j in range(Mk):
                col_ptr.append(nnz_c)
                if j < mk:
                    is_ = np.nonzero(sel[:mq, j])[0]
                    row_idx.extend(is_.tolist())
                    nnz_c += len(is_)
            col_ptr.append(nnz_c)
    return (np.asarray(row_ptr, np.int32), np.asarray(col_idx, np.int32),
            np.asarray(col_ptr, np.int32), np.asarray(row_idx, np.int32))
