"""Seeded synthetic workloads for the block-sparse attention backward.

This module only draws random numbers and builds block masks: it holds none of
the attention arithmetic, so both the fp64 oracle (tests, CPU baseline) and the
CUDA path (tests, bench) can take their inputs from it without sharing any
compute code.

The five shapes follow the workloads of the ``aclnnBlockSparseAttentionGrad``
documentation page (section "参数说明": BNSD/TND layouts, blockShape, GQA via
numKeyValueHeads, per-batch actualSeqLengths), sized as the large-scale cases
this library is measured on:

====  ==========================================================================
name  shape / mask
====  ==========================================================================
w0    BNSD bf16 B1 N2 Nkv2 S256 D64, 64x64 blocks, Bernoulli(0.5) + diagonal
w1    BNSD bf16 B2 N16 Nkv16 S4096 D128, 128x128, Bernoulli(0.25) + diagonal
      (``w1dense``: same shape, mask = None)
w2    BNSD bf16 GQA B1 N32 Nkv8 S8192 D128, 128x128, block-causal window of 4
      blocks + KV blocks 0-1 + Bernoulli(0.1) below the window
w3    TND fp16 8 seqs, L ~ U[512, 8192], N16 Nkv4 D128, 128x64 blocks,
      Bernoulli(0.3) in the valid range + the diagonal block pairs
w4    BNSD bf16 B1 N8 Nkv8 S65536 D128, 128x128, top-k style rows: the
      diagonal, block 0 and 14 uniform picks from the earlier blocks
====  ==========================================================================

With a sliding window (preTokens / nextTokens): ``w2causal`` is w2 with
nextTokens = 0 (token-level causal inside the diagonal blocks), ``w1causal``
is w1dense with nextTokens = 0 (dense causal attention). With a token mask
(attenMask, 1 = masked): ``w1doc`` is w1dense with causal documents of
200-1500 tokens (a pair is masked across documents and above the diagonal:
packed-document training).

Values are N(0, 1) (w3: standard deviation 0.5), drawn from numpy's PCG64 and
rounded to the input dtype with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = ["Workload", "WORKLOADS", "make_workload", "normal", "random_mask",
           "ceil_div", "NO_WINDOW", "window_pairs", "document_mask"]

NO_WINDOW = 2147483647   # preTokens / nextTokens value of "no sliding window"


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) samples (PCG64 stream of ``rng``)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


@dataclasses.dataclass
class Workload:
    name: str
    layout: str                 # "BNSD" or "TND"
    dtype: str                  # "bf16" or "f16"
    B: int
    N1: int
    N2: int
    D: int
    bx: int
    by: int
    seq_q: list                 # per-batch valid query tokens
    seq_kv: list                # per-batch valid key/value tokens
    Sq: int                     # padded (BNSD) / max (TND) query length
    Skv: int
    scale: float
    mask: Optional[np.ndarray]  # uint8 [B, N1, ceil(Sq/bx), ceil(Skv/by)] or None
    std: float = 1.0
    seed: int = 0
    pre_tokens: int = NO_WINDOW     # sliding window: query s sees keys
    next_tokens: int = NO_WINDOW    # s - pre_tokens .. s + next_tokens
    atten_mask: Optional[np.ndarray] = None   # uint8 [Sq, Skv], 1 = masked (maskType 1)
    atten_mask_desc: str = ""

    def windowed(self) -> bool:
        return not (self.pre_tokens >= self.Sq - 1 and self.next_tokens >= self.Skv - 1)

    def token_masked(self) -> bool:
        return self.windowed() or self.atten_mask is not None

    def window_kw(self) -> dict:
        return dict(pre_tokens=self.pre_tokens, next_tokens=self.next_tokens)

    @property
    def Mq(self) -> int:
        return ceil_div(self.Sq, self.bx)

    @property
    def Mk(self) -> int:
        return ceil_div(self.Skv, self.by)

    def q_shape(self):
        if self.layout == "BNSD":
            return (self.B, self.N1, self.Sq, self.D)
        return (int(sum(self.seq_q)), self.N1, self.D)

    def kv_shape(self):
        if self.layout == "BNSD":
            return (self.B, self.N2, self.Skv, self.D)
        return (int(sum(self.seq_kv)), self.N2, self.D)

    def lse_shape(self):
        if self.layout == "BNSD":
            return (self.B, self.N1, self.Sq, 1)
        return (int(sum(self.seq_q)), self.N1, 1)

    def _selected_per_block(self, b):
        """[mq, mk] number of query heads selecting each block of batch b."""
        mq = ceil_div(self.seq_q[b], self.bx)
        mk = ceil_div(self.seq_kv[b], self.by)
        if self.mask is None:
            return np.full((mq, mk), self.N1, dtype=np.int64)
        return np.count_nonzero(self.mask[b, :, :mq, :mk], axis=0).astype(np.int64)

    def active_blocks(self) -> int:
        """Active blocks inside the valid range (and meeting the window),
        summed over batch and q-heads."""
        n = 0
        for b in range(self.B):
            sel = self._selected_per_block(b)
            if self.token_masked():
                sel = sel * (window_pairs(self.seq_q[b], self.seq_kv[b], self.bx, self.by,
                                          self.pre_tokens, self.next_tokens,
                                          self.atten_mask) > 0)
            n += int(sel.sum())
        return n

    def flops(self) -> float:
        """Algorithmic backward FLOPs: 10*D per (query, key) pair that takes
        part, per q-head (5 products of 2*D each: S, dP, dV, dQ, dK). Without a
        window or token mask a selected block counts as bx*by pairs (tail
        blocks included); with one only the pairs they keep inside the lengths
        count."""
        if not self.token_masked():
            return 10.0 * self.bx * self.by * self.D * self.active_blocks()
        pairs = 0
        for b in range(self.B):
            wp = window_pairs(self.seq_q[b], self.seq_kv[b], self.bx, self.by,
                              self.pre_tokens, self.next_tokens, self.atten_mask)
            pairs += int((self._selected_per_block(b) * wp).sum())
        return 10.0 * self.D * pairs

    def tensors(self, seed: Optional[int] = None):
        """(dout, q, k, v) as float32 numpy arrays of the layout's shapes.

        Values are exactly representable in the workload dtype only after the
        caller rounds them (``torch.tensor(x).to(dtype)``); the bench and the
        tests both do that and hand the same rounded bytes to both sides.
        """
        rng = np.random.Generator(np.random.PCG64(self.seed if seed is None else seed))
        q = normal(rng, self.q_shape(), self.std)
        k = normal(rng, self.kv_shape(), self.std)
        v = normal(rng, self.kv_shape(), self.std)
        dout = normal(rng, self.q_shape(), self.std)
        return dout, q, k, v


def window_pairs(lq, lk, bx, by, pre, nxt, atten_mask=None):
    """[ceil(lq/bx), ceil(lk/by)] int64: per block, the (s, t) pairs with s < lq,
    t < lk, s - pre <= t <= s + nxt and (with a token mask) atten_mask[s, t] == 0
    (geometry for FLOP counting)."""
    mq, mk = ceil_div(lq, bx), ceil_div(lk, by)
    if atten_mask is not None:
        s = np.arange(lq, dtype=np.int64)[:, None]
        t = np.arange(lk, dtype=np.int64)[None, :]
        keep = (t >= s - min(int(pre), 1 << 40)) & (t <= s + min(int(nxt), 1 << 40))
        keep &= np.asarray(atten_mask)[:lq, :lk] == 0
        keep = np.pad(keep, ((0, mq * bx - lq), (0, mk * by - lk)))
        return keep.reshape(mq, bx, mk, by).sum(axis=(1, 3)).astype(np.int64)
    s = np.arange(lq, dtype=np.int64)[:, None]
    t0 = (np.arange(mk, dtype=np.int64) * by)[None, :]
    t1 = np.minimum(t0 + by, lk) - 1
    lo = np.maximum(t0, s - min(int(pre), 1 << 40))
    hi = np.minimum(t1, s + min(int(nxt), 1 << 40))
    per_row = np.maximum(hi - lo + 1, 0)                       # [lq, mk]
    pad = mq * bx - lq
    per_row = np.concatenate([per_row, np.zeros((pad, mk), np.int64)])
    return per_row.reshape(mq, bx, mk).sum(axis=1)


def document_mask(S, Skv, seed, lo=40, hi=300, causal=True):
    """uint8 [S, Skv] token mask (1 = masked) of documents with lengths drawn
    uniformly from [lo, hi): a pair is masked when query and key lie in
    different documents and, with ``causal``, when the key comes later."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = max(S, Skv)
    cuts = np.cumsum(rng.integers(lo, hi, size=n // lo + 2))
    doc = np.searchsorted(cuts, np.arange(n), side="right")
    am = doc[:S, None] != doc[None, :Skv]
    if causal:
        am |= np.arange(Skv)[None, :] > np.arange(S)[:, None]
    return am.astype(np.uint8)


def random_mask(rng, B, N, Mq, Mk, p, diag=True):
    m = (rng.random((B, N, Mq, Mk)) < p).astype(np.uint8)
    if diag:
        for i in range(min(Mq, Mk)):
            m[:, :, i, i] = 1
    return m


def _w0():
    rng = np.random.Generator(np.random.PCG64(1000))
    B, N, S, bx = 1, 2, 256, 64
    m = random_mask(rng, B, N, S // bx, S // bx, 0.5)
    return Workload("w0", "BNSD", "bf16", B, N, N, 64, bx, bx, [S] * B, [S] * B,
                    S, S, 1.0 / 8.0, m, seed=2000)


def _w1(dense=False):
    rng = np.random.Generator(np.random.PCG64(1001))
    B, N, S, D, bl = 2, 16, 4096, 128, 128
    m = None if dense else random_mask(rng, B, N, S // bl, S // bl, 0.25)
    return Workload("w1dense" if dense else "w1", "BNSD", "bf16", B, N, N, D, bl, bl,
                    [S] * B, [S] * B, S, S, D ** -0.5, m, seed=2001)


def _w2():
    rng = np.random.Generator(np.random.PCG64(1002))
    B, N1, N2, S, D, bl = 1, 32, 8, 8192, 128, 128
    M = S // bl
    m = np.zeros((B, N1, M, M), np.uint8)
    for b in range(B):
        for h in range(N1):
            r = rng.random((M, M))
            for i in range(M):
                lo = max(0, i - 3)
                m[b, h, i, lo:i + 1] = 1          # local window of 4 blocks
                m[b, h, i, :min(2, M)] = 1         # KV blocks 0-1 always on
                for j in range(2, lo):              # below the window
                    if r[i, j] < 0.1:
                        m[b, h, i, j] = 1
    return Workload("w2", "BNSD", "bf16", B, N1, N2, D, bl, bl, [S] * B, [S] * B,
                    S, S, D ** -0.5, m, seed=2002)


def _w3():
    rng = np.random.Generator(np.random.PCG64(1003))
    B, N1, N2, D, bx, by = 8, 16, 4, 128, 128, 64
    lens = [int(x) for x in rng.integers(512, 8192, size=B, endpoint=True)]
    S = max(lens)
    Mq, Mk = ceil_div(S, bx), ceil_div(S, by)
    m = np.zeros((B, N1, Mq, Mk), np.uint8)
    for b in range(B):
        mq, mk = ceil_div(lens[b], bx), ceil_div(lens[b], by)
        sub = (rng.random((N1, mq, mk)) < 0.3).astype(np.uint8)
        for i in range(mq):
            for j in (2 * i, 2 * i + 1):
                if j < mk:
                    sub[:, i, j] = 1
        m[b, :, :mq, :mk] = sub
    return Workload("w3", "TND", "f16", B, N1, N2, D, bx, by, lens, list(lens), S, S,
                    D ** -0.5, m, std=0.5, seed=2003)


def _w4():
    rng = np.random.Generator(np.random.PCG64(1004))
    B, N, S, D, bl, picks = 1, 8, 65536, 128, 128, 14
    M = S // bl
    m = np.zeros((B, N, M, M), np.uint8)
    for b in range(B):
        for h in range(N):
            for i in range(M):
                m[b, h, i, i] = 1
                m[b, h, i, 0] = 1
                if i - 1 <= picks:
                    m[b, h, i, 1:i] = 1
                else:
                    sel = rng.choice(np.arange(1, i), size=picks, replace=False)
                    m[b, h, i, sel] = 1
    return Workload("w4", "BNSD", "bf16", B, N, N, D, bl, bl, [S] * B, [S] * B, S, S,
                    D ** -0.5, m, seed=2004)


def _documents(w, name):
    w.name = name
    w.atten_mask = document_mask(w.Sq, w.Skv, 1601, lo=200, hi=1500)
    w.atten_mask_desc = "causal documents of U[200,1500) tokens (seed 1601), 1 = masked"
    return w


def _causal(w, name):
    w.name = name
    w.next_tokens = 0
    return w


WORKLOADS = {
    "w0": _w0,
    "w1": _w1,
    "w1dense": lambda: _w1(dense=True),
    "w2": _w2,
    "w3": _w3,
    "w4": _w4,
    "w2causal": lambda: _causal(_w2(), "w2causal"),
    "w1causal": lambda: _causal(_w1(dense=True), "w1causal"),
    "w1doc": lambda: _documents(_w1(dense=True), "w1doc"),
}


def make_workload(name: str) -> Workload:
    return WORKLOADS[name]()


def small_workload(layout="BNSD", dtype="bf16", B=1, N1=2, N2=1, D=64, bx=64, by=64,
                   seq_q=(200,), seq_kv=(200,), Sq=None, Skv=None, p=0.5, seed=7,
                   scale=None, dense=False, std=1.0, name="small", pre_tokens=NO_WINDOW,
                   next_tokens=NO_WINDOW) -> Workload:
    """A small seeded case for parity tests (ragged tails, GQA, both layouts)."""
    seq_q, seq_kv = list(seq_q), list(seq_kv)
    assert len(seq_q) == B and len(seq_kv) == B
    Sq = Sq if Sq is not None else max(seq_q)
    Skv = Skv if Skv is not None else max(seq_kv)
    rng = np.random.Generator(np.random.PCG64(seed))
    Mq, Mk = ceil_div(Sq, bx), ceil_div(Skv, by)
    m = None if dense else random_mask(rng, B, N1, Mq, Mk, p)
    return Workload(name, layout, dtype, B, N1, N2, D, bx, by, seq_q, seq_kv, Sq, Skv,
                    D ** -0.5 if scale is None else scale, m, std=std, seed=seed + 1,
                    pre_tokens=pre_tokens, next_tokens=next_tokens)


def workload_summary(w: Workload) -> dict:
    return {"workload": w.name, "layout": w.layout, "dtype": w.dtype, "B": w.B,
            "N1": w.N1, "N2": w.N2, "Sq": w.Sq, "Skv": w.Skv, "D": w.D,
            "block": [w.bx, w.by], "active_blocks": w.active_blocks(),
            "density": (w.active_blocks() / float(sum(ceil_div(a, w.bx) * ceil_div(c, w.by)
                                                      for a, c in zip(w.seq_q, w.seq_kv)) * w.N1)),
            "scale": w.scale}


if __name__ == "__main__":  # pragma: no cover - manual inspection
    for k in WORKLOADS:
        w = make_workload(k)
        print(k, workload_summary(w), "GFLOP=%.1f" % (w.flops() / 1e9))
        del w
