"""Deterministic dQ mode and the autograd pairing, on the GPU, against the fp64
oracle (attentionOut / softmaxLse from the oracle's forward, as in the other
parity tests) and against themselves (bitwise repeatability)."""
import numpy as np
import pytest
import torch

import block_sparse_attention_attn_gb300 as bsa
from block_sparse_attention_attn_gb300.workloads import make_workload, small_workload
from oracle import bsa_oracle as O
from tests.harness import (TORCH_DT, check, check_whole, f64, host_inputs,
                           oracle_backward_whole, oracle_forward, rounded_out_lse)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_grad(w, dout, q, k, v, out, lse, deterministic, pad_seq=True):
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    res = bsa.block_sparse_attention_grad(
        dout.to(DEV), q.to(DEV), k.to(DEV), v.to(DEV), out.to(DEV), lse.to(DEV),
        block_sparse_mask=mask, block_shape=[w.bx, w.by], actual_seq_lengths=w.seq_q,
        actual_seq_lengths_kv=w.seq_kv, layout=w.layout, num_key_value_heads=w.N2,
        scale_value=w.scale, deterministic=deterministic)
    bsa.bsa_check_status(res[3])
    return res[:3]


def det_case(w, pad_fill=None):
    dout, q, k, v = host_inputs(w, pad_fill)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse, pad_fill)
    got = run_grad(w, dout, q, k, v, tout, tlse, deterministic=True)
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check(f"{w.name}:det:{name}", f64(g), r)
    return dout, q, k, v, tout, tlse, got


@pytest.mark.parametrize("layout,dtype,B,N1,N2,D,bx,by,sq,skv,p", [
    ("BNSD", "bf16", 2, 4, 2, 128, 128, 128, (300, 170), (300, 250), 0.6),
    ("BNSD", "f16", 1, 4, 1, 64, 64, 64, (320,), (260,), 0.5),
    ("BNSD", "bf16", 1, 2, 1, 128, 64, 128, (256,), (384,), 0.5),
    ("TND", "f16", 3, 4, 2, 128, 128, 64, (200, 333, 64), (250, 129, 300), 0.5),
    ("TND", "bf16", 2, 8, 1, 64, 64, 64, (130, 257), (190, 77), 0.7),
])
def test_deterministic_small_full(layout, dtype, B, N1, N2, D, bx, by, sq, skv, p):
    Sq = max(sq) if layout == "TND" else max(sq) + 17
    Skv = max(skv) if layout == "TND" else max(skv) + 5
    w = small_workload(layout=layout, dtype=dtype, B=B, N1=N1, N2=N2, D=D, bx=bx, by=by,
                       seq_q=sq, seq_kv=skv, Sq=Sq, Skv=Skv, p=p, seed=B * 100 + N1 + D + 7)
    det_case(w)


def test_deterministic_padding_garbage_is_ignored():
    w = small_workload(B=2, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(200, 129),
                       seq_kv=(300, 140), Sq=384, Skv=384, p=0.7, seed=15)
    det_case(w, pad_fill=float("nan"))


def test_deterministic_is_bitwise_repeatable_and_matches_default():
    """Several key tiles per query tile, GQA and tails: two deterministic runs
    give identical bytes; the default (reduce-add) path agrees within the
    tolerance and is not required to be bitwise stable."""
    w = small_workload(B=1, N1=8, N2=2, D=128, bx=128, by=128, seq_q=(1500,), seq_kv=(1400,),
                       p=0.5, seed=23)
    dout, q, k, v, tout, tlse, first = det_case(w)
    second = run_grad(w, dout, q, k, v, tout, tlse, deterministic=True)
    for a, b in zip(first, second):
        assert torch.equal(a, b)
    default = run_grad(w, dout, q, k, v, tout, tlse, deterministic=False)
    for name, a, b in zip(("dq", "dk", "dv"), default, first):
        check(f"det-vs-default:{name}", f64(a), f64(b))


def test_deterministic_large_whole():
    """w2 (GQA 4, S 8192) in the deterministic mode: whole dQ, dK, dV against
    the oracle."""
    w = make_workload("w2")
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, blockrows=True)
    tout, tlse = rounded_out_lse(w, out, lse)
    del out, lse
    got = run_grad(w, dout, q, k, v, tout, tlse, deterministic=True)
    check_whole("w2:det", got, oracle_backward_whole(w, dout, q, k, v, tout, tlse))


@pytest.mark.parametrize("deterministic", [False, True])
def test_autograd_function(deterministic):
    """torch.autograd drives the pair: forward = bsa_fwd, backward = bsa_grad on
    the saved Q, K, V, Out and lse. The forward is checked against the oracle's
    forward, the gradients against the oracle's backward fed with the same
    Out / lse bytes the GPU backward used."""
    w = small_workload(layout="BNSD", dtype="bf16", B=2, N1=4, N2=2, D=128, bx=128, by=64,
                       seq_q=(300, 200), seq_kv=(280, 260), Sq=300, Skv=280, p=0.6, seed=31)
    dout, q, k, v = host_inputs(w)
    mask = torch.from_numpy(w.mask).to(DEV)
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    out = bsa.block_sparse_attention(qd, kd, vd, block_sparse_mask=mask, block_shape=[w.bx, w.by],
                                     actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv,
                                     layout="BNSD", num_key_value_heads=w.N2,
                                     scale_value=w.scale, deterministic=deterministic)
    out.backward(dout.to(DEV))
    ref_out, _ = oracle_forward(w, q, k, v)
    check("autograd:out", f64(out.detach()), ref_out)
    # the backward's own inputs: the same forward once more (deterministic)
    fo, fl, fws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[w.bx, w.by],
        actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv, layout="BNSD",
        num_key_value_heads=w.N2, scale_value=w.scale)
    bsa.bsa_check_status(fws)
    assert torch.equal(fo, out.detach())
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(fo), f64(fl), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), ref):
        assert g.dtype == TORCH_DT[w.dtype]
        check(f"autograd:{name}", f64(g), r)


def test_deterministic_large_token_masked():
    """w1doc's shape and token mask (dense B2 N16 S4096 with causal documents
    as attenMask) in the deterministic mode, in fp16 (see
    test_atten_mask_large_whole): two runs give identical bytes, and the whole
    outputs match the oracle."""
    w = make_workload("w1doc")
    w.dtype = "f16"
    dout, q, k, v = host_inputs(w)
    win = dict(atten_mask=w.atten_mask)
    out, lse = oracle_forward(w, q, k, v, blockrows=True, **win)
    tout, tlse = rounded_out_lse(w, out, lse)
    del out, lse
    am = torch.from_numpy(w.atten_mask).to(DEV)

    def grad():
        res = bsa.block_sparse_attention_grad(
            dout.to(DEV), q.to(DEV), k.to(DEV), v.to(DEV), tout.to(DEV), tlse.to(DEV),
            block_shape=[w.bx, w.by], num_key_value_heads=w.N2, scale_value=w.scale,
            deterministic=True, atten_mask=am)
        bsa.bsa_check_status(res[3])
        return res[:3]
    first, second = grad(), grad()
    for a, b in zip(first, second):
        assert torch.equal(a, b)
    check_whole("w1doc:det", first,
                oracle_backward_whole(w, dout, q, k, v, tout, tlse, mask=None, **win))
