"""GPU parity of the 64-key-block backward (executor option key_block64;
blockShape [bx, 64] with D = 128, no sliding window or token mask):
query-major tiles, one pass per key block of a 128-key tile. Whole output
tensors against the fp64 oracle on the same seeded inputs; the cases reach both query-block sizes, ragged query and key
tails, split columns (fp32 slots), key blocks no query selects, strided
outputs (the per-element store path), NaN in BNSD padding, the deterministic
mode and the bounded-wait failure report."""
import numpy as np
import pytest
import torch

import block_sparse_attention_attn_gb300 as bsa
from block_sparse_attention_attn_gb300.workloads import make_workload, small_workload
from oracle import bsa_oracle as O
from tests.harness import (check, check_whole, f64, host_inputs, oracle_backward_whole,
                           oracle_forward, rounded_out_lse)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_grad(w, dout, q, k, v, out, lse, dq=None, dk=None, dv=None, det=False):
    mask = torch.from_numpy(w.mask).to(DEV)
    seq_q = list(w.seq_q) if w.seq_q is not None else None
    seq_kv = list(w.seq_kv) if w.seq_kv is not None else None
    g = [t.to(DEV) for t in (dout, q, k, v, out, lse)]
    dq = torch.empty_like(g[1]) if dq is None else dq
    dk = torch.empty_like(g[2]) if dk is None else dk
    dv = torch.empty_like(g[3]) if dv is None else dv
    size, ex = bsa.bsa_grad_workspace_size(
        *g, mask, None, [w.bx, w.by], seq_q, seq_kv, w.layout, w.layout,
        w.N2, 0, w.scale, dq=dq, dk=dk, dv=dv)
    ex.set_key_block64(True)
    if det:
        ex.set_deterministic(True)
    ws = torch.empty(size, dtype=torch.uint8, device=DEV)
    bsa.bsa_grad(ws, size, ex)
    bsa.bsa_check_status(ws)
    return dq, dk, dv, ex, ws


def reference(w, dout, q, k, v, tout, tlse):
    return O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                      (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)


def full_case(w, pad_fill=None, det=False):
    dout, q, k, v = host_inputs(w, pad_fill)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse, pad_fill)
    dq, dk, dv, _, _ = run_grad(w, dout, q, k, v, tout, tlse, det=det)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), reference(w, dout, q, k, v, tout, tlse)):
        check(f"{w.name}:{name}", f64(got), r)


@pytest.mark.parametrize("layout,dtype,B,N1,N2,bx,sq,skv,p", [
    ("BNSD", "bf16", 1, 2, 1, 128, (384,), (384,), 0.5),
    ("BNSD", "f16", 2, 4, 2, 64, (200, 333), (257, 129), 0.5),
    ("BNSD", "bf16", 1, 8, 1, 64, (384,), (300,), 0.9),       # long columns: split into slots
    ("TND", "bf16", 2, 4, 4, 128, (513, 130), (700, 64), 0.3),
    ("TND", "f16", 3, 6, 2, 64, (100, 257, 1), (190, 64, 65), 0.6),
])
def test_k64_full(layout, dtype, B, N1, N2, bx, sq, skv, p):
    Sq = max(sq) if layout == "TND" else max(sq) + 17
    Skv = max(skv) if layout == "TND" else max(skv) + 5
    w = small_workload(layout=layout, dtype=dtype, B=B, N1=N1, N2=N2, D=128, bx=bx, by=64,
                       seq_q=sq, seq_kv=skv, Sq=Sq, Skv=Skv, p=p, seed=B * 31 + N1 + bx)
    full_case(w)


def test_k64_unselected_blocks_and_padding():
    """Key blocks that no query selects (the pass is empty: its rows come out
    zero), a query block with no key, and NaN in the BNSD padding rows."""
    w = small_workload(B=2, N1=2, N2=1, D=128, bx=128, by=64, seq_q=(300, 129),
                       seq_kv=(330, 200), Sq=384, Skv=384, p=0.7, seed=53)
    w.mask[:, :, :, 1] = 0      # block 1: second half of key tile 0
    w.mask[:, :, :, 2] = 0      # block 2: first half of key tile 1
    w.mask[0, 0, 1, :] = 0      # a query block without keys
    full_case(w, pad_fill=float("nan"))


def test_k64_deterministic():
    w = small_workload(B=1, N1=4, N2=2, D=128, bx=64, by=64, seq_q=(320,), seq_kv=(270,),
                       p=0.6, seed=59)
    full_case(w, det=True)


def test_k64_strided_outputs():
    """dK stored transposed (column stride != 1) and dV with padded rows take
    the per-element store path; nothing outside the views is written."""
    w = small_workload(B=1, N1=2, N2=2, D=128, bx=128, by=64, seq_q=(256,), seq_kv=(256,),
                       p=0.6, seed=61)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    dkt = torch.zeros(1, 2, 128, 256, dtype=torch.bfloat16, device=DEV).transpose(2, 3)
    big = torch.zeros(1, 2, 256, 136, dtype=torch.bfloat16, device=DEV)
    dv = big[..., 4:132]                              # row stride 136, 8-byte aligned rows
    dq, dk, dv, _, _ = run_grad(w, dout, q, k, v, tout, tlse, dk=dkt, dv=dv)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), reference(w, dout, q, k, v, tout, tlse)):
        check(name, f64(got), r)
    assert torch.all(big[..., :4] == 0) and torch.all(big[..., 132:] == 0)


def test_k64_bounded_wait_reports_error():
    """The deliberate never-completed wait of the test switch runs out in this
    kernel too; the host reads 561002 and the next run is correct."""
    w = small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=64, seq_q=(256,), seq_kv=(256,),
                       p=1.0, seed=67)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    g = [t.to(DEV) for t in (dout, q, k, v, tout, tlse)]
    mask = torch.from_numpy(w.mask).to(DEV)
    dq, dk, dv = (torch.empty_like(g[i]) for i in (1, 2, 3))
    size, ex = bsa.bsa_grad_workspace_size(*g, mask, None, [128, 64], None, None, "BNSD", "BNSD",
                                           1, 0, w.scale, dq=dq, dk=dk, dv=dv)
    ex.set_key_block64(True)
    ex.set_wait_test(True)
    ws = torch.empty(size, dtype=torch.uint8, device=DEV)
    bsa.bsa_grad(ws, size, ex)
    with pytest.raises(bsa.BsaError) as err:
        bsa.bsa_check_status(ws)
    assert err.value.status == 561002
    hdr = ws[:128].view(torch.int32).cpu().tolist()
    assert hdr[6] == 12 or hdr[16 + 12] > 0
    full_case(w)


def test_k64_w3_whole():
    """The full-size 128x64 workload (TND fp16, 8 sequences, GQA 4): every
    element of dQ, dK and dV against the oracle's block-row evaluation."""
    w = make_workload("w3")
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, blockrows=True)
    tout, tlse = rounded_out_lse(w, out, lse)
    del out, lse
    dq, dk, dv, _, _ = run_grad(w, dout, q, k, v, tout, tlse)
    check_whole("w3:k64", (dq, dk, dv), oracle_backward_whole(w, dout, q, k, v, tout, tlse))
