"""The run call inside a CUDA graph. bsa_grad is captured once and replayed
twice, in the default and the deterministic dQ mode; the capture includes the
side stream's fork and join. Each replay rewrites every output element (the
outputs are first filled with a wrong value) with the oracle's gradients, and
the deterministic mode gives the same bytes as an eager run."""
import pytest
import torch

import block_sparse_attention_attn_gb300 as bsa
from block_sparse_attention_attn_gb300.workloads import small_workload
from oracle import bsa_oracle as O
from tests.harness import check, f64, host_inputs, oracle_forward, rounded_out_lse

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("det", [False, True], ids=["reduce_add", "deterministic"])
def test_grad_replayed_from_a_cuda_graph(det):
    w = small_workload(B=2, N1=4, N2=2, D=128, bx=128, by=128, seq_q=(300, 257),
                       seq_kv=(384, 129), Sq=384, Skv=384, p=0.5, seed=131)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    g = [t.to(DEV) for t in (dout, q, k, v, tout, tlse)]
    mask = torch.from_numpy(w.mask).to(DEV)
    dq, dk, dv = (torch.empty_like(g[i]) for i in (1, 2, 3))

    def executor():
        size, ex = bsa.bsa_grad_workspace_size(
            *g, mask, None, [w.bx, w.by], list(w.seq_q), list(w.seq_kv), w.layout, w.layout,
            w.N2, 0, w.scale, dq=dq, dk=dk, dv=dv)
        if det:
            ex.set_deterministic(True)
        return size, ex

    size, ex = executor()
    ws = torch.empty(size, dtype=torch.uint8, device=DEV)
    bsa.bsa_grad(ws, size, ex)          # eager: creates the side stream, loads the kernels
    bsa.bsa_check_status(ws)
    eager = [t.clone() for t in (dq, dk, dv)]

    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    _, ex = executor()
    with torch.cuda.stream(s):
        graph.capture_begin()
        bsa.bsa_grad(ws, size, ex, s)
        graph.capture_end()
    torch.cuda.current_stream().wait_stream(s)

    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
    for _ in range(2):
        for t in (dq, dk, dv):
            t.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        bsa.bsa_check_status(ws)
        for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            check(f"graph:{name}", f64(got), r)
        if det:
            for a, b in zip((dq, dk, dv), eager):
                assert torch.equal(a, b)
