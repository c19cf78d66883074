"""Sliding window (preTokens / nextTokens; nextTokens = 0 is the causal mask)
on the GPU against the fp64 oracle: backward (default and deterministic dQ),
the companion forward, the autograd pairing, and the whole outputs of a full-size
workload. attentionOut / softmaxLse come from the oracle's forward with the
same window."""
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
NOW = O.NO_WINDOW


def run_grad(w, dout, q, k, v, out, lse, pre, nxt, deterministic=False):
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    res = bsa.block_sparse_attention_grad(
        dout.to(DEV), q.to(DEV), k.to(DEV), v.to(DEV), out.to(DEV), lse.to(DEV),
        block_sparse_mask=mask, block_shape=[w.bx, w.by], actual_seq_lengths=w.seq_q,
        actual_seq_lengths_kv=w.seq_kv, layout=w.layout, num_key_value_heads=w.N2,
        scale_value=w.scale, deterministic=deterministic, pre_tokens=pre, next_tokens=nxt)
    bsa.bsa_check_status(res[3])
    return res[:3]


def run_fwd(w, q, k, v, pre, nxt):
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    out, lse, ws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[w.bx, w.by],
        actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv, layout=w.layout,
        num_key_value_heads=w.N2, scale_value=w.scale, pre_tokens=pre, next_tokens=nxt)
    bsa.bsa_check_status(ws)
    return out, lse


def window_case(w, pre, nxt, deterministic=False):
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, pre_tokens=pre, next_tokens=nxt)
    tout, tlse = rounded_out_lse(w, out, lse)
    got = run_grad(w, dout, q, k, v, tout, tlse, pre, nxt, deterministic)
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale,
                     pre_tokens=pre, next_tokens=nxt)
    tag = f"{w.name}:pre{pre}:next{nxt}:{'det' if deterministic else 'red'}"
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check(f"{tag}:{name}", f64(g), r)
    return (dout, q, k, v), (out, lse), got


# layout, dtype, B, N1, N2, D, bx, by, seq_q, seq_kv, block density, pre, next, dense
CASES = [
    ("BNSD", "bf16", 2, 4, 2, 128, 128, 128, (300, 517), (300, 517), 1.0, NOW, 0, True),
    ("BNSD", "f16", 1, 4, 1, 64, 64, 64, (600,), (450,), 0.7, NOW, 0, False),
    ("BNSD", "bf16", 1, 4, 2, 128, 128, 64, (700,), (900,), 0.8, 200, 37, False),
    ("TND", "f16", 3, 4, 2, 128, 64, 128, (300, 129, 513), (260, 400, 513), 0.8, 150, 0, False),
    ("BNSD", "bf16", 1, 2, 1, 128, 128, 128, (400,), (400,), 1.0, 100, -20, True),
    ("BNSD", "bf16", 1, 2, 1, 64, 64, 64, (350,), (380,), 1.0, -30, 200, True),
    ("TND", "bf16", 2, 8, 1, 64, 64, 64, (130, 257), (190, 77), 0.9, 5, 5, False),
]


def _workload(case, seed):
    layout, dtype, B, N1, N2, D, bx, by, sq, skv, p, pre, nxt, dense = case
    Sq = max(sq) if layout == "TND" else max(sq) + 11
    Skv = max(skv) if layout == "TND" else max(skv) + 7
    w = small_workload(layout=layout, dtype=dtype, B=B, N1=N1, N2=N2, D=D, bx=bx, by=by,
                       seq_q=sq, seq_kv=skv, Sq=Sq, Skv=Skv, p=p, seed=seed, dense=dense)
    return w, pre, nxt


@pytest.mark.parametrize("i", range(len(CASES)))
def test_window_backward(i):
    w, pre, nxt = _workload(CASES[i], 500 + i)
    window_case(w, pre, nxt)


@pytest.mark.parametrize("i", [0, 3, 4])
def test_window_backward_deterministic(i):
    w, pre, nxt = _workload(CASES[i], 600 + i)
    window_case(w, pre, nxt, deterministic=True)


def test_keyless_rows_and_unreached_keys():
    """nextTokens < 0 leaves the first rows without keys (dQ rows 0) and
    preTokens < 0 leaves the first keys unreached by any row (dK, dV rows 0)."""
    w, pre, nxt = _workload(CASES[4], 700)
    _, (out, lse), got = window_case(w, pre, nxt)
    assert np.all(np.isneginf(lse[0, :, :20, 0])) and np.all(out[0, :, :20] == 0)
    assert torch.all(got[0][0, :, :20] == 0)
    w, pre, nxt = _workload(CASES[5], 701)
    _, _, got = window_case(w, pre, nxt)
    # preTokens = -30: query s reaches keys t >= s + 30 only, so keys 0..29 get nothing
    assert torch.all(got[1][0, :, :30] == 0) and torch.all(got[2][0, :, :30] == 0)
    assert torch.any(got[1][0, :, 30:34] != 0)


@pytest.mark.parametrize("i", [0, 1, 3, 6])
def test_window_forward(i):
    w, pre, nxt = _workload(CASES[i], 800 + i)
    dout, q, k, v = host_inputs(w)
    ref_out, ref_lse = oracle_forward(w, q, k, v, pre_tokens=pre, next_tokens=nxt)
    out, lse = run_fwd(w, q, k, v, pre, nxt)
    check(f"fwd:{i}:out", f64(out), ref_out)
    got_lse = f64(lse)
    fin = np.isfinite(ref_lse)
    np.testing.assert_array_equal(np.isneginf(got_lse), ~fin)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)


def test_no_window_values_agree_with_the_plain_path():
    """A window reaching every pair (and the 2147483647 default) computes the
    same gradients as the call without window arguments."""
    w, _, _ = _workload(CASES[2], 900)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    a = run_grad(w, dout, q, k, v, tout, tlse, NOW, NOW, deterministic=True)
    b = run_grad(w, dout, q, k, v, tout, tlse, max(w.seq_q) - 1, max(w.seq_kv) - 1,
                 deterministic=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_causal_autograd():
    w = small_workload(layout="BNSD", dtype="bf16", B=2, N1=4, N2=2, D=128, bx=128, by=128,
                       seq_q=(384, 300), seq_kv=(384, 350), Sq=384, Skv=384, p=0.8, seed=910)
    dout, q, k, v = host_inputs(w)
    mask = torch.from_numpy(w.mask).to(DEV)
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    out = bsa.block_sparse_attention(qd, kd, vd, block_sparse_mask=mask, block_shape=[128, 128],
                                     actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv,
                                     num_key_value_heads=w.N2, scale_value=w.scale, next_tokens=0)
    out.backward(dout.to(DEV))
    ref_out, _ = oracle_forward(w, q, k, v, next_tokens=0)
    check("causal-autograd:out", f64(out.detach()), ref_out)
    fo, fl = run_fwd(w, q, k, v, NOW, 0)
    assert torch.equal(fo, out.detach())
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(fo), f64(fl), w.mask, (128, 128),
                     w.seq_q, w.seq_kv, "BNSD", w.N2, w.scale, next_tokens=0)
    for name, g, r in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), ref):
        check(f"causal-autograd:{name}", f64(g), r)


@pytest.mark.parametrize("name,pre,nxt", [("w1", NOW, 0), ("w3", 1000, 0)])
def test_window_large_whole(name, pre, nxt):
    """Full-size workloads (w1: BNSD B2 N16 S4096, causal; w3: TND 8 sequences,
    sliding window of 1000 earlier tokens): whole dQ, dK, dV against the
    oracle, plus the forward on the full tensors."""
    w = make_workload(name)
    win = dict(pre_tokens=pre, next_tokens=nxt)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, blockrows=True, **win)
    tout, tlse = rounded_out_lse(w, out, lse)
    del out, lse
    got = run_grad(w, dout, q, k, v, tout, tlse, pre, nxt)
    check_whole(f"{name}:win", got, oracle_backward_whole(w, dout, q, k, v, tout, tlse, **win))
    fo, fl = run_fwd(w, q, k, v, pre, nxt)
    check(f"{name}:win:fwd_out", f64(fo), f64(tout))
    fin = np.isfinite(f64(tlse))
    np.testing.assert_array_equal(np.isneginf(f64(fl)), ~fin)
    np.testing.assert_allclose(f64(fl)[fin], f64(tlse)[fin], rtol=1e-4, atol=2e-3)


def test_diagonal_only_window_closed_form():
    """preTokens = nextTokens = 0: each query sees only the key at its own
    position, so P = 1, dQ = dK = 0 and dV = dOut (up to rounding), on a
    multi-tile BNSD case with a ragged tail, against the closed form and the
    oracle."""
    w = small_workload(layout="BNSD", dtype="bf16", B=1, N1=2, N2=2, D=128, bx=128, by=128,
                       seq_q=(300,), seq_kv=(300,), p=1.0, seed=1700, dense=True)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, pre_tokens=0, next_tokens=0)
    tout, tlse = rounded_out_lse(w, out, lse)
    dq, dk, dv = run_grad(w, dout, q, k, v, tout, tlse, 0, 0)
    assert float(dq.abs().max()) < 1e-2 and float(dk.abs().max()) < 1e-2
    check("diag:dv-vs-dout", f64(dv)[0, :, :300], f64(dout)[0, :, :300])
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), None,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale,
                     pre_tokens=0, next_tokens=0)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        check(f"diag:{name}", f64(g), r)
