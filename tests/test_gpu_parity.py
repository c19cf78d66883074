"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs. attentionOut and softmaxLse always come from the oracle's
forward (never from the CUDA path). Every case compares whole output
tensors: small cases (several tiles and a ragged tail) against the dense
oracle, the full-size workloads against its block-row evaluation."""
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


def run_grad(w, dout, q, k, v, out, lse, dq=None, dk=None, dv=None, seq=True):
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    use_seq = seq or w.layout == "TND"
    res = bsa.block_sparse_attention_grad(
        dout.to(DEV), q.to(DEV), k.to(DEV), v.to(DEV), out.to(DEV), lse.to(DEV),
        block_sparse_mask=mask, block_shape=[w.bx, w.by],
        actual_seq_lengths=w.seq_q if use_seq else None,
        actual_seq_lengths_kv=w.seq_kv if use_seq else None, layout=w.layout,
        num_key_value_heads=w.N2, scale_value=w.scale, dq=dq, dk=dk, dv=dv)
    bsa.bsa_check_status(res[3])
    return res[:3]


def full_case(w, pad_fill=None, seq=True):
    dout, q, k, v = host_inputs(w, pad_fill)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse, pad_fill)
    dq, dk, dv = run_grad(w, dout, q, k, v, tout, tlse, seq=seq)
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        check(f"{w.name}:{name}", f64(got), r)


# ----------------------------------------------------------- full-tensor cases
def test_w0_full():
    full_case(make_workload("w0"))


@pytest.mark.parametrize("layout,dtype,B,N1,N2,D,bx,by,sq,skv,p", [
    ("BNSD", "bf16", 1, 2, 2, 128, 128, 128, (384,), (384,), 0.5),
    ("BNSD", "bf16", 2, 4, 2, 128, 128, 128, (300, 170), (300, 250), 0.6),
    ("BNSD", "f16", 1, 4, 1, 64, 64, 64, (320,), (260,), 0.5),
    ("BNSD", "bf16", 1, 2, 1, 128, 64, 128, (256,), (384,), 0.5),
    ("BNSD", "bf16", 1, 2, 2, 64, 128, 64, (384,), (200,), 0.5),
    ("TND", "f16", 3, 4, 2, 128, 128, 64, (200, 333, 64), (250, 129, 300), 0.5),
    ("TND", "bf16", 2, 8, 1, 64, 64, 64, (130, 257), (190, 77), 0.7),
])
def test_small_full(layout, dtype, B, N1, N2, D, bx, by, sq, skv, p):
    Sq = max(sq) if layout == "TND" else max(sq) + 17
    Skv = max(skv) if layout == "TND" else max(skv) + 5
    w = small_workload(layout=layout, dtype=dtype, B=B, N1=N1, N2=N2, D=D, bx=bx, by=by,
                       seq_q=sq, seq_kv=skv, Sq=Sq, Skv=Skv, p=p, seed=B * 100 + N1 + D)
    full_case(w)


def test_padding_garbage_is_ignored():
    """BNSD padding rows filled with NaN must not leak into the results."""
    w = small_workload(B=2, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(200, 129),
                       seq_kv=(300, 140), Sq=384, Skv=384, p=0.7, seed=5)
    full_case(w, pad_fill=float("nan"))


def test_dense_mask_none_equals_all_ones():
    w = small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(320,), seq_kv=(290,),
                       p=1.0, seed=9, dense=True)
    full_case(w)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    a = run_grad(w, dout, q, k, v, tout, tlse)
    w.mask = np.ones((1, 2, 3, 3), np.uint8)
    b = run_grad(w, dout, q, k, v, tout, tlse)
    for x, y in zip(a, b):   # same arithmetic, fp32 atomics may reorder: tolerance only
        check("dense-vs-ones", f64(x), f64(y))


def test_empty_rows_and_columns():
    w = small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(512,), seq_kv=(512,),
                       p=0.5, seed=11)
    w.mask[0, 0, 1, :] = 0      # query tile without keys
    w.mask[0, :, :, 2] = 0      # key tile nobody selects
    w.mask[0, 1, :, :] = 0      # head without any block
    full_case(w)


def test_strided_outputs():
    w = small_workload(B=1, N1=2, N2=2, D=128, bx=128, by=128, seq_q=(256,), seq_kv=(256,),
                       p=0.6, seed=13)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    big = torch.zeros(1, 2, 256, 256, dtype=torch.bfloat16, device=DEV)
    dq = big[..., 64:192]                             # row stride 256
    dkt = torch.zeros(1, 2, 128, 256, dtype=torch.bfloat16, device=DEV).transpose(2, 3)
    dv = torch.zeros(1, 2, 256, 128, dtype=torch.bfloat16, device=DEV)
    got = run_grad(w, dout, q, k, v, tout, tlse, dq=dq, dk=dkt, dv=dv)
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check(name, f64(g), r)
    assert torch.all(big[..., :64] == 0) and torch.all(big[..., 192:] == 0)


def test_guard_regions_untouched():
    """Outputs are views into larger buffers whose margins hold a canary."""
    w = small_workload(B=1, N1=2, N2=1, D=64, bx=64, by=64, seq_q=(65,), seq_kv=(127,),
                       Sq=65, Skv=127, p=1.0, seed=17)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    canary = -12345.0
    bufs, views = [], []
    for shape in ((1, 2, 65, 64), (1, 1, 127, 64), (1, 1, 127, 64)):
        n = int(np.prod(shape))
        b = torch.full((n + 2048,), canary, dtype=torch.bfloat16, device=DEV)
        bufs.append(b)
        views.append(b[1024:1024 + n].view(shape))
    got = run_grad(w, dout, q, k, v, tout, tlse, *views)
    for b in bufs:
        assert torch.all(b[:1024] == canary) and torch.all(b[-1024:] == canary)
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check(name, f64(g), r)


def test_single_token_sequences():
    w = small_workload(layout="TND", dtype="bf16", B=3, N1=2, N2=1, D=128, bx=128, by=128,
                       seq_q=(1, 129, 1), seq_kv=(1, 1, 200), p=1.0, seed=19)
    full_case(w)


def test_page_call_example():
    """The page's call example (fp16, S = 128, D = 128, 64x64 blocks): dQ = dK = 0
    and every dV element equals 128 * exp(scale*128*q^2 - 5) * dout."""
    S, D = 128, 128
    x = torch.full((1, 1, S, D), 0.1, dtype=torch.float16)
    dout = torch.full((1, 1, S, D), 0.01, dtype=torch.float16)
    lse = torch.full((1, 1, S), 5.0, dtype=torch.float32)
    mask = torch.ones((1, 1, 2, 2), dtype=torch.uint8)
    dq, dk, dv, ws = bsa.block_sparse_attention_grad(
        dout.to(DEV), x.to(DEV), x.to(DEV), x.to(DEV), x.to(DEV), lse.to(DEV),
        block_sparse_mask=mask.to(DEV), block_shape=[64, 64], actual_seq_lengths=[S],
        actual_seq_lengths_kv=[S], layout="BNSD", num_key_value_heads=1,
        scale_value=1.0 / np.sqrt(D))
    bsa.bsa_check_status(ws)
    xv, dv_ = float(x[0, 0, 0, 0]), float(dout[0, 0, 0, 0])
    expect = S * np.exp(D * xv * xv / np.sqrt(D) - 5.0) * dv_
    assert torch.all(dq == 0) and torch.all(dk == 0)
    check("dv", f64(dv), np.full((1, 1, S, D), expect))


# ------------------------------------------------------- large workloads
@pytest.mark.parametrize("name", ["w1", "w1dense", "w2", "w3", "w4"])
def test_large_workload_whole(name):
    """The full-size workloads in the launch configuration the bench times:
    every element of dQ, dK and dV against the oracle (per-element bound and
    relative Frobenius error over the whole tensors), plus the companion
    forward on the full tensors."""
    w = make_workload(name)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, blockrows=True)
    tout, tlse = rounded_out_lse(w, out, lse)
    del out, lse
    got = run_grad(w, dout, q, k, v, tout, tlse)
    check_whole(name, got, oracle_backward_whole(w, dout, q, k, v, tout, tlse))
    # the companion forward on the full workload (many query tiles per CTA)
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    fo, fl, fws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[w.bx, w.by],
        actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv, layout=w.layout,
        num_key_value_heads=w.N2, scale_value=w.scale)
    bsa.bsa_check_status(fws)
    check(f"{name}:fwd_out", f64(fo), f64(tout))
    np.testing.assert_allclose(f64(fl), f64(tlse), rtol=1e-4, atol=2e-3)


# ------------------------------------------------------------- compaction
@pytest.mark.parametrize("name", ["w0", "w3", "w4"])
def test_compaction_bit_exact(name):
    w = make_workload(name)
    m = torch.from_numpy(w.mask)
    got = bsa.bsa_mask_compact(m.to(DEV), w.bx, w.by, w.seq_q, w.seq_kv)
    ref = O.compact_mask(w.mask, w.bx, w.by, w.seq_q, w.seq_kv)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g.cpu().numpy(), r)


def test_compaction_garbage_and_lengths():
    rng = np.random.Generator(np.random.PCG64(23))
    m = (rng.random((3, 5, 9, 7)) < 0.4).astype(np.uint8) * rng.integers(1, 255, (3, 5, 9, 7)).astype(np.uint8)
    sq, skv = [1100, 130, 1], [890, 64, 65]
    got = bsa.bsa_mask_compact(torch.from_numpy(m).to(DEV), 128, 128, sq, skv)
    ref = O.compact_mask(m, 128, 128, sq, skv)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g.cpu().numpy(), r)


# ------------------------------------------------------------------ forward
@pytest.mark.parametrize("layout,dtype,B,N1,N2,D,bx,by,sq,skv", [
    ("BNSD", "bf16", 2, 4, 2, 128, 128, 128, (300, 170), (300, 250)),
    ("BNSD", "f16", 1, 2, 1, 64, 64, 64, (200,), (333,)),
    ("TND", "f16", 3, 4, 2, 128, 128, 64, (200, 333, 64), (250, 129, 300)),
])
def test_forward_full(layout, dtype, B, N1, N2, D, bx, by, sq, skv):
    Sq = max(sq) if layout == "TND" else max(sq) + 9
    Skv = max(skv) if layout == "TND" else max(skv) + 3
    w = small_workload(layout=layout, dtype=dtype, B=B, N1=N1, N2=N2, D=D, bx=bx, by=by,
                       seq_q=sq, seq_kv=skv, Sq=Sq, Skv=Skv, p=0.5, seed=31 + D)
    w.mask[0, 0, 0, :] = 0                  # a query block with no keys
    dout, q, k, v = host_inputs(w)
    ref_out, ref_lse = oracle_forward(w, q, k, v)
    mask = torch.from_numpy(w.mask).to(DEV)
    out, lse, ws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[bx, by],
        actual_seq_lengths=list(sq), actual_seq_lengths_kv=list(skv), layout=layout,
        num_key_value_heads=N2, scale_value=w.scale)
    bsa.bsa_check_status(ws)
    check("out", f64(out), ref_out)
    fin = np.isfinite(ref_lse)
    got_lse = f64(lse)
    np.testing.assert_array_equal(np.isneginf(got_lse), ~fin)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)


# ------------------------------------------------------------ failure path
def test_bounded_wait_reports_error_and_context_survives():
    """A wait on a barrier nothing completes gives up after its bound; the host
    reads 561002 and the next run on the same context is correct."""
    w = small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(256,), seq_kv=(256,),
                       p=1.0, seed=41)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    g = [t.to(DEV) for t in (dout, q, k, v, tout, tlse)]
    mask = torch.from_numpy(w.mask).to(DEV)
    dq, dk, dv = (torch.empty_like(g[i]) for i in (1, 2, 3))
    size, ex = bsa.bsa_grad_workspace_size(*g, mask, None, [128, 128], None, None, "BNSD", "BNSD",
                                           1, 0, w.scale, dq=dq, dk=dk, dv=dv)
    ex.set_wait_test(True)
    ws = torch.empty(size, dtype=torch.uint8, device=DEV)
    bsa.bsa_grad(ws, size, ex)
    with pytest.raises(bsa.BsaError) as err:
        bsa.bsa_check_status(ws)
    assert err.value.status == 561002
    hdr = ws[:128].view(torch.int32).cpu().tolist()
    assert hdr[6] == 12 or hdr[16 + 12] > 0       # the test wait is among the recorded codes
    full_case(w)                                   # the context still computes correctly


def test_zero_length_sequences():
    """TND batches with no queries, no keys or neither, between non-empty ones:
    nothing is read or written for them, rows without keys get dQ = 0, and the
    forward gives Out = 0 and lse = -inf there."""
    w = small_workload(layout="TND", dtype="bf16", B=5, N1=4, N2=2, D=128, bx=128, by=64,
                       seq_q=(0, 150, 70, 0, 200), seq_kv=(90, 0, 130, 0, 260), p=0.8, seed=29)
    full_case(w)
    dout, q, k, v = host_inputs(w)
    ref_out, ref_lse = oracle_forward(w, q, k, v)
    mask = torch.from_numpy(w.mask).to(DEV)
    out, lse, ws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[w.bx, w.by],
        actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv, layout="TND",
        num_key_value_heads=w.N2, scale_value=w.scale)
    bsa.bsa_check_status(ws)
    check("zero-len:fwd_out", f64(out), ref_out)
    np.testing.assert_array_equal(np.isneginf(f64(lse)), np.isneginf(ref_lse))
    assert np.all(np.isneginf(f64(lse)[0:150]))        # batch 1: 150 queries, no keys


def test_largest_gqa_group():
    """G = N1/N2 = 256, the largest group the work lists encode (8 bits of
    local head), with ragged tiles. In fp16: dK and dV of a key sum 256 heads'
    contributions, and with bf16 operands the rounding of P and dS alone (the
    kernel's exact arithmetic, emulated on the host, lands on the GPU's
    values) exceeds the per-element bound on some elements."""
    w = small_workload(layout="BNSD", dtype="f16", B=1, N1=256, N2=1, D=64, bx=64, by=64,
                       seq_q=(130,), seq_kv=(200,), p=0.5, seed=37)
    full_case(w)


def test_many_short_sequences():
    """TND with 1200 sequences of 1-40 tokens (a few zero-length): the
    per-batch tables (7 ints per sequence) reach the device in two
    kernel-parameter uploads, and every sequence is a single ragged tile.
    In fp16: rows that see a handful of keys have large P and dS whose terms
    cancel in dQ, where the bf16 rounding of P and dS alone exceeds the
    per-element bound on a few elements (2 of ~3 M in bf16)."""
    rng = np.random.Generator(np.random.PCG64(97))
    sq = [int(x) for x in rng.integers(0, 41, size=1200)]
    skv = [int(x) for x in rng.integers(1, 41, size=1200)]
    w = small_workload(layout="TND", dtype="f16", B=1200, N1=2, N2=1, D=64, bx=64, by=64,
                       seq_q=sq, seq_kv=skv, p=0.8, seed=101)
    full_case(w)
