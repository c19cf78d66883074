"""Token mask attenMaskOptional (maskType 1; 1 = the pair is masked out) on the
GPU against the fp64 oracle: backward in both dQ modes, the forward, the
autograd pairing and the whole outputs of a full-size workload, alone and together
with the block mask and the sliding window."""
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


def random_am(S, Skv, p, seed):
    return np.random.Generator(np.random.PCG64(seed)).random((S, Skv)) < p


def document_am(S, Skv, seed, lo=40, hi=300, causal=True):
    """Documents of random lengths: a pair is masked when query and key lie in
    different documents (and, with ``causal``, when the key comes later)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = max(S, Skv)
    cuts = np.cumsum(rng.integers(lo, hi, size=n // lo + 2))
    doc = np.searchsorted(cuts, np.arange(n), side="right")
    am = doc[:S, None] != doc[None, :Skv]
    if causal:
        am |= np.arange(Skv)[None, :] > np.arange(S)[:, None]
    return am


def run_grad(w, dout, q, k, v, out, lse, am, pre=NOW, nxt=NOW, deterministic=False):
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    amt = am if isinstance(am, torch.Tensor) else torch.from_numpy(am).to(DEV)
    res = bsa.block_sparse_attention_grad(
        dout.to(DEV), q.to(DEV), k.to(DEV), v.to(DEV), out.to(DEV), lse.to(DEV),
        block_sparse_mask=mask, block_shape=[w.bx, w.by], actual_seq_lengths=w.seq_q,
        actual_seq_lengths_kv=w.seq_kv, layout=w.layout, num_key_value_heads=w.N2,
        scale_value=w.scale, deterministic=deterministic, pre_tokens=pre, next_tokens=nxt,
        atten_mask=amt)
    bsa.bsa_check_status(res[3])
    return res[:3]


def run_fwd(w, q, k, v, am, pre=NOW, nxt=NOW):
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(DEV)
    out, lse, ws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[w.bx, w.by],
        actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv, layout=w.layout,
        num_key_value_heads=w.N2, scale_value=w.scale, pre_tokens=pre, next_tokens=nxt,
        atten_mask=torch.from_numpy(am).to(DEV))
    bsa.bsa_check_status(ws)
    return out, lse


def am_case(w, am, pre=NOW, nxt=NOW, deterministic=False, am_dev=None):
    dout, q, k, v = host_inputs(w)
    win = dict(pre_tokens=pre, next_tokens=nxt, atten_mask=am)
    out, lse = oracle_forward(w, q, k, v, **win)
    tout, tlse = rounded_out_lse(w, out, lse)
    got = run_grad(w, dout, q, k, v, tout, tlse, am if am_dev is None else am_dev, pre, nxt,
                   deterministic)
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                     (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale, **win)
    tag = f"{w.name}:am:{'det' if deterministic else 'red'}"
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check(f"{tag}:{name}", f64(g), r)
    return (dout, q, k, v), (out, lse), got


# layout, dtype, B, N1, N2, D, bx, by, seq_q, seq_kv, block density, dense, mask kind, pre, next
CASES = [
    ("BNSD", "bf16", 2, 4, 2, 128, 128, 128, (300, 517), (300, 517), 0.8, False, "random", NOW, NOW),
    ("BNSD", "f16", 1, 4, 1, 64, 64, 64, (600,), (450,), 1.0, True, "document", NOW, NOW),
    ("TND", "f16", 3, 4, 2, 128, 64, 128, (300, 129, 513), (260, 400, 513), 0.8, False, "random",
     200, 10),
    ("BNSD", "bf16", 1, 2, 1, 128, 128, 64, (384,), (700,), 0.7, False, "document", NOW, NOW),
    # fp16: the first rows of each causal document see a handful of keys, so P
    # and dS are large there and their bf16 rounding alone (8-bit mantissa;
    # the kernel's exact arithmetic, emulated on the host, lands on the same
    # values) can exceed the per-element bound on elements near zero
    ("TND", "f16", 2, 8, 1, 64, 64, 64, (130, 257), (190, 77), 0.9, False, "document", NOW, 0),
]


def _setup(i, seed):
    layout, dtype, B, N1, N2, D, bx, by, sq, skv, p, dense, kind, pre, nxt = CASES[i]
    Sq = max(sq) if layout == "TND" else max(sq) + 11
    Skv = max(skv) if layout == "TND" else max(skv) + 7
    w = small_workload(layout=layout, dtype=dtype, B=B, N1=N1, N2=N2, D=D, bx=bx, by=by,
                       seq_q=sq, seq_kv=skv, Sq=Sq, Skv=Skv, p=p, seed=seed, dense=dense)
    am = random_am(Sq, Skv, 0.3, seed + 1) if kind == "random" else document_am(Sq, Skv, seed + 1)
    return w, am.astype(np.uint8), pre, nxt


@pytest.mark.parametrize("i", range(len(CASES)))
def test_atten_mask_backward(i):
    w, am, pre, nxt = _setup(i, 1000 + i)
    am_case(w, am, pre, nxt)


@pytest.mark.parametrize("i", [0, 2, 4])
def test_atten_mask_backward_deterministic(i):
    w, am, pre, nxt = _setup(i, 1100 + i)
    am_case(w, am, pre, nxt, deterministic=True)


def test_atten_mask_strided_and_larger_than_needed():
    """A bool view with strides (transposed storage) that is larger than
    [maxSq, maxSkv]: only its top-left corner is read."""
    w, am, pre, nxt = _setup(0, 1200)
    big = random_am(700, 800, 0.3, 1201)
    big[:am.shape[0], :am.shape[1]] = am != 0
    dev = torch.from_numpy(np.ascontiguousarray(big.T)).to(DEV).t()   # strides (1, 700)
    assert dev.stride() == (1, 700) and dev.dtype == torch.bool
    am_case(w, am, pre, nxt, am_dev=dev)


@pytest.mark.parametrize("i", [0, 1, 2])
def test_atten_mask_forward(i):
    w, am, pre, nxt = _setup(i, 1300 + i)
    if i == 1:
        am[5:9, :] = 1                       # rows with every key masked: Out 0, lse -inf
    dout, q, k, v = host_inputs(w)
    ref_out, ref_lse = oracle_forward(w, q, k, v, pre_tokens=pre, next_tokens=nxt, atten_mask=am)
    out, lse = run_fwd(w, q, k, v, am, pre, nxt)
    check(f"fwd:am:{i}:out", f64(out), ref_out)
    got_lse = f64(lse)
    fin = np.isfinite(ref_lse)
    np.testing.assert_array_equal(np.isneginf(got_lse), ~fin)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=1e-4, atol=1e-4)
    if i == 1:
        assert np.all(np.isneginf(got_lse[0, :, 5:9])) and np.all(f64(out)[0, :, 5:9] == 0)


def test_atten_mask_all_zero_equals_no_mask_and_all_ones_gives_zeros():
    w, _, _, _ = _setup(3, 1400)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v)
    tout, tlse = rounded_out_lse(w, out, lse)
    zero = np.zeros((w.Sq, w.Skv), np.uint8)
    a = run_grad(w, dout, q, k, v, tout, tlse, zero, deterministic=True)
    mask = torch.from_numpy(w.mask).to(DEV)
    b = bsa.block_sparse_attention_grad(
        dout.to(DEV), q.to(DEV), k.to(DEV), v.to(DEV), tout.to(DEV), tlse.to(DEV),
        block_sparse_mask=mask, block_shape=[w.bx, w.by], actual_seq_lengths=w.seq_q,
        actual_seq_lengths_kv=w.seq_kv, layout=w.layout, num_key_value_heads=w.N2,
        scale_value=w.scale, deterministic=True)
    bsa.bsa_check_status(b[3])
    for x, y in zip(a, b[:3]):
        assert torch.equal(x, y)
    ones = np.ones((w.Sq, w.Skv), np.uint8)
    for g in run_grad(w, dout, q, k, v, tout, tlse, ones):
        assert torch.all(g == 0)


def test_atten_mask_autograd():
    w = small_workload(layout="BNSD", dtype="bf16", B=2, N1=4, N2=2, D=128, bx=128, by=128,
                       seq_q=(384, 300), seq_kv=(384, 350), Sq=384, Skv=384, p=0.9, seed=1500)
    am = document_am(384, 384, 1501).astype(np.uint8)
    dout, q, k, v = host_inputs(w)
    mask = torch.from_numpy(w.mask).to(DEV)
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    out = bsa.block_sparse_attention(qd, kd, vd, block_sparse_mask=mask, block_shape=[128, 128],
                                     actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv,
                                     num_key_value_heads=w.N2, scale_value=w.scale,
                                     atten_mask=torch.from_numpy(am).to(DEV))
    out.backward(dout.to(DEV))
    ref_out, _ = oracle_forward(w, q, k, v, atten_mask=am)
    check("am-autograd:out", f64(out.detach()), ref_out)
    fo, fl = run_fwd(w, q, k, v, am)
    assert torch.equal(fo, out.detach())
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(fo), f64(fl), w.mask, (128, 128),
                     w.seq_q, w.seq_kv, "BNSD", w.N2, w.scale, atten_mask=am)
    for name, g, r in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), ref):
        check(f"am-autograd:{name}", f64(g), r)


def test_atten_mask_large_whole():
    """w1's shape and mask (BNSD B2 N16 S4096, Bernoulli(0.25) blocks) with
    causal documents of 200-1500 tokens as attenMask: whole dQ, dK, dV against
    the oracle, plus the forward on the full tensors. In fp16: the first rows
    of a document see a handful of keys, where P and dS are large and their
    rounding to bf16 operands alone (emulated on the host, it lands on the
    GPU's value) exceeds the per-element bound on single elements."""
    w = make_workload("w1")
    w.dtype = "f16"
    am = document_am(w.Sq, w.Skv, 1601, lo=200, hi=1500).astype(np.uint8)
    win = dict(atten_mask=am)
    dout, q, k, v = host_inputs(w)
    out, lse = oracle_forward(w, q, k, v, blockrows=True, **win)
    tout, tlse = rounded_out_lse(w, out, lse)
    del out, lse
    got = run_grad(w, dout, q, k, v, tout, tlse, am)
    check_whole("w1:am", got, oracle_backward_whole(w, dout, q, k, v, tout, tlse, **win))
    fo, fl = run_fwd(w, q, k, v, am)
    check("w1:am:fwd_out", f64(fo), f64(tout))
    fin = np.isfinite(f64(tlse))
    np.testing.assert_array_equal(np.isneginf(f64(fl)), ~fin)
    np.testing.assert_allclose(f64(fl)[fin], f64(tlse)[fin], rtol=1e-4, atol=2e-3)


def test_token_mask_drops_fully_masked_blocks():
    """Blocks whose every pair the token mask masks never reach the work lists:
    the number of (query tile, key tile) entries the compaction writes (header
    word 3) equals a host count of the selected blocks that keep a pair. A
    plan that lost the packed mask still computes correct gradients (the
    element masks zero the extra tiles), so only this count shows it."""
    w = small_workload(B=1, N1=2, N2=2, D=128, bx=128, by=128, seq_q=(1024,), seq_kv=(1024,),
                       p=0.6, seed=71)
    am = document_am(1024, 1024, seed=73, lo=60, hi=400)
    dout, q, k, v = host_inputs(w)
    g = [t.to(DEV) for t in (dout, q, k, v)]
    out, lse = run_fwd(w, q, k, v, am)
    dq, dk, dv = (torch.empty_like(g[i]) for i in (1, 2, 3))
    # the masks stay allocated until the run has read them (the executor keeps
    # their addresses, as it keeps every tensor's)
    mask_d, am_d = torch.from_numpy(w.mask).to(DEV), torch.from_numpy(am).to(DEV)
    size, ex = bsa.bsa_grad_workspace_size(*g, out, lse, mask_d, am_d, [128, 128],
                                           list(w.seq_q), list(w.seq_kv), "BNSD", "BNSD", 2, 1,
                                           w.scale, dq=dq, dk=dk, dv=dv)
    ws = torch.empty(size, dtype=torch.uint8, device=DEV)
    bsa.bsa_grad(ws, size, ex)
    bsa.bsa_check_status(ws)
    hdr = ws[:64].view(torch.int32).cpu().numpy()
    keeps = ~am.reshape(8, 128, 8, 128).all(axis=(1, 3))     # block (i, j) keeps a pair
    expect = int(((w.mask[0] != 0) & keeps[None]).sum())
    assert 0 < expect < w.mask[0].size
    assert int(hdr[3]) == expect
