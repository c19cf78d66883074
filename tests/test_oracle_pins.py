"""Pins for the fp64 oracle: each test checks it against something other than
itself (a library routine, autograd, finite differences, a closed form,
invariants of softmax attention, brute force), chosen so that a plausible
mistake (dropped term, wrong sign or index, transposed operand, wrong head
group, wrong block index) fails at least one of them. ``test_planted_mistakes``
plants such mistakes in the oracle and checks that the pins catch them."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import bsa_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(shape, seed, std=1.0):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape) * std


def _case(B=1, N1=2, N2=1, S=40, Skv=None, D=8, bx=8, by=8, p=0.5, seed=0, diag=True):
    Skv = S if Skv is None else Skv
    q = _rand((B, N1, S, D), seed)
    k = _rand((B, N2, Skv, D), seed + 1)
    v = _rand((B, N2, Skv, D), seed + 2)
    do = _rand((B, N1, S, D), seed + 3)
    Mq, Mk = -(-S // bx), -(-Skv // by)
    rng = np.random.Generator(np.random.PCG64(seed + 4))
    m = (rng.random((B, N1, Mq, Mk)) < p).astype(np.uint8)
    if diag:
        for i in range(min(Mq, Mk)):
            m[:, :, i, i] = 1
        m[:, :, :, 0] = np.maximum(m[:, :, :, 0], 1)   # every query row has a key
    return q, k, v, do, m


def _sdpa_fwd_bwd(q, k, v, do, m, bx, by, scale, G):
    """torch SDPA (float64, CPU) with the block mask expanded to tokens."""
    B, N1, S, D = q.shape
    Skv = k.shape[2]
    if m is None:
        tm = np.ones((B, N1, S, Skv), dtype=bool)
    else:   # expanded here with np.repeat, independently of the oracle
        tm = np.repeat(np.repeat(np.asarray(m) != 0, bx, axis=2), by, axis=3)[:, :, :S, :Skv]
    Q = torch.tensor(q, requires_grad=True)
    K = torch.tensor(k, requires_grad=True)
    V = torch.tensor(v, requires_grad=True)
    Kr = K.repeat_interleave(G, dim=1)
    Vr = V.repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(
        Q, Kr, Vr, attn_mask=torch.tensor(tm), scale=scale)
    out.backward(torch.tensor(do))
    return out.detach().numpy(), Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


# ---------------------------------------------------------------- forward pins
@pytest.mark.parametrize("N1,N2,S,Skv,bx,by", [(2, 2, 40, 40, 8, 8), (4, 2, 33, 50, 8, 16),
                                               (3, 1, 64, 24, 16, 8)])
def test_forward_matches_sdpa(N1, N2, S, Skv, bx, by):
    q, k, v, do, m = _case(N1=N1, N2=N2, S=S, Skv=Skv, bx=bx, by=by, seed=11)
    out, lse = O.forward(q, k, v, m, (bx, by), num_kv_heads=N2, scale=0.37)
    ref, *_ = _sdpa_fwd_bwd(q, k, v, do, m, bx, by, 0.37, N1 // N2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # lse against its definition, spelled out per row with the math library
    b, h, s = 0, N1 - 1, S - 1
    keys = [t for t in range(Skv) if m[b, h, s // bx, t // by]]
    g = h // (N1 // N2)
    xs = [0.37 * float(np.dot(q[b, h, s], k[b, g, t])) for t in keys]
    mx = max(xs)
    assert abs(lse[b, h, s, 0] - (mx + math.log(sum(math.exp(x - mx) for x in xs)))) < 1e-12


def test_forward_dense_matches_sdpa_no_mask():
    q, k, v, do, _ = _case(N1=2, N2=1, S=48, D=16)
    out, _ = O.forward(q, k, v, None, (16, 16), num_kv_heads=1, scale=0.25)
    ref, *_ = _sdpa_fwd_bwd(q, k, v, do, None, 16, 16, 0.25, 2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_forward_blockrows_matches_forward():
    q, k, v, do, m = _case(N1=4, N2=2, S=70, Skv=90, bx=16, by=32, seed=5, diag=False)
    m[0, 1, 2, :] = 0                                   # an empty query block row
    a = O.forward(q, k, v, m, (16, 32), num_kv_heads=2, scale=0.5)
    b = O.forward_blockrows(q, k, v, m, (16, 32), num_kv_heads=2, scale=0.5)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(a[1]), np.isinf(b[1]))
    fin = np.isfinite(a[1])
    np.testing.assert_allclose(a[1][fin], b[1][fin], rtol=1e-12, atol=1e-12)
    # reading R6: an empty row has out 0 and lse -inf
    assert np.all(a[0][0, 1, 32:48] == 0) and np.all(np.isneginf(a[1][0, 1, 32:48]))


# --------------------------------------------------------------- backward pins
@pytest.mark.parametrize("N1,N2,S,Skv,D,bx,by,seed", [(2, 2, 40, 40, 8, 8, 8, 1),
                                                      (4, 2, 37, 52, 16, 8, 16, 2),
                                                      (4, 1, 64, 64, 8, 16, 16, 3),
                                                      (2, 1, 24, 70, 4, 8, 32, 4)])
def test_backward_matches_sdpa_autograd(N1, N2, S, Skv, D, bx, by, seed):
    q, k, v, do, m = _case(N1=N1, N2=N2, S=S, Skv=Skv, D=D, bx=bx, by=by, seed=seed)
    scale = D ** -0.5
    out, lse = O.forward(q, k, v, m, (bx, by), num_kv_heads=N2, scale=scale)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, m, (bx, by), num_kv_heads=N2, scale=scale)
    _, gq, gk, gv = _sdpa_fwd_bwd(q, k, v, do, m, bx, by, scale, N1 // N2)
    for a, b in ((dq, gq), (dk, gk), (dv, gv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_backward_finite_differences():
    """Central differences of L = <dOut, Out(Q, K, V)> on a tiny case."""
    q, k, v, do, m = _case(B=1, N1=2, N2=1, S=12, Skv=10, D=4, bx=4, by=4, seed=21)
    scale, bs = 0.6, (4, 4)

    def loss(q_, k_, v_):
        o, _ = O.forward(q_, k_, v_, m, bs, num_kv_heads=1, scale=scale)
        return float((o * do).sum())

    out, lse = O.forward(q, k, v, m, bs, num_kv_heads=1, scale=scale)
    grads = O.backward(do, q, k, v, out, lse, m, bs, num_kv_heads=1, scale=scale)
    h = 1e-6
    for which, (x, g) in enumerate(zip((q, k, v), grads)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(fd - g).max() / max(1e-3, np.abs(g).max())
        assert err < 1e-6, (which, err)


def test_softmax_shift_invariants():
    """Shifting every key by c leaves the softmax unchanged, so sum_t dK_t = 0
    (equivalently sum_t dS_st = 0 per row); shifting every value by c shifts Out
    by c, so sum_t dV_t = sum over rows with keys of dOut_s. Both need a
    consistent fp64 Out and lse."""
    q, k, v, do, m = _case(N1=4, N2=2, S=50, Skv=45, D=8, bx=8, by=8, seed=31, diag=False)
    m[0, 0, 3, :] = 0                              # rows 24..31 of head 0: no keys
    out, lse = O.forward(q, k, v, m, (8, 8), num_kv_heads=2, scale=0.4)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, m, (8, 8), num_kv_heads=2, scale=0.4)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12 * max(1.0, np.abs(dk).max()) * 100
    has = np.isfinite(lse[..., 0])
    rhs = np.where(has[..., None], do, 0.0).reshape(1, 2, 2, 50, 8).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), rhs, rtol=1e-10, atol=1e-10)
    assert np.all(dq[0, 0, 24:32] == 0)


def test_null_mask_equals_all_ones():
    q, k, v, do, _ = _case(N1=2, N2=1, S=40, Skv=40, D=8)
    ones = np.ones((1, 2, 5, 5), np.uint8)
    out, lse = O.forward(q, k, v, None, (8, 8), num_kv_heads=1, scale=0.3)
    a = O.backward(do, q, k, v, out, lse, None, (8, 8), num_kv_heads=1, scale=0.3)
    b = O.backward(do, q, k, v, out, lse, ones, (8, 8), num_kv_heads=1, scale=0.3)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_unselected_blocks_contribute_nothing():
    q, k, v, do, m = _case(N1=2, N2=1, S=32, Skv=48, D=8, bx=8, by=8, seed=41, diag=False)
    m[:, :, :, 0] = 1
    m[:, :, :, 3] = 0                                   # key block 3 (rows 24..31): unused
    out, lse = O.forward(q, k, v, m, (8, 8), num_kv_heads=1, scale=0.5)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, m, (8, 8), num_kv_heads=1, scale=0.5)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 24:32] += 100.0
    v2[:, :, 24:32] -= 100.0
    dq2, dk2, dv2 = O.backward(do, q, k2, v2, out, lse, m, (8, 8), num_kv_heads=1, scale=0.5)
    np.testing.assert_array_equal(dq, dq2)
    assert np.all(dk[:, :, 24:32] == 0) and np.all(dv[:, :, 24:32] == 0)
    assert np.all(dk2[:, :, 24:32] == 0) and np.all(dv2[:, :, 24:32] == 0)


def test_bits_outside_valid_range_are_ignored():
    q, k, v, do, m = _case(N1=2, N2=1, S=64, Skv=64, D=8, bx=16, by=16, seed=51)
    sq, skv = [37], [45]                                # BNSD with actual lengths
    out, lse = O.forward(q, k, v, m, (16, 16), sq, skv, num_kv_heads=1, scale=0.5)
    a = O.backward(do, q, k, v, out, lse, m, (16, 16), sq, skv, num_kv_heads=1, scale=0.5)
    m2 = m.copy()
    m2[:, :, 3, :] = 1                                  # block row 3 starts at 48 >= 37
    m2[:, :, :, 3] = 1                                  # block col 3 starts at 48 >= 45
    b = O.backward(do, q, k, v, out, lse, m2, (16, 16), sq, skv, num_kv_heads=1, scale=0.5)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert np.all(a[0][:, :, 37:] == 0) and np.all(a[1][:, :, 45:] == 0)
    # padding contents do not matter
    q3, k3 = q.copy(), k.copy()
    q3[:, :, 37:] = 1e6
    k3[:, :, 45:] = -1e6
    c = O.backward(do, q3, k3, v, out, lse, m, (16, 16), sq, skv, num_kv_heads=1, scale=0.5)
    for x, y in zip(a, c):
        np.testing.assert_array_equal(x, y)


def test_page_call_example_closed_form():
    """The page's call example: q = k = v = out = 0.1, dout = 0.01 (fp16), lse = 5,
    S = 128, D = 128, 64x64 blocks, all-ones mask, scale = 1/sqrt(128)."""
    with open(os.path.join(HERE, "golden", "p1_call_example.json")) as f:
        g = json.load(f)
    S, D = g["q_seqlen"], g["head_dim"]
    x = float(np.float16(g["q_k_v_out_value"]))
    assert x == g["q_k_v_out_f16"]
    d = float(np.float16(g["dout_value"]))
    assert d == g["dout_f16"]
    q = np.full((1, 1, S, D), x)
    dout = np.full((1, 1, S, D), d)
    lse = np.full((1, 1, S), g["lse_value"])
    mask = np.ones((1, 1, 2, 2), np.uint8)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = O.backward(dout, q, q, q, q, lse, mask, tuple(g["block_shape"]),
                            num_kv_heads=1, scale=scale)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    expect = S * math.exp(scale * D * x * x - g["lse_value"]) * d
    assert abs(expect - g["closed_form"]["dv_value"]) < 1e-15
    np.testing.assert_allclose(dv, expect, rtol=1e-12)


def test_gqa_equals_mha_with_repeated_heads():
    q, k, v, do, m = _case(N1=6, N2=2, S=30, Skv=40, D=8, bx=8, by=8, seed=61)
    out, lse = O.forward(q, k, v, m, (8, 8), num_kv_heads=2, scale=0.4)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, m, (8, 8), num_kv_heads=2, scale=0.4)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    dq2, dk2, dv2 = O.backward(do, q, kr, vr, out, lse, m, (8, 8), num_kv_heads=6, scale=0.4)
    np.testing.assert_allclose(dq, dq2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(1, 2, 3, 40, 8).sum(2), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(1, 2, 3, 40, 8).sum(2), rtol=1e-12, atol=1e-13)


def test_tnd_equals_bnsd_per_sequence():
    lens_q, lens_k = [13, 30, 7], [21, 9, 30]
    N1, N2, D, bx, by = 4, 2, 8, 8, 8
    Mq, Mk = 4, 4
    rng = np.random.Generator(np.random.PCG64(71))
    m = (rng.random((3, N1, Mq, Mk)) < 0.6).astype(np.uint8)
    m[:, :, :, 0] = 1
    qt = _rand((sum(lens_q), N1, D), 72)
    kt = _rand((sum(lens_k), N2, D), 73)
    vt = _rand((sum(lens_k), N2, D), 74)
    dot = _rand((sum(lens_q), N1, D), 75)
    out, lse = O.forward(qt, kt, vt, m, (bx, by), lens_q, lens_k, "TND", N2, 0.3)
    dq, dk, dv = O.backward(dot, qt, kt, vt, out, lse, m, (bx, by), lens_q, lens_k, "TND", N2, 0.3)
    oq, ok = O.seq_offsets(lens_q), O.seq_offsets(lens_k)
    for b in range(3):
        sl_q, sl_k = slice(oq[b], oq[b + 1]), slice(ok[b], ok[b + 1])
        to_bnsd = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2))[None]
        o1, l1 = O.forward(to_bnsd(qt[sl_q]), to_bnsd(kt[sl_k]), to_bnsd(vt[sl_k]),
                           m[b:b + 1], (bx, by), num_kv_heads=N2, scale=0.3)
        np.testing.assert_allclose(o1[0].transpose(1, 0, 2), out[sl_q], rtol=1e-13, atol=1e-14)
        g1 = O.backward(to_bnsd(dot[sl_q]), to_bnsd(qt[sl_q]), to_bnsd(kt[sl_k]), to_bnsd(vt[sl_k]),
                        o1, l1, m[b:b + 1], (bx, by), num_kv_heads=N2, scale=0.3)
        for x, y, sl in zip(g1, (dq, dk, dv), (sl_q, sl_k, sl_k)):
            np.testing.assert_allclose(x[0].transpose(1, 0, 2), y[sl], rtol=1e-12, atol=1e-13)


def test_bruteforce_every_tiny_mask():
    """B = N = 1, S = 8, 4x4 blocks: all 16 masks against SDPA + autograd."""
    q, k, v, do, _ = _case(B=1, N1=1, N2=1, S=8, D=4, bx=4, by=4, seed=81)
    for bits in range(16):
        m = np.array([(bits >> i) & 1 for i in range(4)], np.uint8).reshape(1, 1, 2, 2)
        out, lse = O.forward(q, k, v, m, (4, 4), num_kv_heads=1, scale=0.7)
        dq, dk, dv = O.backward(do, q, k, v, out, lse, m, (4, 4), num_kv_heads=1, scale=0.7)
        rows_with_keys = [i for i in range(2) if m[0, 0, i].any()]
        if len(rows_with_keys) < 2:
            # SDPA gives NaN for rows without keys; check them by reading R6
            for i in range(2):
                if i not in rows_with_keys:
                    assert np.all(out[0, 0, 4 * i:4 * i + 4] == 0)
                    assert np.all(dq[0, 0, 4 * i:4 * i + 4] == 0)
            if not rows_with_keys:
                assert np.all(dk == 0) and np.all(dv == 0)
                continue
            r = slice(4 * rows_with_keys[0], 4 * rows_with_keys[0] + 4)
            ref, gq, gk, gv = _sdpa_fwd_bwd(q[:, :, r], k, v, do[:, :, r],
                                            m[:, :, rows_with_keys[0]:rows_with_keys[0] + 1],
                                            4, 4, 0.7, 1)
            np.testing.assert_allclose(out[:, :, r], ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(dq[:, :, r], gq, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dk, gk, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dv, gv, rtol=1e-10, atol=1e-12)
            continue
        ref, gq, gk, gv = _sdpa_fwd_bwd(q, k, v, do, m, 4, 4, 0.7, 1)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
        for a, b in ((dq, gq), (dk, gk), (dv, gv)):
            np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_sampled_rows_match_full_backward():
    q, k, v, do, m = _case(N1=4, N2=2, S=60, Skv=50, D=8, bx=16, by=8, seed=91)
    out, lse = O.forward(q, k, v, m, (16, 8), num_kv_heads=2, scale=0.3)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, m, (16, 8), num_kv_heads=2, scale=0.3)
    rows = np.array([0, 17, 59])
    np.testing.assert_allclose(
        O.backward_dq_rows(do, q, k, v, out, lse, 0, 3, rows, m, (16, 8), num_kv_heads=2, scale=0.3),
        dq[0, 3, rows], rtol=1e-13, atol=1e-14)
    a, b = O.backward_dkdv_rows(do, q, k, v, out, lse, 0, 1, np.array([1, 25, 49]), m, (16, 8),
                                num_kv_heads=2, scale=0.3)
    np.testing.assert_allclose(a, dk[0, 1, [1, 25, 49]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b, dv[0, 1, [1, 25, 49]], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ compaction pins
def test_compaction_brute_force():
    rng = np.random.Generator(np.random.PCG64(101))
    B, N, Mq, Mk, bx, by = 2, 3, 7, 5, 16, 32
    m = (rng.random((B, N, Mq, Mk)) < 0.4).astype(np.uint8) * rng.integers(1, 255, (B, N, Mq, Mk)).astype(np.uint8)
    sq, skv = [100, 112], [150, 70]                     # clips rows/cols per batch
    rp, ci, cp, ri = O.compact_mask(m, bx, by, sq, skv)
    assert rp.dtype == np.int32 and len(rp) == B * N * (Mq + 1) and len(cp) == B * N * (Mk + 1)
    dense_r = np.zeros_like(m, dtype=bool)
    dense_c = np.zeros_like(m, dtype=bool)
    for b in range(B):
        for h in range(N):
            sl = b * N + h
            for i in range(Mq):
                cols = ci[rp[sl * (Mq + 1) + i]:rp[sl * (Mq + 1) + i + 1]]
                assert np.all(np.diff(cols) > 0)
                dense_r[b, h, i, cols] = True
            for j in range(Mk):
                rws = ri[cp[sl * (Mk + 1) + j]:cp[sl * (Mk + 1) + j + 1]]
                assert np.all(np.diff(rws) > 0)
                dense_c[b, h, rws, j] = True
    valid = np.zeros_like(dense_r)
    for b in range(B):
        valid[b, :, :-(-sq[b] // bx), :-(-skv[b] // by)] = True
    expect = (m != 0) & valid
    np.testing.assert_array_equal(dense_r, expect)
    np.testing.assert_array_equal(dense_c, expect)
    assert len(ci) == len(ri) == int(expect.sum())


# -------------------------------------------------------- planted mistakes
def _planted(kind):
    def head_backward(Qm, Km, Vm, dOm, Om, lse, M, scale):
        Dv = (dOm * Om).sum(axis=1)
        if kind == "drop_D":
            Dv = 0 * Dv
        S = scale * (Qm @ Km.T)
        if kind == "lse_sign":
            S = S + 2 * lse[:, None]
        P = np.where(M, np.exp(np.where(M, S - lse[:, None], 0.0)), 0.0)
        if kind == "mask_ignored":
            P = np.exp(np.minimum(S - lse[:, None], 50.0))
        dP = dOm @ Vm.T
        dS = P * (dP - Dv[:, None])
        if kind == "dS_sign":
            dS = P * (Dv[:, None] - dP)
        dV = P.T @ dOm
        if kind == "dV_uses_dS":
            dV = dS.T @ dOm
        dQ = scale * (dS @ Km)
        if kind == "dq_no_scale":
            dQ = dS @ Km
        dK = scale * (dS.T @ Qm)
        if kind == "dk_uses_P":
            dK = scale * (P.T @ Qm)
        return dQ, dK, dV
    return head_backward


PINS = [
    lambda: test_backward_matches_sdpa_autograd(4, 2, 37, 52, 16, 8, 16, 2),
    test_softmax_shift_invariants,
    test_page_call_example_closed_form,
    test_unselected_blocks_contribute_nothing,
]


@pytest.mark.parametrize("kind", ["drop_D", "lse_sign", "mask_ignored", "dS_sign",
                                  "dV_uses_dS", "dq_no_scale", "dk_uses_P"])
def test_planted_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(O, "_head_backward", _planted(kind))
    caught = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught >= 1, kind


def test_planted_block_index_mistake_is_caught(monkeypatch):
    """mask[b, h, j, i] read instead of mask[b, h, i, j]."""
    real = O.token_mask
    monkeypatch.setattr(O, "token_mask", lambda bm, bx, by, Lq, Lk, *w:
                        real(None if bm is None else np.asarray(bm).T, bx, by, Lq, Lk, *w))
    with pytest.raises(AssertionError):
        test_backward_matches_sdpa_autograd(2, 2, 40, 40, 8, 8, 8, 1)


def test_planted_gqa_mapping_mistake_is_caught(monkeypatch):
    """Query head h paired with key head h % N2 instead of h // (N1/N2)."""
    def wrong(dout, q, k, v, out, lse, mask=None, block_shape=(128, 128), seq_q=None,
              seq_kv=None, layout="BNSD", num_kv_heads=None, scale=1.0):
        B, N1, S, D = q.shape
        N2, Skv = k.shape[1], k.shape[2]
        dq = np.zeros(q.shape)
        dk = np.zeros(k.shape)
        dv = np.zeros(v.shape)
        for b in range(B):
            for h in range(N1):
                g = h % N2
                M = O.token_mask(mask[b, h], block_shape[0], block_shape[1], S, Skv)
                a, c, e = O._head_backward(q[b, h], k[b, g], v[b, g], dout[b, h], out[b, h],
                                           lse[b, h, :, 0], M, scale)
                dq[b, h] = a
                dk[b, g] += c
                dv[b, g] += e
        return dq, dk, dv
    monkeypatch.setattr(O, "backward", wrong)
    with pytest.raises(AssertionError):
        test_backward_matches_sdpa_autograd(4, 2, 37, 52, 16, 8, 16, 2)


def test_token_mask_at_matches_full_expansion():
    rng = np.random.Generator(np.random.PCG64(111))
    bm = (rng.random((5, 7)) < 0.5).astype(np.uint8)
    full = O.token_mask(bm, 16, 8, 70, 50)
    rows, cols = np.array([0, 15, 16, 69]), np.array([0, 7, 8, 49])
    np.testing.assert_array_equal(O.token_mask_at(bm, 16, 8, rows, cols), full[rows][:, cols])
    ref = np.repeat(np.repeat(bm != 0, 16, axis=0), 8, axis=1)[:70, :50]   # independent expansion
    np.testing.assert_array_equal(full, ref)


# -------------------------------------------- sliding window (reading R18) pins
def _sdpa_rows(q, k, v, do, tm, scale, G):
    """torch SDPA + autograd (float64, CPU) per (b, h) on the query rows that
    have at least one key in the token mask tm [B, N1, S, Skv]; rows without a
    key are left at 0 (reading R6), which SDPA itself cannot express (NaN)."""
    B, N1, S, D = q.shape
    out, dq = np.zeros(q.shape), np.zeros(q.shape)
    dk, dv = np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        for h in range(N1):
            rows = np.nonzero(tm[b, h].any(axis=1))[0]
            if len(rows) == 0:
                continue
            g = h // G
            Q = torch.tensor(q[b, h, rows][None, None], requires_grad=True)
            K = torch.tensor(k[b, g][None, None], requires_grad=True)
            V = torch.tensor(v[b, g][None, None], requires_grad=True)
            o = torch.nn.functional.scaled_dot_product_attention(
                Q, K, V, attn_mask=torch.tensor(tm[b, h][rows][None, None]), scale=scale)
            o.backward(torch.tensor(do[b, h, rows][None, None]))
            out[b, h, rows] = o.detach().numpy()[0, 0]
            dq[b, h, rows] = Q.grad.numpy()[0, 0]
            dk[b, g] += K.grad.numpy()[0, 0]
            dv[b, g] += V.grad.numpy()[0, 0]
    return out, dq, dk, dv


@pytest.mark.parametrize("S,Skv", [(37, 37), (29, 50), (50, 29)])
def test_causal_matches_sdpa_is_causal(S, Skv):
    """nextTokens = 0, preTokens = no limit, no block mask: torch's is_causal
    (lower triangle anchored at the top-left corner, also for S != Skv)."""
    q, k, v, do, _ = _case(N1=4, N2=2, S=S, Skv=Skv, D=8, seed=121)
    out, lse = O.forward(q, k, v, None, (8, 8), num_kv_heads=2, scale=0.45, next_tokens=0)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, None, (8, 8), num_kv_heads=2, scale=0.45,
                            next_tokens=0)
    Q, K, V = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K.repeat_interleave(2, dim=1), V.repeat_interleave(2, dim=1), is_causal=True,
        scale=0.45)
    ref.backward(torch.tensor(do))
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-12, atol=1e-13)
    for a, g in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        np.testing.assert_allclose(a, g.numpy(), rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("pre,nxt", [(13, 6), (9, -3), (-2, 5), (0, 0), (3, 40)])
def test_window_with_blocks_matches_sdpa(pre, nxt):
    """Window x block mask against SDPA with the token mask built from
    torch.tril / torch.triu diagonals and np.repeat (not the oracle's formula)."""
    S, Skv, bx, by = 40, 45, 8, 16
    q, k, v, do, m = _case(N1=4, N2=2, S=S, Skv=Skv, D=8, bx=bx, by=by, seed=131, p=0.6)
    blocks = np.repeat(np.repeat(m != 0, bx, axis=2), by, axis=3)[:, :, :S, :Skv]
    band = torch.ones(S, Skv, dtype=torch.bool).tril(nxt).triu(-pre).numpy()
    tm = blocks & band[None, None]
    out, lse = O.forward(q, k, v, m, (bx, by), num_kv_heads=2, scale=0.5, pre_tokens=pre,
                         next_tokens=nxt)
    grads = O.backward(do, q, k, v, out, lse, m, (bx, by), num_kv_heads=2, scale=0.5,
                       pre_tokens=pre, next_tokens=nxt)
    ref, *rg = _sdpa_rows(q, k, v, do, tm, 0.5, 2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    for a, b in zip(grads, rg):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)
    keyless = ~tm.any(axis=3)
    assert np.all(np.isneginf(lse[..., 0][keyless])) and np.all(np.isfinite(lse[..., 0][~keyless]))
    if pre == 9:   # rows 0..2 see no key of the window at all
        assert keyless[:, :, :3].all()
    bo = O.forward_blockrows(q, k, v, m, (bx, by), num_kv_heads=2, scale=0.5, pre_tokens=pre,
                             next_tokens=nxt)
    np.testing.assert_allclose(bo[0], out, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(bo[1]), np.isneginf(lse))


def test_window_edges_and_no_window():
    """preTokens >= Lq - 1 and nextTokens >= Lk - 1 reach every pair, so the
    result equals no window bit for bit; one less on either side drops exactly
    the corner pair (Lq-1, 0) or (0, Lk-1)."""
    S, Skv = 24, 30
    q, k, v, do, m = _case(N1=2, N2=1, S=S, Skv=Skv, D=8, bx=8, by=8, seed=141)
    kw = dict(num_kv_heads=1, scale=0.4)
    out, lse = O.forward(q, k, v, m, (8, 8), **kw)
    base = O.backward(do, q, k, v, out, lse, m, (8, 8), **kw)
    for pre, nxt in ((S - 1, Skv - 1), (10 ** 6, 10 ** 6), (2 ** 62, 2 ** 62)):
        o2, l2 = O.forward(q, k, v, m, (8, 8), pre_tokens=pre, next_tokens=nxt, **kw)
        np.testing.assert_array_equal(o2, out)
        np.testing.assert_array_equal(l2, lse)
        for a, b in zip(O.backward(do, q, k, v, out, lse, m, (8, 8), pre_tokens=pre,
                                   next_tokens=nxt, **kw), base):
            np.testing.assert_array_equal(a, b)
    m1 = np.ones_like(m)
    full = O.token_mask(m1[0, 0], 8, 8, S, Skv)
    lo = O.token_mask(m1[0, 0], 8, 8, S, Skv, pre_tokens=S - 2, next_tokens=Skv - 1)
    hi = O.token_mask(m1[0, 0], 8, 8, S, Skv, pre_tokens=S - 1, next_tokens=Skv - 2)
    assert full.all() and (~lo).sum() == 1 and not lo[S - 1, 0]
    assert (~hi).sum() == 1 and not hi[0, Skv - 1]


def test_tnd_window_restarts_per_sequence():
    """In TND the window positions count from each sequence's own start: the
    TND result equals per-sequence BNSD runs with the same window (BNSD itself
    is pinned to SDPA above)."""
    lens_q, lens_k = [13, 30, 7], [21, 9, 30]
    N1, N2, D, bx, by = 4, 2, 8, 8, 8
    rng = np.random.Generator(np.random.PCG64(151))
    m = (rng.random((3, N1, 4, 4)) < 0.7).astype(np.uint8)
    m[:, :, :, 0] = 1
    qt = _rand((sum(lens_q), N1, D), 152)
    kt = _rand((sum(lens_k), N2, D), 153)
    vt = _rand((sum(lens_k), N2, D), 154)
    dot = _rand((sum(lens_q), N1, D), 155)
    w = dict(pre_tokens=6, next_tokens=1)
    out, lse = O.forward(qt, kt, vt, m, (bx, by), lens_q, lens_k, "TND", N2, 0.3, **w)
    dq, dk, dv = O.backward(dot, qt, kt, vt, out, lse, m, (bx, by), lens_q, lens_k, "TND", N2,
                            0.3, **w)
    oq, ok = O.seq_offsets(lens_q), O.seq_offsets(lens_k)
    to_bnsd = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2))[None]
    for b in range(3):
        sl_q, sl_k = slice(oq[b], oq[b + 1]), slice(ok[b], ok[b + 1])
        o1, l1 = O.forward(to_bnsd(qt[sl_q]), to_bnsd(kt[sl_k]), to_bnsd(vt[sl_k]),
                           m[b:b + 1], (bx, by), num_kv_heads=N2, scale=0.3, **w)
        np.testing.assert_allclose(o1[0].transpose(1, 0, 2), out[sl_q], rtol=1e-13, atol=1e-14)
        g1 = O.backward(to_bnsd(dot[sl_q]), to_bnsd(qt[sl_q]), to_bnsd(kt[sl_k]),
                        to_bnsd(vt[sl_k]), o1, l1, m[b:b + 1], (bx, by), num_kv_heads=N2,
                        scale=0.3, **w)
        for x, y, sl in zip(g1, (dq, dk, dv), (sl_q, sl_k, sl_k)):
            np.testing.assert_allclose(x[0].transpose(1, 0, 2), y[sl], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", ["swap", "strict", "shifted"])
def test_planted_window_mistakes_are_caught(kind, monkeypatch):
    """pre and next exchanged, strict instead of inclusive edges, or the window
    shifted by one: each fails a window pin."""
    real = O.window_mask

    def wrong(rows, cols, pre_tokens=O.NO_WINDOW, next_tokens=O.NO_WINDOW):
        if kind == "swap":
            return real(rows, cols, next_tokens, pre_tokens)
        if kind == "strict":
            return real(rows, cols, pre_tokens - 1, next_tokens - 1)
        return real(rows, cols, pre_tokens + 1, next_tokens - 1)
    monkeypatch.setattr(O, "window_mask", wrong)
    caught = 0
    for pin in (lambda: test_window_with_blocks_matches_sdpa(13, 6),
                lambda: test_causal_matches_sdpa_is_causal(37, 37)):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught >= 1, kind


# ----------------------------------------- token mask attenMask (reading R19) pins
def _am(S, Skv, p, seed):
    return (np.random.Generator(np.random.PCG64(seed)).random((S, Skv)) < p).astype(np.uint8)


@pytest.mark.parametrize("pre,nxt", [(O.NO_WINDOW, O.NO_WINDOW), (20, 3)])
def test_atten_mask_with_blocks_matches_sdpa(pre, nxt):
    """attenMask (1 = masked) x window x block mask against SDPA with the
    combined token mask built here from np.repeat, torch.tril/triu and the
    inverted attenMask."""
    S, Skv, bx, by = 40, 45, 8, 16
    q, k, v, do, m = _case(N1=4, N2=2, S=S, Skv=Skv, D=8, bx=bx, by=by, seed=161, p=0.7)
    am = _am(S, Skv, 0.3, 162)
    blocks = np.repeat(np.repeat(m != 0, bx, axis=2), by, axis=3)[:, :, :S, :Skv]
    band = torch.ones(S, Skv, dtype=torch.bool).tril(min(nxt, Skv)).triu(-min(pre, S)).numpy()
    tm = blocks & band[None, None] & (am == 0)[None, None]
    kw = dict(num_kv_heads=2, scale=0.5, pre_tokens=pre, next_tokens=nxt, atten_mask=am)
    out, lse = O.forward(q, k, v, m, (bx, by), **kw)
    grads = O.backward(do, q, k, v, out, lse, m, (bx, by), **kw)
    ref, *rg = _sdpa_rows(q, k, v, do, tm, 0.5, 2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    for a, b in zip(grads, rg):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)
    bo = O.forward_blockrows(q, k, v, m, (bx, by), **kw)
    np.testing.assert_allclose(bo[0], out, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(bo[1]), np.isneginf(lse))


def test_atten_mask_upper_triangle_is_causal_and_zero_mask_is_none():
    """attenMask = np.triu(ones, 1) reproduces nextTokens = 0 bit for bit, a
    band written as a mask reproduces the window, and an all-zero attenMask
    changes nothing."""
    S, Skv = 33, 41
    q, k, v, do, m = _case(N1=2, N2=1, S=S, Skv=Skv, D=8, bx=8, by=8, seed=171)
    kw = dict(num_kv_heads=1, scale=0.4)

    def run(**extra):
        o, l = O.forward(q, k, v, m, (8, 8), **kw, **extra)
        return (o, l) + O.backward(do, q, k, v, o, l, m, (8, 8), **kw, **extra)
    base, causal, band = run(), run(next_tokens=0), run(pre_tokens=6, next_tokens=2)
    as_causal = run(atten_mask=np.triu(np.ones((S, Skv), np.uint8), 1))
    keep = np.tril(np.ones((S, Skv), bool), 2) & np.triu(np.ones((S, Skv), bool), -6)
    as_band = run(atten_mask=(~keep).astype(np.uint8))
    zero = run(atten_mask=np.zeros((S, Skv), np.uint8))
    for x, y in zip(causal, as_causal):
        np.testing.assert_array_equal(x, y)
    for x, y in zip(band, as_band):
        np.testing.assert_array_equal(x, y)
    for x, y in zip(base, zero):
        np.testing.assert_array_equal(x, y)
    full = run(atten_mask=np.ones((S, Skv), np.uint8))   # every pair masked: R6 everywhere
    assert np.all(full[0] == 0) and np.all(np.isneginf(full[1]))
    assert all(np.all(g == 0) for g in full[2:])


def test_tnd_atten_mask_is_per_sequence_top_left():
    lens_q, lens_k = [13, 30, 7], [21, 9, 30]
    N1, N2, D, bx, by = 4, 2, 8, 8, 8
    rng = np.random.Generator(np.random.PCG64(181))
    m = (rng.random((3, N1, 4, 4)) < 0.8).astype(np.uint8)
    am = _am(30, 30, 0.35, 182)
    qt = _rand((sum(lens_q), N1, D), 183)
    kt = _rand((sum(lens_k), N2, D), 184)
    vt = _rand((sum(lens_k), N2, D), 185)
    dot = _rand((sum(lens_q), N1, D), 186)
    w = dict(atten_mask=am, pre_tokens=9, next_tokens=4)
    out, lse = O.forward(qt, kt, vt, m, (bx, by), lens_q, lens_k, "TND", N2, 0.3, **w)
    dq, dk, dv = O.backward(dot, qt, kt, vt, out, lse, m, (bx, by), lens_q, lens_k, "TND", N2,
                            0.3, **w)
    oq, ok = O.seq_offsets(lens_q), O.seq_offsets(lens_k)
    to_bnsd = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2))[None]
    for b in range(3):
        sl_q, sl_k = slice(oq[b], oq[b + 1]), slice(ok[b], ok[b + 1])
        o1, l1 = O.forward(to_bnsd(qt[sl_q]), to_bnsd(kt[sl_k]), to_bnsd(vt[sl_k]),
                           m[b:b + 1], (bx, by), num_kv_heads=N2, scale=0.3, **w)
        np.testing.assert_allclose(o1[0].transpose(1, 0, 2), out[sl_q], rtol=1e-13, atol=1e-14)
        g1 = O.backward(to_bnsd(dot[sl_q]), to_bnsd(qt[sl_q]), to_bnsd(kt[sl_k]),
                        to_bnsd(vt[sl_k]), o1, l1, m[b:b + 1], (bx, by), num_kv_heads=N2,
                        scale=0.3, **w)
        for x, y, sl in zip(g1, (dq, dk, dv), (sl_q, sl_k, sl_k)):
            np.testing.assert_allclose(x[0].transpose(1, 0, 2), y[sl], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", ["keep_polarity", "transposed"])
def test_planted_atten_mask_mistakes_are_caught(kind, monkeypatch):
    """attenMask read as a keep-mask, or indexed [t, s]: the SDPA pin fails."""
    real = O.token_mask_at

    def wrong(bm, bx, by, rows, cols, pre=O.NO_WINDOW, nxt=O.NO_WINDOW, am=None):
        if am is not None:
            am = np.asarray(am)
            if kind == "keep_polarity":
                am = (am == 0).astype(np.uint8)
            else:
                sq = max(am.shape)
                pad = np.zeros((sq, sq), np.uint8)
                pad[:am.shape[0], :am.shape[1]] = am
                am = pad.T
        return real(bm, bx, by, rows, cols, pre, nxt, am)
    monkeypatch.setattr(O, "token_mask_at", wrong)
    with pytest.raises(AssertionError):
        test_atten_mask_with_blocks_matches_sdpa(O.NO_WINDOW, O.NO_WINDOW)


@pytest.mark.parametrize("how", ["blocks", "window", "atten_mask"])
def test_single_key_per_row_closed_form(how):
    """Each query sees only the key at its own position (an identity mask of
    1x1 blocks, the window pre = next = 0, or an attenMask that masks all but
    the diagonal): P = 1, so Out_s = V_s and lse_s = scale q_s.k_s, and
    dS = P (dP - D) = 0 since D_s = dOut_s.Out_s = dOut_s.V_s = dP_ss: dQ = dK = 0
    and dV_t = dOut_t."""
    S, D = 12, 8
    q, k, v, do, _ = _case(N1=1, N2=1, S=S, D=D, seed=191)
    kw = dict(num_kv_heads=1, scale=0.3)
    if how == "blocks":
        mask, bs = np.eye(S, dtype=np.uint8)[None, None], (1, 1)
    elif how == "window":
        mask, bs = None, (4, 4)
        kw.update(pre_tokens=0, next_tokens=0)
    else:
        mask, bs = None, (4, 4)
        kw.update(atten_mask=(1 - np.eye(S, dtype=np.uint8)))
    out, lse = O.forward(q, k, v, mask, bs, **kw)
    np.testing.assert_allclose(out, v, rtol=1e-14, atol=1e-14)
    expect_lse = 0.3 * np.einsum("bhsd,bhsd->bhs", q, k)[..., None]
    np.testing.assert_allclose(lse, expect_lse, rtol=1e-13, atol=1e-13)
    dq, dk, dv = O.backward(do, q, k, v, out, lse, mask, bs, **kw)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv, do, rtol=1e-13, atol=1e-14)


# -------------------------------------------- block-row backward (whole tensors)
def _blockrows_cases():
    """(args, kwargs) cases: BNSD GQA with non-square blocks, an empty block
    row and ragged tails; TND with a zero-length sequence; a window; a token
    mask; no block mask; garbage bits past the lengths."""
    cases = []
    q, k, v, do, m = _case(N1=4, N2=2, S=70, Skv=90, D=8, bx=16, by=32, seed=201, diag=False)
    m[0, 1, 2, :] = 0
    out, lse = O.forward(q, k, v, m, (16, 32), num_kv_heads=2, scale=0.5)
    cases.append(((do, q, k, v, out, lse, m, (16, 32)), dict(num_kv_heads=2, scale=0.5)))
    lens_q, lens_k = [13, 0, 30, 7], [21, 9, 30, 0]
    rng = np.random.Generator(np.random.PCG64(202))
    mt = (rng.random((4, 4, 4, 4)) < 0.6).astype(np.uint8)
    qt, kt, vt, dot = (_rand((sum(lens_q), 4, 8), 203), _rand((sum(lens_k), 2, 8), 204),
                       _rand((sum(lens_k), 2, 8), 205), _rand((sum(lens_q), 4, 8), 206))
    kwt = dict(seq_q=lens_q, seq_kv=lens_k, layout="TND", num_kv_heads=2, scale=0.3)
    ot, lt = O.forward(qt, kt, vt, mt, (8, 8), **kwt)
    cases.append(((dot, qt, kt, vt, ot, lt, mt, (8, 8)), kwt))
    q, k, v, do, m = _case(N1=2, N2=1, S=40, Skv=45, D=8, bx=8, by=16, seed=207, p=0.6)
    for extra in (dict(pre_tokens=9, next_tokens=-3), dict(atten_mask=_am(40, 45, 0.3, 208))):
        kw = dict(num_kv_heads=1, scale=0.5, **extra)
        o, l = O.forward(q, k, v, m, (8, 16), **kw)
        cases.append(((do, q, k, v, o, l, m, (8, 16)), kw))
    o, l = O.forward(q, k, v, None, (8, 16), num_kv_heads=1, scale=0.5)
    cases.append(((do, q, k, v, o, l, None, (8, 16)), dict(num_kv_heads=1, scale=0.5)))
    g = (rng.random(m.shape) < 0.5).astype(np.uint8)
    g[:, :, :2, :2] = m[:, :, :2, :2]
    kwl = dict(seq_q=[23], seq_kv=[30], num_kv_heads=1, scale=0.5)   # blocks past 23 / 30 are garbage
    o, l = O.forward(q, k, v, g, (8, 16), **kwl)
    cases.append(((do, q, k, v, o, l, g, (8, 16)), kwl))
    return cases


def test_backward_blockrows_matches_backward():
    for args, kw in _blockrows_cases():
        ref = O.backward(*args, **kw)
        got = O.backward_blockrows(*args, **kw)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_backward_blockrows_matches_sdpa_autograd():
    """Independently of the dense oracle: autograd of the fp64 SDPA with the
    block mask expanded by np.repeat (GQA, non-square blocks, tails)."""
    q, k, v, do, m = _case(N1=4, N2=2, S=37, Skv=52, D=16, bx=8, by=16, seed=211)
    out, lse = O.forward(q, k, v, m, (8, 16), num_kv_heads=2, scale=0.25)
    got = O.backward_blockrows(do, q, k, v, out, lse, m, (8, 16), num_kv_heads=2, scale=0.25)
    _, gq, gk, gv = _sdpa_fwd_bwd(q, k, v, do, m, 8, 16, 0.25, 2)
    for a, b in zip(got, (gq, gk, gv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


_BLOCKROWS_MUTATIONS = {
    "dk_assigned": ("dKh[keys] += c", "dKh[keys] = c"),          # later block rows overwrite
    "dv_assigned": ("dVh[keys] += e", "dVh[keys] = e"),
    "no_group_sum": ("for h in range(g * G, (g + 1) * G):", "for h in range(g * G, g * G + 1):"),
    "mask_of_kv_head": ("mask[b, h, i, :mk]", "mask[b, g, i, :mk]"),
    "window_rows_shifted": ("window_mask(np.arange(s0, s1), keys,",
                            "window_mask(np.arange(s0, s1) + 1, keys,"),
    "key_block_by_bx": ("np.arange(j * by, min(lk[b], (j + 1) * by))",
                        "np.arange(j * bx, min(lk[b], j * bx + by))"),
}


@pytest.mark.parametrize("kind", sorted(_BLOCKROWS_MUTATIONS))
def test_planted_blockrows_mistakes_are_caught(kind, monkeypatch):
    """Each mutation of the block-row backward's source (a plausible slip)
    fails one of its pins."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(O.backward_blockrows))
    old, new = _BLOCKROWS_MUTATIONS[kind]
    assert src.count(old) == 1, kind
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(O, "backward_blockrows", ns["backward_blockrows"])
    caught = 0
    for pin in (test_backward_blockrows_matches_backward,
                test_backward_blockrows_matches_sdpa_autograd):
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught += 1
    assert caught >= 1, kind
