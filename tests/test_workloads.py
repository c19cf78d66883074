"""CPU checks of the measurement bookkeeping: the FLOP counts of windowed and
token-masked workloads (pair counting) against brute force, the document
token mask's structure, and the JSON line of bench.py's reference arm."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from block_sparse_attention_attn_gb300.workloads import (NO_WINDOW, document_mask, make_workload,
                                                          small_workload, window_pairs)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("lq,lk,bx,by,pre,nxt,am_p", [
    (37, 50, 8, 16, 5, 0, None), (40, 33, 16, 8, NO_WINDOW, 0, None), (20, 20, 4, 4, 3, -1, None),
    (37, 45, 8, 16, NO_WINDOW, NO_WINDOW, 0.3), (64, 64, 16, 16, 10, 2, 0.5), (30, 50, 8, 8, -4, 9, 0.2),
])
def test_window_pairs_brute_force(lq, lk, bx, by, pre, nxt, am_p):
    am = None
    if am_p is not None:
        am = (np.random.Generator(np.random.PCG64(lq * lk)).random((lq + 3, lk + 5)) < am_p).astype(np.uint8)
    wp = window_pairs(lq, lk, bx, by, pre, nxt, am)
    bf = np.zeros((-(-lq // bx), -(-lk // by)), np.int64)
    for s in range(lq):
        for t in range(lk):
            if s - pre <= t <= s + nxt and (am is None or am[s, t] == 0):
                bf[s // bx, t // by] += 1
    np.testing.assert_array_equal(wp, bf)


def test_flops_without_and_with_a_full_window():
    w = small_workload(B=2, N1=4, N2=2, D=64, bx=64, by=64, seq_q=(256, 192), seq_kv=(256, 256),
                       p=0.5, seed=3)
    base = w.flops()
    assert base == 10.0 * 64 * 64 * 64 * w.active_blocks()
    w.pre_tokens, w.next_tokens = 10 ** 6, 10 ** 6   # reaches every pair: not a window
    assert not w.token_masked() and w.flops() == base
    w.next_tokens = 0                                # causal: fewer pairs, fewer blocks
    assert w.token_masked() and w.flops() < base
    w.pre_tokens, w.next_tokens = NO_WINDOW, NO_WINDOW
    w.atten_mask = np.zeros((256, 256), np.uint8)   # a token mask that masks nothing
    assert w.token_masked() and w.flops() == base   # (all blocks are full: lengths are multiples of 64)


def test_causal_workloads_count_half_the_dense_pairs():
    w = make_workload("w1causal")
    S, D, heads = w.Sq, w.D, w.B * w.N1
    assert w.flops() == 10.0 * D * heads * S * (S + 1) // 2
    assert w.active_blocks() == heads * (S // 128) * (S // 128 + 1) // 2


def test_document_mask_structure():
    am = document_mask(500, 500, 7, lo=40, hi=120)
    assert am.dtype == np.uint8 and am.shape == (500, 500)
    assert np.all(am[np.triu_indices(500, 1)] == 1)           # causal
    assert np.all(np.diag(am) == 0)                              # every query sees itself
    # each row's kept keys are one contiguous run ending at the diagonal
    for s in range(0, 500, 37):
        kept = np.nonzero(am[s] == 0)[0]
        assert kept[-1] == s and np.all(np.diff(kept) == 1)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "w0", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config", "dtype"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
