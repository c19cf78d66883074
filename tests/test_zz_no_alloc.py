"""The allocation-free compaction entry point (bsa_mask_compact_noalloc).

It serves callers that cannot allocate device memory (a caller-owned pool that
forbids new allocations, an embedded runtime without a device allocator): it
keeps its scratch in an array built into the library instead of a workspace.
Its output must equal the workspace-based bsa_mask_compact and the oracle's
compaction exactly (integer index lists), on two calls in a row: the shared scratch keeps the previous
call's contents, and a stale count must not leak into the next result.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it."""
import numpy as np
import pytest
import torch

import block_sparse_attention_attn_gb300 as bsa
from block_sparse_attention_attn_gb300 import binding as B
from oracle import bsa_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _outputs(B_, N, Mq, Mk):
    return (torch.full((B_ * N * (Mq + 1),), -7, dtype=torch.int32, device=DEV),
            torch.full((B_ * N * Mq * Mk,), -7, dtype=torch.int32, device=DEV),
            torch.full((B_ * N * (Mk + 1),), -7, dtype=torch.int32, device=DEV),
            torch.full((B_ * N * Mq * Mk,), -7, dtype=torch.int32, device=DEV))


def _case(seed, B_, N, Mq, Mk, bx, by, p):
    rng = np.random.Generator(np.random.PCG64(seed))
    m = ((rng.random((B_, N, Mq, Mk)) < p) * rng.integers(1, 256, (B_, N, Mq, Mk))).astype(np.uint8)
    sq = [int(x) for x in rng.integers(1, Mq * bx + 1, size=B_)]
    skv = [int(x) for x in rng.integers(1, Mk * by + 1, size=B_)]
    return torch.from_numpy(m).to(DEV), sq, skv


def test_noalloc_matches_workspace_compaction_twice():
    # a larger call first, then a smaller one: the second must not see the first's counts
    cases = [_case(5, 3, 4, 40, 33, 128, 64, 0.4), _case(6, 2, 3, 9, 17, 64, 128, 0.6)]
    for mask, sq, skv in cases:
        B_, N, Mq, Mk = mask.shape
        bx, by = (128, 64) if Mq == 40 else (64, 128)
        ref = bsa.bsa_mask_compact(mask, bx, by, sq, skv)
        out = _outputs(B_, N, Mq, Mk)
        bsa.bsa_mask_compact_noalloc(mask, bx, by, *out, actual_seq_lengths=sq,
                                     actual_seq_lengths_kv=skv)
        torch.cuda.synchronize()
        nnz = int(out[0][-1].item())
        got = (out[0], out[1][:nnz], out[2], out[3][:nnz])
        assert nnz == ref[1].numel()
        for g, r in zip(got, ref):
            np.testing.assert_array_equal(g.cpu().numpy(), r.cpu().numpy())
        # and directly against the oracle's compaction (brute force on the host)
        oref = O.compact_mask(mask.cpu().numpy(), bx, by, sq, skv)
        for g, r in zip(got, oref):
            np.testing.assert_array_equal(g.cpu().numpy(), r)


def test_noalloc_rejects_masks_beyond_its_scratch():
    # 1.1M query blocks x 1 key block: a 1.1 MB mask whose row counts alone need
    # more than the 4 MiB built-in scratch
    big = torch.ones((1, 1, 1_100_000, 1), dtype=torch.uint8, device=DEV)
    out = _outputs(1, 1, 1, 1)
    with pytest.raises(B.BsaError) as e:
        bsa.bsa_mask_compact_noalloc(big, 64, 64, *out)
    assert e.value.status == B.BSA_ERR_PARAM_INVALID
    assert "scratch" in str(e.value)
