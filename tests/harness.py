"""Shared helpers of the parity tests: seeded inputs (from the workload
generators), the oracle's forward for attentionOut / softmaxLse, and the
tolerance check (per element |err| <= 1e-2 + 2e-2*|ref|, relative Frobenius
error <= 5e-3)."""
import numpy as np
import torch

from oracle import bsa_oracle as O

ATOL, RTOL, FRO = 1e-2, 2e-2, 5e-3
TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16}


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def host_inputs(w, pad_fill=None):
    """(dout, q, k, v) rounded to the workload dtype (CPU torch tensors). With
    ``pad_fill`` the BNSD padding rows (past the actual lengths) hold that value."""
    dt = TORCH_DT[w.dtype]
    ts = [torch.from_numpy(x).to(dt) for x in w.tensors()]
    if pad_fill is not None and w.layout == "BNSD":
        dout, q, k, v = ts
        for b in range(w.B):
            for t in (dout, q):
                t[b, :, w.seq_q[b]:] = pad_fill
            for t in (k, v):
                t[b, :, w.seq_kv[b]:] = pad_fill
    return ts


def oracle_forward(w, q, k, v, blockrows=False, **window):
    """The oracle's (out, lse); ``window``: pre_tokens / next_tokens."""
    fn = O.forward_blockrows if blockrows else O.forward
    out, lse = fn(f64(q), f64(k), f64(v), w.mask, (w.bx, w.by), w.seq_q, w.seq_kv, w.layout,
                  w.N2, w.scale, **window)
    return out, lse


def rounded_out_lse(w, out, lse, pad_fill=None):
    dt = TORCH_DT[w.dtype]
    tout = torch.from_numpy(out).to(dt)
    tlse = torch.from_numpy(lse).to(torch.float32)
    if pad_fill is not None and w.layout == "BNSD":
        for b in range(w.B):
            tout[b, :, w.seq_q[b]:] = pad_fill
            tlse[b, :, w.seq_q[b]:] = pad_fill
    return tout, tlse


def check(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (ATOL + RTOL * np.abs(ref))), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r}")
    nr = np.linalg.norm(ref)
    fro = np.linalg.norm(got - ref) / nr if nr > 0 else np.linalg.norm(got)
    assert fro <= FRO, f"{name}: relative Frobenius error {fro:.3e}"
    return float(err.max()), float(fro)


def oracle_backward_whole(w, dout, q, k, v, tout, tlse, mask="workload", **window):
    """The oracle's whole dQ, dK, dV (block-row evaluation over the selected
    keys), fed the same Out / lse bytes the GPU backward consumes."""
    m = w.mask if isinstance(mask, str) else mask
    return O.backward_blockrows(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), m,
                                (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale,
                                **window)


def check_whole(name, got, ref):
    """Element-wise and relative-Frobenius check of whole output tensors."""
    for part, g, r in zip(("dq", "dk", "dv"), got, ref):
        check(f"{name}:{part}", f64(g) if isinstance(g, torch.Tensor) else g, r)
