"""The bounds-check build (libbsa_checks.so, kernels compiled with
BSA_CHECKS=1, selected with BSA_LIBRARY=checks) on the GPU, in child
processes so the library choice is read fresh:
* on small shapes (GQA, two 64-key blocks per tile with the 64-key-block
  kernel, TND, split columns) the whole outputs match the fp64 oracle and no
  check fails;
* a planted out-of-range list entry (BSA_CHECK_TEST=1, honoured by the bounds-check variant
  only: the fill names a query tile past the last one in column 0) is caught
  by the backward kernel's entry check: the run reports 561002 with check id 2
  (kCheckEntry) in header word 9, nothing faults, and the next run in the same
  process is correct again."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

COMMON = textwrap.dedent("""
    import os, torch
    import block_sparse_attention_attn_gb300 as bsa
    from block_sparse_attention_attn_gb300 import binding as B
    from block_sparse_attention_attn_gb300.workloads import small_workload
    from oracle import bsa_oracle as O
    from tests.harness import check, f64, host_inputs, oracle_forward, rounded_out_lse
    assert B.library_path().endswith("libbsa_checks.so"), B.library_path()
    DEV = "cuda:0"

    def run(w, k64=False):
        dout, q, k, v = host_inputs(w)
        out, lse = oracle_forward(w, q, k, v)
        tout, tlse = rounded_out_lse(w, out, lse)
        g = [t.to(DEV) for t in (dout, q, k, v, tout, tlse)]
        dq, dk, dv = (torch.empty_like(g[i]) for i in (1, 2, 3))
        # the mask must stay allocated until the run has read it (the executor
        # keeps its address, as it keeps every tensor's)
        mask = torch.from_numpy(w.mask).to(DEV)
        size, ex = bsa.bsa_grad_workspace_size(
            *g, mask, None, [w.bx, w.by],
            list(w.seq_q) if w.seq_q is not None else None,
            list(w.seq_kv) if w.seq_kv is not None else None, w.layout, w.layout, w.N2, 0,
            w.scale, dq=dq, dk=dk, dv=dv)
        if k64:
            ex.set_key_block64(True)
        ws = torch.empty(size, dtype=torch.uint8, device=DEV)
        bsa.bsa_grad(ws, size, ex)
        ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(tout), f64(tlse), w.mask,
                         (w.bx, w.by), w.seq_q, w.seq_kv, w.layout, w.N2, w.scale)
        torch.cuda.synchronize()  # the run is done with `mask` and the inputs
        return (dq, dk, dv), ref, ws
""")

CLEAN = COMMON + textwrap.dedent("""
    cases = [
        (small_workload(B=2, N1=4, N2=2, D=128, bx=128, by=128, seq_q=(300, 129),
                        seq_kv=(257, 300), Sq=384, Skv=384, p=0.5, seed=101), False),
        (small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=64, seq_q=(384,), seq_kv=(300,),
                        p=0.6, seed=103), True),
        (small_workload(layout="TND", dtype="f16", B=2, N1=4, N2=4, D=64, bx=64, by=64,
                        seq_q=(200, 65), seq_kv=(130, 190), p=0.5, seed=107), False),
        (small_workload(B=1, N1=256, N2=1, D=64, bx=128, by=128, seq_q=(256,), seq_kv=(128,),
                        p=1.0, dtype="f16", seed=109), False),  # long columns: split
    ]
    for w, k64 in cases:
        got, ref, ws = run(w, k64)
        bsa.bsa_check_status(ws)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            check(f"{w.name}:{name}", f64(a), r)
    print("CLEAN OK")
""")

PLANTED = COMMON + textwrap.dedent("""
    w = small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(384,), seq_kv=(384,),
                       p=1.0, seed=113)
    os.environ["BSA_CHECK_TEST"] = "1"
    got, ref, ws = run(w)
    try:
        bsa.bsa_check_status(ws)
        raise SystemExit("the planted entry was not reported")
    except B.BsaError as e:
        assert e.status == 561002, e.status
        assert "bounds check" in str(e), str(e)
    hdr = ws[:128].view(torch.int32).cpu().tolist()  # header words 0..31
    assert hdr[9] == 2 and hdr[6] == 13 and hdr[16 + 13] > 0, hdr
    del os.environ["BSA_CHECK_TEST"]
    got, ref, ws = run(w)
    bsa.bsa_check_status(ws)
    for name, a, r in zip(("dq", "dk", "dv"), got, ref):
        check(name, f64(a), r)
    print("PLANTED OK")
""")


@pytest.fixture(scope="module")
def checks_lib():
    from block_sparse_attention_attn_gb300 import build
    return build.build(checks=True)


@pytest.mark.parametrize("script,marker", [(CLEAN, "CLEAN OK"), (PLANTED, "PLANTED OK")],
                         ids=["clean", "planted_entry"])
def test_checks_build(checks_lib, script, marker):
    env = dict(os.environ, BSA_LIBRARY="checks", PYTHONPATH=ROOT)
    env.pop("BSA_CHECK_TEST", None)
    r = subprocess.run([sys.executable, "-c", script], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and marker in r.stdout, (r.stdout[-2000:], r.stderr[-3000:])
