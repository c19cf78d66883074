"""BSA_LOG=1 (environment): the first-stage call prints the plan, the run call
the kernels it launches and bsa_check_status the device work-list counts, one
line each on stderr. Run in a child process so the setting is read fresh; the
active-tile count it reports equals the selected blocks of the mask."""
import os
import re
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import numpy as np, torch
    import block_sparse_attention_attn_gb300 as bsa
    from block_sparse_attention_attn_gb300.workloads import small_workload
    w = small_workload(B=1, N1=2, N2=1, D=128, bx=128, by=128, seq_q=(512,), seq_kv=(512,),
                       p=0.5, seed=83)
    dev = "cuda:0"
    dout, q, k, v = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in w.tensors())
    mask = torch.from_numpy(w.mask).to(dev)
    out, lse, fws = bsa.block_sparse_attention_fwd(q, k, v, block_sparse_mask=mask,
                                                   block_shape=[128, 128], layout="BNSD",
                                                   num_key_value_heads=1, scale_value=w.scale)
    dq, dk, dv, ws = bsa.block_sparse_attention_grad(dout, q, k, v, out, lse,
                                                     block_sparse_mask=mask, block_shape=[128, 128],
                                                     layout="BNSD", num_key_value_heads=1,
                                                     scale_value=w.scale, deterministic=True)
    bsa.bsa_check_status(ws)
    print("EXPECT", int((w.mask[0] != 0).sum()))
""")


def test_bsa_log_lines():
    env = dict(os.environ, BSA_LOG="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    err = r.stderr
    assert re.search(r"\[bsa\] grad plan: layout=BNSD dtype=bf16 B=1 N1=2 N2=1 D=128 Sq=512 "
                     r"Skv=512 block=\[128,128\] tiles q=4 k=4 block_mask=yes", err), err
    assert re.search(r"\[bsa\] grad run: kernel=k_bwd dQ=deterministic", err), err
    expect = int(re.search(r"EXPECT (\d+)", r.stdout).group(1))
    m = re.search(r"\[bsa\] status: active tiles=(\d+) work items=(\d+) .* error=0", err)
    assert m, err
    assert int(m.group(1)) == expect > 0
