"""The autograd pairing runs without host synchronizations: several layers of
forward + backward are enqueued behind a long GPU sleep and the host returns
from backward() while the GPU is still busy; a failed run still surfaces,
through the asynchronously copied error words."""
import pytest
import torch

import block_sparse_attention_attn_gb300 as bsa
from block_sparse_attention_attn_gb300 import binding
from block_sparse_attention_attn_gb300.workloads import small_workload
from oracle import bsa_oracle as O
from tests.harness import check, f64, host_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_multi_layer_backward_does_not_sync():
    w = small_workload(layout="BNSD", dtype="bf16", B=1, N1=2, N2=1, D=128, bx=128, by=128,
                       seq_q=(384,), seq_kv=(384,), p=0.7, seed=51)
    dout, q, k, v = host_inputs(w)
    mask = torch.from_numpy(w.mask).to(DEV)
    layers = 4

    def step():
        qs = [q.to(DEV).requires_grad_(True) for _ in range(layers)]
        kd, vd = k.to(DEV).requires_grad_(True), v.to(DEV).requires_grad_(True)
        outs = [bsa.block_sparse_attention(x, kd, vd, block_sparse_mask=mask,
                                           block_shape=[128, 128], num_key_value_heads=w.N2,
                                           scale_value=w.scale)
                for x in qs]
        loss = sum((o.float() * dout.to(DEV).float()).sum() for o in outs)
        return qs, kd, vd, outs, loss
    # one warm-up step: first-use set-up (device and page-locked allocations,
    # the library's side stream) may wait for the device
    step()[-1].backward()
    bsa.check_pending_status()
    qs, kd, vd, outs, loss = step()
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000_000)     # ~1 s of GPU time ahead of the backward
    loss.backward()
    busy = not torch.cuda.current_stream().query()
    bsa.check_pending_status()           # waits for the runs and reads their words
    assert busy, "backward() waited for the GPU"
    # gradients against the oracle fed the Out / lse the backward used (every
    # layer has the same inputs; the forward is deterministic)
    fo, flse, fws = bsa.block_sparse_attention_fwd(
        q.to(DEV), k.to(DEV), v.to(DEV), block_sparse_mask=mask, block_shape=[128, 128],
        num_key_value_heads=1, scale_value=w.scale)
    bsa.bsa_check_status(fws)
    assert torch.equal(fo, outs[0].detach())
    ref = O.backward(f64(dout), f64(q), f64(k), f64(v), f64(fo), f64(flse), w.mask, (128, 128),
                     num_kv_heads=1, scale=w.scale)
    for x in qs:
        check("nosync:dq", f64(x.grad), ref[0])
    check("nosync:dk", f64(kd.grad) / layers, ref[1])
    check("nosync:dv", f64(vd.grad) / layers, ref[2])


def test_failed_run_surfaces_later():
    """A workspace whose error word is set (as a kernel that gave up a wait
    leaves it) is reported by the next poll, not at enqueue time."""
    ws = torch.zeros(64, dtype=torch.int32, device=DEV)
    ws[0] = 1
    ws[6] = 12
    binding._PENDING.push(ws.view(torch.uint8))
    with pytest.raises(bsa.BsaError) as err:
        bsa.check_pending_status()
    assert err.value.status == binding.BSA_ERR_INNER and "code 12" in str(err.value)
    bsa.check_pending_status()           # reported once, then cleared
