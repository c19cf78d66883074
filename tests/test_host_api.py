"""CPU-only checks of the C ABI: the library loads without a GPU, exports every
symbol include/bsa.h declares, and the first-stage calls return the page's
status codes (161001 / 161002) for invalid arguments. The first stage never
dereferences tensor data, so CPU tensors stand in for device tensors here."""
import os
import re

import pytest
import torch

import block_sparse_attention_attn_gb300 as bsa
from block_sparse_attention_attn_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_attn_gb300 import build
    build.build()
    return bsa.load_library()


def test_exports_every_declared_symbol(lib):
    with open(os.path.join(ROOT, "include", "bsa.h")) as f:
        hdr = f.read()
    names = set(re.findall(r"^\s*(?:bsa_status|const char\*|int32_t)\s+(bsa_\w+)\s*\(", hdr, re.M))
    assert len(names) >= 10, names
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert lib.bsa_version() >= 100


def test_checks_build_exports_every_declared_symbol():
    """The bounds-check variant (kernels compiled with BSA_CHECKS=1) builds and
    exports the same C ABI."""
    import ctypes
    from block_sparse_attention_attn_gb300 import build
    path = build.build(checks=True)
    assert path.endswith("libbsa_checks.so")
    chk = ctypes.CDLL(path)
    with open(os.path.join(ROOT, "include", "bsa.h")) as f:
        names = set(re.findall(r"^\s*(?:bsa_status|const char\*|int32_t)\s+(bsa_\w+)\s*\(", f.read(), re.M))
    for n in sorted(names):
        assert hasattr(chk, n), n
    assert chk.bsa_version() >= 100


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def _grad_args(layout="BNSD", B_=1, N1=2, N2=1, S=256, D=128, dtype=torch.bfloat16, mask=True):
    if layout == "BNSD":
        q, kk = _t(B_, N1, S, D, dtype=dtype), _t(B_, N2, S, D, dtype=dtype)
        lse = _t(B_, N1, S, 1, dtype=torch.float32)
    else:
        q, kk = _t(S, N1, D, dtype=dtype), _t(S, N2, D, dtype=dtype)
        lse = _t(S, N1, 1, dtype=torch.float32)
    m = torch.ones(B_, N1, 2, 2, dtype=torch.uint8) if mask else None
    return dict(dout=q.clone(), query=q, key=kk, value=kk.clone(), attention_out=q.clone(),
                softmax_lse=lse, block_sparse_mask=m, block_shape=[128, 128], q_layout=layout,
                num_key_value_heads=N2, scale_value=D ** -0.5, dq=q.clone(), dk=kk.clone(),
                dv=kk.clone())


def _status(**kw):
    try:
        bsa.bsa_grad_workspace_size(**kw)
    except B.BsaError as e:
        return e.status
    return 0


def test_valid_arguments_reach_the_device_query(lib):
    st = _status(**_grad_args())
    # with a GPU the call succeeds; without one it fails only at the device query
    assert st == (0 if torch.cuda.is_available() else B.BSA_ERR_RUNTIME)


@pytest.mark.parametrize("pre,nxt", [(1024, 0), (-3, 5), (7, -7), (2 ** 63 - 1, 2 ** 63 - 1),
                                     (0, 0)])
def test_windows_that_overlap_the_diagonal_are_accepted(lib, pre, nxt):
    st = _status(**_grad_args(), pre_tokens=pre, next_tokens=nxt)
    assert st == (0 if torch.cuda.is_available() else B.BSA_ERR_RUNTIME)


def test_atten_mask_with_mask_type_1_is_accepted(lib):
    kw = _grad_args()
    kw.update(atten_mask=torch.zeros(300, 260, dtype=torch.bool), mask_type=1)
    assert _status(**kw) == (0 if torch.cuda.is_available() else B.BSA_ERR_RUNTIME)


@pytest.mark.parametrize("am,mt", [
    (torch.zeros(256, 256, dtype=torch.uint8), 0),        # a mask needs maskType 1
    (None, 1),                                            # maskType 1 needs a mask
    (torch.zeros(256, 256, dtype=torch.uint8), 2),        # unknown maskType
    (torch.zeros(1, 256, 256, dtype=torch.uint8), 1),     # not 2-D
    (torch.zeros(255, 256, dtype=torch.uint8), 1),        # smaller than [maxSq, maxSkv]
    (torch.zeros(256, 256, dtype=torch.float16), 1),      # not BOOL/UINT8
])
def test_invalid_atten_mask(lib, am, mt):
    kw = _grad_args()
    kw.update(atten_mask=am, mask_type=mt)
    assert _status(**kw) == B.BSA_ERR_PARAM_INVALID


def test_null_required_tensors(lib):
    for name in ("dout", "query", "key", "value", "attention_out"):
        kw = _grad_args()
        kw[name] = None
        assert _status(**kw) == B.BSA_ERR_PARAM_NULLPTR, name


def test_tnd_without_lengths_is_nullptr(lib):
    kw = _grad_args(layout="TND")
    assert _status(**kw) == B.BSA_ERR_PARAM_NULLPTR


@pytest.mark.parametrize("change", [
    dict(q_layout="BSND"), dict(kv_layout="TND"), dict(mask_type=1),
    dict(pre_tokens=-5, next_tokens=4), dict(pre_tokens=3, next_tokens=-10),
    dict(pre_tokens=-(2 ** 63), next_tokens=2 ** 63 - 1), dict(block_shape=[128]),
    dict(block_shape=[0, 128]), dict(block_shape=[96, 128]), dict(num_key_value_heads=3),
])
def test_invalid_scalars(lib, change):
    kw = _grad_args()
    kw.update(change)
    assert _status(**kw) == B.BSA_ERR_PARAM_INVALID, change


def test_invalid_tensors(lib):
    cases = []
    kw = _grad_args(); kw["key"] = _t(1, 1, 256, 128, dtype=torch.float16); cases.append(kw)
    kw = _grad_args(D=96); cases.append(kw)
    kw = _grad_args(N1=3, N2=2); cases.append(kw)
    kw = _grad_args(); kw["softmax_lse"] = _t(1, 2, 256, 1); cases.append(kw)      # bf16 lse
    kw = _grad_args(); kw["query"] = _t(1, 2, 128, 256).transpose(2, 3); cases.append(kw)
    kw = _grad_args(); kw["block_sparse_mask"] = torch.ones(1, 2, 3, 2, dtype=torch.uint8); cases.append(kw)
    kw = _grad_args(); kw["atten_mask"] = torch.ones(256, 256, dtype=torch.uint8); cases.append(kw)
    kw = _grad_args(); kw["dq"] = _t(1, 2, 256, 64); cases.append(kw)
    kw = _grad_args(S=0); cases.append(kw)
    for i, c in enumerate(cases):
        assert _status(**c) == B.BSA_ERR_PARAM_INVALID, i


def test_tnd_length_sum_must_match(lib):
    kw = _grad_args(layout="TND", S=300, mask=False)
    kw.update(actual_seq_lengths=[100, 150], actual_seq_lengths_kv=[100, 200])
    assert _status(**kw) == B.BSA_ERR_PARAM_INVALID


def test_run_call_rejects_null_executor(lib):
    assert lib.bsa_grad(None, 0, None, None) == B.BSA_ERR_PARAM_NULLPTR
    assert lib.bsa_fwd(None, 0, None, None) == B.BSA_ERR_PARAM_NULLPTR
    assert "executor" in lib.bsa_last_error().decode()
    assert lib.bsa_executor_destroy(None) == 0


def test_wait_test_switch_needs_an_executor(lib):
    assert lib.bsa_executor_set_wait_test(None, 1) == B.BSA_ERR_PARAM_NULLPTR


def test_deterministic_switch_needs_a_backward_executor(lib):
    assert lib.bsa_executor_set_deterministic(None, 1) == B.BSA_ERR_PARAM_NULLPTR


def test_key_block64_switch_needs_a_backward_executor(lib):
    assert lib.bsa_executor_set_key_block64(None, 1) == B.BSA_ERR_PARAM_NULLPTR


def _fwd_status(**kw):
    try:
        bsa.bsa_fwd_workspace_size(**kw)
    except B.BsaError as e:
        return e.status
    return 0


def _fwd_args():
    g = _grad_args()
    return dict(query=g["query"], key=g["key"], value=g["value"],
                block_sparse_mask=g["block_sparse_mask"], block_shape=[128, 128],
                num_key_value_heads=1, scale_value=g["scale_value"],
                attention_out=g["attention_out"], softmax_lse=g["softmax_lse"])


def test_forward_first_stage_validation(lib):
    ok = 0 if torch.cuda.is_available() else B.BSA_ERR_RUNTIME
    assert _fwd_status(**_fwd_args()) == ok
    assert _fwd_status(**_fwd_args(), pre_tokens=100, next_tokens=0) == ok
    assert _fwd_status(**_fwd_args(), atten_mask=torch.zeros(256, 256, dtype=torch.bool)) == ok
    bad = [dict(pre_tokens=-3, next_tokens=2),
           dict(atten_mask=torch.zeros(256, 256, dtype=torch.uint8), mask_type=0),
           dict(mask_type=1),
           dict(atten_mask=torch.zeros(200, 256, dtype=torch.uint8)),
           dict(block_shape=[32, 128])]
    for extra in bad:
        kw = _fwd_args()
        kw.update(extra)
        assert _fwd_status(**kw) == B.BSA_ERR_PARAM_INVALID, extra
    kw = _fwd_args()
    kw["softmax_lse"] = None
    assert _fwd_status(**kw) == B.BSA_ERR_PARAM_NULLPTR
