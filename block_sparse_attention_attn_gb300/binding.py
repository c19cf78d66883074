"""ctypes binding of libbsa (include/bsa.h): argument marshalling only.

Every function named like a C entry point takes torch tensors (device memory
owned by the caller), builds the ``bsa_tensor`` descriptors and calls the
library; all computation happens in the library's CUDA kernels. If the library
has not been built, every call raises :class:`BsaError` (there is no fallback).
"""
from __future__ import annotations

import collections
import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# BSA_LIBRARY=checks selects the bounds-check build (libbsa_checks.so, built by
# `python -m block_sparse_attention_attn_gb300.build --checks`)
_LIB_PATH = os.path.join(_HERE, "lib", "libbsa_checks.so" if os.environ.get("BSA_LIBRARY") == "checks"
                         else "libbsa.so")
_lib = None

BSA_OK = 0
BSA_ERR_PARAM_NULLPTR = 161001
BSA_ERR_PARAM_INVALID = 161002
BSA_ERR_RUNTIME = 361001
NO_WINDOW = 2147483647   # preTokens / nextTokens value meaning "no sliding window"
BSA_ERR_INNER = 561002

_DTYPES = {torch.float16: 1, torch.bfloat16: 2, torch.float32: 3, torch.uint8: 4, torch.bool: 4}


class BsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libbsa status {status}: {message}")
        self.status = status


class BsaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads libbsa.so (once). Raises BsaError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise BsaError(BSA_ERR_RUNTIME, f"{_LIB_PATH} not built; run "
                       "`python -m block_sparse_attention_attn_gb300.build`"
                       + (" --checks" if _LIB_PATH.endswith("_checks.so") else ""))
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER
    T = P(BsaTensor)
    i64, u64, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
    lib.bsa_grad_workspace_size.argtypes = [
        T, T, T, T, T, T, T, T, P(i64), i64, P(i64), i64, P(i64), i64, ctypes.c_char_p,
        ctypes.c_char_p, i64, i64, ctypes.c_double, i64, i64, T, T, T, P(u64), P(vp)]
    lib.bsa_grad.argtypes = [vp, u64, vp, vp]
    lib.bsa_fwd_workspace_size.argtypes = [
        T, T, T, T, T, P(i64), i64, P(i64), i64, P(i64), i64, ctypes.c_char_p, ctypes.c_char_p,
        i64, i64, ctypes.c_double, i64, i64, T, T, P(u64), P(vp)]
    lib.bsa_fwd.argtypes = [vp, u64, vp, vp]
    lib.bsa_executor_destroy.argtypes = [vp]
    lib.bsa_executor_set_timing_events.argtypes = [vp, vp, vp]
    lib.bsa_executor_set_wait_test.argtypes = [vp, ctypes.c_int32]
    lib.bsa_executor_set_deterministic.argtypes = [vp, ctypes.c_int32]
    lib.bsa_executor_set_key_block64.argtypes = [vp, ctypes.c_int32]
    lib.bsa_mask_compact_workspace_size.argtypes = [T, i64, i64, P(u64)]
    lib.bsa_mask_compact.argtypes = [T, i64, i64, P(i64), i64, P(i64), i64, vp, vp, vp, vp, vp,
                                     u64, vp]
    lib.bsa_mask_compact_noalloc.argtypes = [T, i64, i64, P(i64), i64, P(i64), i64, vp, vp, vp,
                                             vp, vp]
    lib.bsa_check_status.argtypes = [vp, vp]
    lib.bsa_status_async.argtypes = [vp, vp, vp]
    lib.bsa_last_error.restype = ctypes.c_char_p
    lib.bsa_version.restype = ctypes.c_int32
    for name in ("bsa_grad_workspace_size", "bsa_grad", "bsa_fwd_workspace_size", "bsa_fwd",
                 "bsa_executor_destroy", "bsa_executor_set_timing_events",
                 "bsa_executor_set_wait_test", "bsa_executor_set_deterministic",
                 "bsa_executor_set_key_block64",
                 "bsa_mask_compact_workspace_size", "bsa_mask_compact",
                 "bsa_mask_compact_noalloc", "bsa_check_status", "bsa_status_async"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status != BSA_OK:
        raise BsaError(status, load_library().bsa_last_error().decode())


def _desc(t: Optional[torch.Tensor]):
    if t is None:
        return None
    d = BsaTensor()
    d.data = t.data_ptr()
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return ctypes.byref(d), d


def _ptr(x):
    return None if x is None else x[0]


def _i64_array(v: Optional[Sequence[int]]):
    if v is None:
        return None, 0
    arr = (ctypes.c_int64 * len(v))(*[int(a) for a in v])
    return arr, len(v)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class Executor:
    """Owns a C executor until a run call consumes it."""

    def __init__(self, handle: int, keep):
        self.handle = handle
        self._keep = keep   # the descriptors' tensors must outlive the run

    def take(self) -> int:
        h, self.handle = self.handle, None
        if h is None:
            raise BsaError(BSA_ERR_PARAM_NULLPTR, "executor already consumed")
        return h

    def set_timing_events(self, before, after):
        """Records torch.cuda.Event `before`/`after` around the main kernel."""
        lib = load_library()
        _check(lib.bsa_executor_set_timing_events(
            self.handle, None if before is None else before.cuda_event,
            None if after is None else after.cuda_event))

    def set_wait_test(self, enable: bool = True):
        """Failure-path test: the run's backward kernel waits once on a barrier
        nothing completes; bsa_check_status then reports 561002."""
        _check(load_library().bsa_executor_set_wait_test(self.handle, 1 if enable else 0))

    def set_deterministic(self, enable: bool = True):
        """dQ from a separate query-tile pass: bitwise identical results on
        every run (backward executors only)."""
        _check(load_library().bsa_executor_set_deterministic(self.handle, 1 if enable else 0))

    def set_key_block64(self, enable: bool = True):
        """blockShape [bx, 64], D = 128, no window or token mask: one
        query-major step per selected 64-key block (backward executors only;
        ignored otherwise)."""
        _check(load_library().bsa_executor_set_key_block64(self.handle, 1 if enable else 0))

    def __del__(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.bsa_executor_destroy(self.handle)


def bsa_grad_workspace_size(dout, query, key, value, attention_out, softmax_lse,
                            block_sparse_mask=None, atten_mask=None, block_shape=None,
                            actual_seq_lengths=None, actual_seq_lengths_kv=None,
                            q_layout="BNSD", kv_layout=None, num_key_value_heads=None,
                            mask_type=0, scale_value=1.0, pre_tokens=NO_WINDOW,
                            next_tokens=NO_WINDOW, dq=None, dk=None, dv=None):
    """First stage of the backward. Returns (workspace_size, Executor)."""
    lib = load_library()
    kv_layout = q_layout if kv_layout is None else kv_layout
    if num_key_value_heads is None:
        num_key_value_heads = key.shape[1]
    ds = [_desc(t) for t in (dout, query, key, value, attention_out, softmax_lse,
                             block_sparse_mask, atten_mask, dq, dk, dv)]
    bs, nbs = _i64_array(block_shape)
    sq, nsq = _i64_array(actual_seq_lengths)
    sk, nsk = _i64_array(actual_seq_lengths_kv)
    ws = ctypes.c_uint64(0)
    ex = ctypes.c_void_p(None)
    _check(lib.bsa_grad_workspace_size(
        *[_ptr(d) for d in ds[:8]], bs, nbs, sq, nsq, sk, nsk, q_layout.encode(),
        kv_layout.encode(), int(num_key_value_heads), int(mask_type), float(scale_value),
        int(pre_tokens), int(next_tokens), *[_ptr(d) for d in ds[8:]], ctypes.byref(ws),
        ctypes.byref(ex)))
    return ws.value, Executor(ex.value, ds)


def bsa_grad(workspace: torch.Tensor, workspace_size: int, executor: Executor, stream=None):
    """Second stage of the backward; asynchronous on `stream` (default: current)."""
    lib = load_library()
    _check(lib.bsa_grad(workspace.data_ptr(), int(workspace_size), executor.take(),
                        _stream(stream)))


def bsa_fwd_workspace_size(query, key, value, block_sparse_mask=None, block_shape=None,
                           actual_seq_lengths=None, actual_seq_lengths_kv=None,
                           q_layout="BNSD", kv_layout=None, num_key_value_heads=None,
                           scale_value=1.0, pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW,
                           attention_out=None, softmax_lse=None, atten_mask=None,
                           mask_type=None):
    lib = load_library()
    kv_layout = q_layout if kv_layout is None else kv_layout
    if num_key_value_heads is None:
        num_key_value_heads = key.shape[1]
    if mask_type is None:
        mask_type = 0 if atten_mask is None else 1
    ds = [_desc(t) for t in (query, key, value, block_sparse_mask, attention_out, softmax_lse,
                             atten_mask)]
    bs, nbs = _i64_array(block_shape)
    sq, nsq = _i64_array(actual_seq_lengths)
    sk, nsk = _i64_array(actual_seq_lengths_kv)
    ws = ctypes.c_uint64(0)
    ex = ctypes.c_void_p(None)
    _check(lib.bsa_fwd_workspace_size(
        _ptr(ds[0]), _ptr(ds[1]), _ptr(ds[2]), _ptr(ds[3]), _ptr(ds[6]), bs, nbs, sq, nsq, sk,
        nsk, q_layout.encode(), kv_layout.encode(), int(num_key_value_heads), int(mask_type),
        float(scale_value), int(pre_tokens), int(next_tokens), _ptr(ds[4]), _ptr(ds[5]),
        ctypes.byref(ws), ctypes.byref(ex)))
    return ws.value, Executor(ex.value, ds)


def bsa_fwd(workspace: torch.Tensor, workspace_size: int, executor: Executor, stream=None):
    lib = load_library()
    _check(lib.bsa_fwd(workspace.data_ptr(), int(workspace_size), executor.take(), _stream(stream)))


def bsa_check_status(workspace: torch.Tensor, stream=None):
    lib = load_library()
    _check(lib.bsa_check_status(workspace.data_ptr(), _stream(stream)))


class _PendingStatus:
    """Error words of recent runs, read without a host synchronization: each
    run enqueues a copy of its workspace's error words into a slot of a
    page-locked ring (bsa_status_async) and records an event; `poll` inspects
    the copies whose event has completed and raises on a failed run. The
    workspace stays referenced until its words have been read. The ring is
    allocated once (`reserve`, called by the autograd forward), since a
    page-locked allocation may itself wait for the device."""

    SLOTS = 64

    def __init__(self):
        self.pending = collections.deque()
        self.words = None
        self.next = 0

    def reserve(self):
        if self.words is None:
            self.words = torch.zeros((self.SLOTS, 8), dtype=torch.int32, pin_memory=True)

    def push(self, workspace: torch.Tensor):
        """After a run on the current stream."""
        self.reserve()
        while len(self.pending) >= self.SLOTS:   # slots are reused in FIFO order
            self._pop(block=True)
        slot = self.next
        self.next = (slot + 1) % self.SLOTS
        words = self.words[slot]
        words.zero_()
        stream = torch.cuda.current_stream()
        _check(load_library().bsa_status_async(workspace.data_ptr(), words.data_ptr(),
                                               stream.cuda_stream))
        ev = torch.cuda.Event()
        ev.record(stream)
        self.pending.append((words, ev, workspace))

    def _pop(self, block: bool) -> bool:
        words, ev, _ = self.pending[0]
        if block:
            ev.synchronize()
        elif not ev.query():
            return False
        self.pending.popleft()
        if int(words[0]) != 0:
            raise BsaError(BSA_ERR_INNER, "a kernel of an earlier backward gave up a bounded "
                                          f"wait (code {int(words[6])})")
        return True

    def poll(self, block: bool = False):
        while self.pending and self._pop(block):
            pass


_PENDING = _PendingStatus()


def check_pending_status(block: bool = True):
    """Raises BsaError if any backward run by the autograd function since the
    last check failed (block=True waits for all of them; False inspects only
    those that have finished)."""
    _PENDING.poll(block)


def bsa_mask_compact(mask: torch.Tensor, bx: int, by: int, actual_seq_lengths=None,
                     actual_seq_lengths_kv=None, stream=None):
    """Block-level CSR/CSC of a block mask: (row_ptr, col_idx, col_ptr, row_idx),
    int32 device tensors; col_idx/row_idx trimmed to nnz."""
    lib = load_library()
    B, N, Mq, Mk = mask.shape
    d = _desc(mask)
    need = ctypes.c_uint64(0)
    _check(lib.bsa_mask_compact_workspace_size(d[0], int(bx), int(by), ctypes.byref(need)))
    dev = mask.device
    ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=dev)
    row_ptr = torch.empty(B * N * (Mq + 1), dtype=torch.int32, device=dev)
    col_ptr = torch.empty(B * N * (Mk + 1), dtype=torch.int32, device=dev)
    col_idx = torch.empty(max(B * N * Mq * Mk, 1), dtype=torch.int32, device=dev)
    row_idx = torch.empty(max(B * N * Mq * Mk, 1), dtype=torch.int32, device=dev)
    sq, nsq = _i64_array(actual_seq_lengths)
    sk, nsk = _i64_array(actual_seq_lengths_kv)
    _check(lib.bsa_mask_compact(d[0], int(bx), int(by), sq, nsq, sk, nsk, row_ptr.data_ptr(),
                                col_idx.data_ptr(), col_ptr.data_ptr(), row_idx.data_ptr(),
                                ws.data_ptr(), int(need.value), _stream(stream)))
    torch.cuda.synchronize(dev)
    nnz = int(row_ptr[-1].item())
    return row_ptr, col_idx[:nnz], col_ptr, row_idx[:nnz]


def bsa_mask_compact_noalloc(mask: torch.Tensor, bx: int, by: int, row_ptr, col_idx, col_ptr,
                             row_idx, actual_seq_lengths=None, actual_seq_lengths_kv=None,
                             stream=None):
    """The allocation-free compaction: writes the CSR/CSC into the given int32
    device tensors (col_idx/row_idx sized for the dense bound) using only the
    library's built-in scratch array. For callers that cannot allocate device
    memory; calls that overlap on the GPU race on the shared scratch."""
    lib = load_library()
    d = _desc(mask)
    sq, nsq = _i64_array(actual_seq_lengths)
    sk, nsk = _i64_array(actual_seq_lengths_kv)
    _check(lib.bsa_mask_compact_noalloc(d[0], int(bx), int(by), sq, nsq, sk, nsk,
                                        row_ptr.data_ptr(), col_idx.data_ptr(),
                                        col_ptr.data_ptr(), row_idx.data_ptr(), _stream(stream)))


def block_sparse_attention_grad(dout, query, key, value, attention_out, softmax_lse,
                                block_sparse_mask=None, block_shape=None,
                                actual_seq_lengths=None, actual_seq_lengths_kv=None,
                                layout="BNSD", num_key_value_heads=None, scale_value=None,
                                dq=None, dk=None, dv=None, workspace=None, stream=None,
                                deterministic=False, pre_tokens=NO_WINDOW,
                                next_tokens=NO_WINDOW, atten_mask=None):
    """Both stages; allocates outputs/workspace with torch when not given.
    pre_tokens / next_tokens: sliding window (query s and key t of a sequence
    pair up iff s - pre_tokens <= t <= s + next_tokens; next_tokens=0 is
    causal). atten_mask: optional 2-D bool/uint8 [>= maxSq, >= maxSkv] token
    mask, True = masked (maskType 1). Returns (dq, dk, dv, workspace)."""
    if scale_value is None:
        scale_value = query.shape[-1] ** -0.5
    dq = torch.empty_like(query) if dq is None else dq
    dk = torch.empty_like(key) if dk is None else dk
    dv = torch.empty_like(value) if dv is None else dv
    size, ex = bsa_grad_workspace_size(
        dout, query, key, value, attention_out, softmax_lse, block_sparse_mask, atten_mask,
        block_shape, actual_seq_lengths, actual_seq_lengths_kv, layout, layout,
        num_key_value_heads, 0 if atten_mask is None else 1, scale_value, pre_tokens,
        next_tokens, dq=dq, dk=dk, dv=dv)
    if deterministic:
        ex.set_deterministic(True)
    if workspace is None or workspace.numel() < size:
        workspace = torch.empty(max(size, 256), dtype=torch.uint8, device=query.device)
    bsa_grad(workspace, size, ex, stream)
    return dq, dk, dv, workspace


def block_sparse_attention_fwd(query, key, value, block_sparse_mask=None, block_shape=None,
                               actual_seq_lengths=None, actual_seq_lengths_kv=None,
                               layout="BNSD", num_key_value_heads=None, scale_value=None,
                               out=None, lse=None, workspace=None, stream=None,
                               pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW, atten_mask=None):
    """Companion forward (same sliding window arguments as the backward);
    returns (out, lse [..., 1] fp32, workspace)."""
    if scale_value is None:
        scale_value = query.shape[-1] ** -0.5
    out = torch.empty_like(query) if out is None else out
    if lse is None:
        lse = torch.empty((*query.shape[:-1], 1), dtype=torch.float32, device=query.device)
    size, ex = bsa_fwd_workspace_size(query, key, value, block_sparse_mask, block_shape,
                                      actual_seq_lengths, actual_seq_lengths_kv, layout, layout,
                                      num_key_value_heads, scale_value, pre_tokens,
                                      next_tokens, out, lse, atten_mask)
    if workspace is None or workspace.numel() < size:
        workspace = torch.empty(max(size, 256), dtype=torch.uint8, device=query.device)
    bsa_fwd(workspace, size, ex, stream)
    return out, lse, workspace


class BlockSparseAttentionFunction(torch.autograd.Function):
    """Autograd pairing of the companion forward (Out, lse) and the backward:
    forward runs bsa_fwd, backward runs bsa_grad on the saved Q, K, V, Out and
    lse (the page's call sequence, with PyTorch driving it). The mask, block
    shape, lengths and options are not differentiable. Neither direction
    synchronizes the host: a backward run's error words are copied
    asynchronously and checked by later calls or by check_pending_status()."""

    @staticmethod
    def forward(ctx, query, key, value, block_sparse_mask, block_shape, actual_seq_lengths,
                actual_seq_lengths_kv, layout, num_key_value_heads, scale_value, deterministic,
                pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW, atten_mask=None):
        _PENDING.reserve()
        _PENDING.poll()   # failures of earlier backward runs surface here, without a sync
        if scale_value is None:
            scale_value = query.shape[-1] ** -0.5
        query, key, value = query.contiguous(), key.contiguous(), value.contiguous()
        out, lse, _ = block_sparse_attention_fwd(
            query, key, value, block_sparse_mask, block_shape, actual_seq_lengths,
            actual_seq_lengths_kv, layout, num_key_value_heads, scale_value,
            pre_tokens=pre_tokens, next_tokens=next_tokens, atten_mask=atten_mask)
        ctx.save_for_backward(query, key, value, out, lse)
        ctx.mask = block_sparse_mask
        ctx.atten_mask = atten_mask
        ctx.args = (block_shape, actual_seq_lengths, actual_seq_lengths_kv, layout,
                    num_key_value_heads, scale_value, deterministic, pre_tokens, next_tokens)
        return out

    @staticmethod
    def backward(ctx, dout):
        query, key, value, out, lse = ctx.saved_tensors
        (block_shape, actual_seq_lengths, actual_seq_lengths_kv, layout, num_key_value_heads,
         scale_value, deterministic, pre_tokens, next_tokens) = ctx.args
        dq, dk, dv, ws = block_sparse_attention_grad(
            dout.contiguous(), query, key, value, out, lse, ctx.mask, block_shape,
            actual_seq_lengths, actual_seq_lengths_kv, layout, num_key_value_heads, scale_value,
            deterministic=deterministic, pre_tokens=pre_tokens, next_tokens=next_tokens,
            atten_mask=ctx.atten_mask)
        # no host synchronization here: the run's error words are read later
        # (next forward, or check_pending_status())
        _PENDING.poll()
        _PENDING.push(ws)
        return dq, dk, dv, None, None, None, None, None, None, None, None, None, None, None


def block_sparse_attention(query, key, value, block_sparse_mask=None, block_shape=None,
                           actual_seq_lengths=None, actual_seq_lengths_kv=None, layout="BNSD",
                           num_key_value_heads=None, scale_value=None, deterministic=False,
                           pre_tokens=NO_WINDOW, next_tokens=NO_WINDOW, atten_mask=None):
    """Differentiable block-sparse attention: Out = softmax(scale*Q K^T over the
    selected blocks, inside the sliding window) V; gradients for Q, K and V come
    from the backward kernels."""
    return BlockSparseAttentionFunction.apply(
        query, key, value, block_sparse_mask, block_shape, actual_seq_lengths,
        actual_seq_lengths_kv, layout, num_key_value_heads, scale_value, deterministic,
        pre_tokens, next_tokens, atten_mask)
