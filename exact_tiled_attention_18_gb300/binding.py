"""ctypes binding of libfa.so: the C ABI of include/fa.h, name for name.

Argument marshalling only -- every step of the computation runs in the CUDA
kernels behind these calls.  There is no fallback: if the library was not
built (``python -m exact_tiled_attention_18_gb300.build``) every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED_D = 2
FA_ERR_MISALIGNED = 3
FA_ERR_LAUNCH = 4
FA_ERR_TIMEOUT = 5
FA_ERR_DEVICE_FAULT = 6
FA_DECODE_MAX_Q = 8
FA_DTYPE_F32 = 0
FA_DTYPE_BF16 = 1

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    """A library call returned a status other than FA_OK."""

    def __init__(self, call: str, status: int, text: str):
        super().__init__(f"{call}: {text}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libfa.so once; raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise FileNotFoundError(
                f"{LIB_PATH} is missing: build it with `python -m exact_tiled_attention_18_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int
        ll = ctypes.c_longlong
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd.restype = st
        L.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_fwd_varlen.restype = st
        L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_fwd_ex.restype = st
        L.fa_fwd_bias.argtypes = [vp, vp, vp, vp, i, vp, vp, ll, ll, ll, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_fwd_bias.restype = st
        L.fa_bwd_ex.argtypes = [vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_bwd_ex.restype = st
        L.fa_bwd_bias.argtypes = [vp, vp, vp, vp, i, vp, vp, vp, ll, ll, ll, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                  i, vp]
        L.fa_bwd_bias.restype = st
        L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd_fp8.restype = st
        L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd_splitkv.restype = st
        L.fa_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i]
        L.fa_fwd_splitkv_workspace_bytes.restype = ctypes.c_size_t
        L.fa_fwd_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_fwd_decode.restype = st
        L.fa_fwd_decode_workspace_bytes.argtypes = [i, i, i, i, i]
        L.fa_fwd_decode_workspace_bytes.restype = ctypes.c_size_t
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_bwd.restype = st
        L.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_bwd_varlen.restype = st
        L.fa_bwd_single_pass.argtypes = [vp, vp, vp, vp, vp, vp, ll, ll, ll, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                         i, vp]
        L.fa_bwd_single_pass.restype = st
        L.fa_bwd_stage.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_bwd_stage.restype = st
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_bwd_noalloc.restype = st
        L.fa_bwd_workspace_bytes.argtypes = [i, i, i]
        L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.fa_sync_status.argtypes = [vp]
        L.fa_sync_status.restype = st
        L.fa_test_set_stall.argtypes = [i]
        L.fa_test_set_stall.restype = st
        L.fa_last_failure.argtypes = [ctypes.POINTER(ctypes.c_int)]
        L.fa_last_failure.restype = st
        L.fa_status_string.argtypes = [st]
        L.fa_status_string.restype = ctypes.c_char_p
        ip = ctypes.POINTER(ctypes.c_int)
        L.fa_sched_enumerate.argtypes = [i, i, i, i, i, ll, ip, ip, ip, ll]
        L.fa_sched_enumerate.restype = ll
        _lib = L
        return L


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _check(call: str, status: int) -> None:
    if status != FA_OK:
        raise FAError(call, status, fa_status_string(status))


def fa_fwd(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int, scale: float,
           causal: int, stream: int) -> int:
    """Raw C call; pointers and stream are integers.  Returns the status."""
    return lib().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)


def fa_fwd_varlen(q: int, k: int, v: int, o: int, lse: int, seqlens_q: int, seqlens_k: int, B: int, H: int,
                  Nq: int, Nk: int, d: int, scale: float, causal: int, stream: int) -> int:
    return lib().fa_fwd_varlen(q, k, v, o, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream)


def fa_fwd_ex(q: int, k: int, v: int, o: int, o_dtype: int, lse: int, seqlens_q: int, seqlens_k: int, B: int,
              H: int, Nq: int, Nk: int, d: int, scale: float, causal: int, stream: int) -> int:
    return lib().fa_fwd_ex(q, k, v, o, o_dtype, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream)


def fa_fwd_bias(q: int, k: int, v: int, o: int, o_dtype: int, lse: int, bias: int, bias_stride_b: int,
                bias_stride_h: int, bias_stride_q: int, seqlens_q: int, seqlens_k: int, B: int, H: int, Nq: int,
                Nk: int, d: int, scale: float, causal: int, stream: int) -> int:
    return lib().fa_fwd_bias(q, k, v, o, o_dtype, lse, bias, bias_stride_b, bias_stride_h, bias_stride_q, seqlens_q,
                             seqlens_k, B, H, Nq, Nk, d, scale, causal, stream)


def fa_bwd_ex(q: int, k: int, v: int, o: int, o_dtype: int, lse: int, do: int, dq: int, dk: int, dv: int,
              workspace: int, seqlens_q: int, seqlens_k: int, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
              causal: int, stream: int) -> int:
    return lib().fa_bwd_ex(q, k, v, o, o_dtype, lse, do, dq, dk, dv, workspace, seqlens_q, seqlens_k, B, H, Nq, Nk,
                           d, scale, causal, stream)


def fa_bwd_bias(q: int, k: int, v: int, o: int, o_dtype: int, lse: int, do: int, bias: int, bias_stride_b: int,
                bias_stride_h: int, bias_stride_q: int, dq: int, dk: int, dv: int, workspace: int, seqlens_q: int,
                seqlens_k: int, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, causal: int,
                stream: int) -> int:
    return lib().fa_bwd_bias(q, k, v, o, o_dtype, lse, do, bias, bias_stride_b, bias_stride_h, bias_stride_q, dq, dk,
                             dv, workspace, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream)


def fa_fwd_fp8(q8: int, k8: int, vt8: int, o: int, lse: int, B: int, H: int, N: int, d: int, scale: float,
               causal: int, stream: int) -> int:
    return lib().fa_fwd_fp8(q8, k8, vt8, o, lse, B, H, N, d, scale, causal, stream)


def fa_fwd_splitkv(q: int, k: int, v: int, o: int, lse: int, workspace: int, B: int, H: int, N: int, d: int,
                   scale: float, causal: int, stream: int) -> int:
    return lib().fa_fwd_splitkv(q, k, v, o, lse, workspace, B, H, N, d, scale, causal, stream)


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().fa_fwd_splitkv_workspace_bytes(B, H, N, d))


def fa_fwd_decode(q: int, k: int, v: int, o: int, lse: int, seqlens_q: int, seqlens_k: int, workspace: int, B: int,
                  H: int, Nq: int, Nk: int, d: int, scale: float, causal: int, stream: int) -> int:
    return lib().fa_fwd_decode(q, k, v, o, lse, seqlens_q, seqlens_k, workspace, B, H, Nq, Nk, d, scale, causal,
                               stream)


def fa_fwd_decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return lib().fa_fwd_decode_workspace_bytes(B, H, Nq, Nk, d)


def fa_bwd(q: int, k: int, v: int, o: int, lse: int, dO: int, dq: int, dk: int, dv: int, workspace: int,
           B: int, H: int, N: int, d: int, scale: float, causal: int, stream: int) -> int:
    return lib().fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, H, N, d, scale, causal, stream)


def fa_bwd_varlen(q: int, k: int, v: int, o: int, lse: int, do: int, dq: int, dk: int, dv: int, workspace: int,
                  seqlens_q: int, seqlens_k: int, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                  causal: int, stream: int) -> int:
    return lib().fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, workspace, seqlens_q, seqlens_k, B, H, Nq, Nk, d,
                               scale, causal, stream)


def fa_bwd_single_pass(q: int, k: int, v: int, lse: int, do: int, bias: int, bias_stride_b: int, bias_stride_h: int,
                       bias_stride_q: int, dq: int, dk: int, dv: int, workspace: int, seqlens_q: int, seqlens_k: int,
                       B: int, H: int, Nq: int, Nk: int, d: int, scale: float, causal: int, stream: int) -> int:
    return lib().fa_bwd_single_pass(q, k, v, lse, do, bias, bias_stride_b, bias_stride_h, bias_stride_q, dq, dk, dv,
                                    workspace, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream)


def fa_bwd_stage(stage: int, q: int, k: int, v: int, o: int, lse: int, dO: int, dq: int, dk: int, dv: int,
                 workspace: int, B: int, H: int, N: int, d: int, scale: float, causal: int, stream: int) -> int:
    """Raw C call of one backward stage (two-pass: 0 dQ and the row term,
    1 dK/dV; single-pass: 2 the row term and dQ = 0, 3 dK/dV/dQ)."""
    return lib().fa_bwd_stage(stage, q, k, v, o, lse, dO, dq, dk, dv, workspace, B, H, N, d, scale, causal, stream)


def fa_bwd_noalloc(q: int, k: int, v: int, o: int, lse: int, dO: int, dq: int, dk: int, dv: int,
                   B: int, H: int, N: int, d: int, scale: float, causal: int, stream: int) -> int:
    """Raw C call of the allocation-free backward (scratch held inside the
    library, at most FA_NOALLOC_MAX_ROWS = B*H*N rows).  Returns the status."""
    return lib().fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, stream)


FA_NOALLOC_MAX_ROWS = 1 << 20


def fa_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N))


def fa_sync_status(stream: int) -> int:
    return lib().fa_sync_status(stream)


def fa_test_set_stall(unit: int) -> int:
    """Testing hook: from the next call on, CTA 0 leaves one tile of its
    unit-th work unit unloaded (-1: off).  Returns the status."""
    return lib().fa_test_set_stall(int(unit))


def fa_last_failure() -> list:
    out = (ctypes.c_int * 4)()
    _check("fa_last_failure", lib().fa_last_failure(out))
    return list(out)


def fa_sched_enumerate(heads: int, N: int, d: int, causal: int, grid: int, l2_budget_bytes: int = 0):
    """Host-only: list of (cta, head, pair) the kernels' scheduler deals."""
    L = lib()
    total = L.fa_sched_enumerate(heads, N, d, causal, grid, l2_budget_bytes, None, None, None, 0)
    if total < 0:
        raise ValueError("invalid scheduler arguments")
    arr = [(ctypes.c_int * max(total, 1))() for _ in range(3)]
    L.fa_sched_enumerate(heads, N, d, causal, grid, l2_budget_bytes, arr[0], arr[1], arr[2], total)
    return [(arr[0][i], arr[1][i], arr[2][i]) for i in range(total)]


# ----------------------------------------------------------------- torch side
# PyTorch supplies device memory and the current stream; nothing else.

def _stream_handle(device) -> int:
    import torch
    return int(torch.cuda.current_stream(device).cuda_stream)


def _check_inputs(*ts):
    import torch
    ref = ts[0]
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape != ref.shape \
                or t.device != ref.device or t.dim() != 4:
            raise ValueError("q, k, v (and dO) must be contiguous bf16 CUDA tensors of one shape [B, H, N, d]")


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None):
    """O, LSE = attention(q, k, v) through fa_fwd on the current stream.

    q, k, v: bf16 CUDA tensors [B, H, N, d].  Returns fp32 O [B, H, N, d]
    and fp32 LSE [B, H, N].  ``out`` may supply preallocated (O, LSE).
    """
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        o = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    _check("fa_fwd", fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, scale, int(bool(causal)), _stream_handle(q.device)))
    return o, lse


def forward_splitkv(q, k, v, causal: bool = False, scale: float | None = None, workspace=None, out=None):
    """O, LSE through fa_fwd_splitkv (each query tile's keys split over
    several CTAs; for batches with few query tiles).  Arguments as forward;
    ``workspace`` an optional fp32 CUDA tensor of
    fa_fwd_splitkv_workspace_bytes(B, H, N, d) bytes."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        o = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    _check("fa_fwd_splitkv", fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                            workspace.data_ptr() if workspace is not None else 0, B, H, N, d, scale,
                                            int(bool(causal)), _stream_handle(q.device)))
    return o, lse


def forward_varlen(q, k, v, seqlens_q=None, seqlens_k=None, causal: bool = False, scale: float | None = None,
                   out=None, o_dtype=None):
    """O, LSE through fa_fwd_varlen: q [B,H,Nq,d], k and v [B,H,Nk,d] (bf16,
    CUDA); seqlens_q / seqlens_k optional int32 CUDA tensors of B valid
    lengths.  Causal alignment is bottom-right (see include/fa.h).  With
    o_dtype=torch.bfloat16 O is written as bf16 through fa_fwd_ex."""
    import torch
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with the batch, heads and d of q")
    for t in (seqlens_q, seqlens_k):
        if t is not None and (not t.is_cuda or t.dtype != torch.int32 or t.numel() != B or not t.is_contiguous()):
            raise ValueError("seqlens must be contiguous int32 CUDA tensors of B entries")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        o = torch.empty((B, H, Nq, d), dtype=o_dtype or torch.float32, device=q.device)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    sq = seqlens_q.data_ptr() if seqlens_q is not None else 0
    sk = seqlens_k.data_ptr() if seqlens_k is not None else 0
    if o.dtype == torch.float32:
        _check("fa_fwd_varlen", fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                              sq, sk, B, H, Nq, Nk, d, scale, int(bool(causal)),
                                              _stream_handle(q.device)))
    elif o.dtype == torch.bfloat16:
        _check("fa_fwd_ex", fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), FA_DTYPE_BF16,
                                      lse.data_ptr(), sq, sk, B, H, Nq, Nk, d, scale, int(bool(causal)),
                                      _stream_handle(q.device)))
    else:
        raise ValueError("O must be float32 or bfloat16")
    return o, lse


def _bias_strides(bias, B, H, Nq, Nk):
    """Element strides (b, h, query) of a bf16 CUDA mask broadcastable to
    [B, H, Nq, Nk] with contiguous keys."""
    import torch
    if not bias.is_cuda or bias.dtype != torch.bfloat16:
        raise ValueError("bias must be a bf16 CUDA tensor")
    bias = bias.expand(B, H, Nq, Nk)
    if bias.stride(3) != 1:
        raise ValueError("the bias's key dimension must be contiguous")
    return bias.stride(0), bias.stride(1), bias.stride(2)


def forward_bias(q, k, v, bias, seqlens_q=None, seqlens_k=None, causal: bool = False, scale: float | None = None,
                 o_dtype=None, out=None):
    """O, LSE through fa_fwd_bias: softmax(scale * q k^T + bias) v.  ``bias``
    is a bf16 CUDA tensor broadcastable to [B, H, Nq, Nk] (e.g. made with
    expand()) whose last dimension is contiguous; other arguments as
    forward_varlen."""
    import torch
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with the batch, heads and d of q")
    sb, sh, sq = _bias_strides(bias, B, H, Nq, Nk)
    for t in (seqlens_q, seqlens_k):
        if t is not None and (not t.is_cuda or t.dtype != torch.int32 or t.numel() != B or not t.is_contiguous()):
            raise ValueError("seqlens must be contiguous int32 CUDA tensors of B entries")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        o = torch.empty((B, H, Nq, d), dtype=o_dtype or torch.float32, device=q.device)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    if o.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("O must be float32 or bfloat16")
    _check("fa_fwd_bias", fa_fwd_bias(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      FA_DTYPE_BF16 if o.dtype == torch.bfloat16 else FA_DTYPE_F32, lse.data_ptr(),
                                      bias.data_ptr(), sb, sh, sq,
                                      seqlens_q.data_ptr() if seqlens_q is not None else 0,
                                      seqlens_k.data_ptr() if seqlens_k is not None else 0,
                                      B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(q.device)))
    return o, lse


def forward_fp8(q8, k8, vt8, causal: bool = False, scale: float | None = None, out=None):
    """O, LSE through fa_fwd_fp8: q8, k8 [B,H,N,128] and vt8 (V transposed)
    [B,H,128,N], E4M3 CUDA tensors (torch.float8_e4m3fn, or uint8 holding
    the bit patterns), contiguous; O fp32."""
    import torch
    for t in (q8, k8, vt8):
        if not t.is_cuda or t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q8, k8, vt8 must be contiguous 4-D E4M3 (or uint8) CUDA tensors")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or vt8.shape != (B, H, d, N):
        raise ValueError("k8 must be [B, H, N, d] and vt8 [B, H, d, N]")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        o = torch.empty((B, H, N, d), dtype=torch.float32, device=q8.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    else:
        o, lse = out
    _check("fa_fwd_fp8", fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    B, H, N, d, scale, int(bool(causal)), _stream_handle(q8.device)))
    return o, lse


def forward_decode(q, k, v, seqlens_q=None, seqlens_k=None, causal: bool = False, scale: float | None = None,
                   workspace=None, out=None):
    """O, LSE through fa_fwd_decode: q [B,H,Nq,d] with Nq <= FA_DECODE_MAX_Q,
    k and v [B,H,Nk,d] (bf16, CUDA); same results as forward_varlen."""
    import torch
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with the batch, heads and d of q")
    for t in (seqlens_q, seqlens_k):
        if t is not None and (not t.is_cuda or t.dtype != torch.int32 or t.numel() != B or not t.is_contiguous()):
            raise ValueError("seqlens must be contiguous int32 CUDA tensors of B entries")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        o = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    _check("fa_fwd_decode", fa_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                          seqlens_q.data_ptr() if seqlens_q is not None else 0,
                                          seqlens_k.data_ptr() if seqlens_k is not None else 0,
                                          workspace.data_ptr() if workspace is not None else 0,
                                          B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(q.device)))
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, workspace=None,
             out=None):
    """dQ, dK, dV through fa_bwd on the current stream (fp32 outputs)."""
    import torch
    _check_inputs(q, k, v, do)
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        dq, dk, dv = (torch.empty((B, H, N, d), dtype=torch.float32, device=q.device) for _ in range(3))
    else:
        dq, dk, dv = out
    ws = workspace.data_ptr() if workspace is not None else 0
    _check("fa_bwd", fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws,
                            B, H, N, d, scale, int(bool(causal)), _stream_handle(q.device)))
    return dq, dk, dv


def backward_varlen(q, k, v, o, lse, do, seqlens_q=None, seqlens_k=None, causal: bool = False,
                    scale: float | None = None, workspace=None, out=None):
    """dQ, dK, dV through fa_bwd_ex: q, do, o [B,H,Nq,d] (o fp32 or bf16),
    lse [B,H,Nq], k and v [B,H,Nk,d]; seqlens as forward_varlen (fp32
    outputs)."""
    return _backward(q, k, v, o, lse, do, None, seqlens_q, seqlens_k, causal, scale, workspace, out)


def backward_bias(q, k, v, o, lse, do, bias, seqlens_q=None, seqlens_k=None, causal: bool = False,
                  scale: float | None = None, workspace=None, out=None):
    """dQ, dK, dV of forward_bias through fa_bwd_bias; ``bias`` exactly as
    given to forward_bias, other arguments as backward_varlen."""
    return _backward(q, k, v, o, lse, do, bias, seqlens_q, seqlens_k, causal, scale, workspace, out)


def _backward(q, k, v, o, lse, do, bias, seqlens_q, seqlens_k, causal, scale, workspace, out):
    import torch
    for t in (q, k, v, do):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v, do must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape or do.shape != q.shape:
        raise ValueError("k, v must be [B, H, Nk, d] and do [B, H, Nq, d]")
    for t in (seqlens_q, seqlens_k):
        if t is not None and (not t.is_cuda or t.dtype != torch.int32 or t.numel() != B or not t.is_contiguous()):
            raise ValueError("seqlens must be contiguous int32 CUDA tensors of B entries")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        dq = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device)
        dk, dv = (torch.empty((B, H, Nk, d), dtype=torch.float32, device=q.device) for _ in range(2))
    else:
        dq, dk, dv = out
    ws = workspace.data_ptr() if workspace is not None else 0
    if o.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("O must be float32 or bfloat16")
    o_dtype = FA_DTYPE_BF16 if o.dtype == torch.bfloat16 else FA_DTYPE_F32
    lq = seqlens_q.data_ptr() if seqlens_q is not None else 0
    lk = seqlens_k.data_ptr() if seqlens_k is not None else 0
    if bias is None:
        _check("fa_bwd_ex",
               fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), o_dtype, lse.data_ptr(),
                         do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws, lq, lk,
                         B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(q.device)))
    else:
        sb, sh, sq = _bias_strides(bias, B, H, Nq, Nk)
        _check("fa_bwd_bias",
               fa_bwd_bias(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), o_dtype, lse.data_ptr(),
                           do.data_ptr(), bias.data_ptr(), sb, sh, sq, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                           ws, lq, lk, B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(q.device)))
    return dq, dk, dv


def backward_single_pass(q, k, v, lse, do, bias=None, seqlens_q=None, seqlens_k=None, causal: bool = False,
                         scale: float | None = None, workspace=None, out=None):
    """dQ, dK, dV through fa_bwd_single_pass: q, do [B,H,Nq,d], lse
    [B,H,Nq], k and v [B,H,Nk,d] (bf16 CUDA); optional bias and seqlens as
    backward_bias / backward_varlen (fp32 outputs)."""
    import torch
    for t in (q, k, v, do):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v, do must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape or do.shape != q.shape:
        raise ValueError("k, v must be [B, H, Nk, d] and do [B, H, Nq, d]")
    for t in (seqlens_q, seqlens_k):
        if t is not None and (not t.is_cuda or t.dtype != torch.int32 or t.numel() != B or not t.is_contiguous()):
            raise ValueError("seqlens must be contiguous int32 CUDA tensors of B entries")
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    if out is None:
        dq = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device)
        dk, dv = (torch.empty((B, H, Nk, d), dtype=torch.float32, device=q.device) for _ in range(2))
    else:
        dq, dk, dv = out
    sb = sh = sq = 0
    if bias is not None:
        sb, sh, sq = _bias_strides(bias, B, H, Nq, Nk)
    _check("fa_bwd_single_pass",
           fa_bwd_single_pass(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(), do.data_ptr(),
                              bias.data_ptr() if bias is not None else 0, sb, sh, sq, dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), workspace.data_ptr() if workspace is not None else 0,
                              seqlens_q.data_ptr() if seqlens_q is not None else 0,
                              seqlens_k.data_ptr() if seqlens_k is not None else 0,
                              B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(q.device)))
    return dq, dk, dv


def backward_stage(stage: int, q, k, v, o, lse, do, dq, dk, dv, workspace, causal: bool = False,
                   scale: float | None = None):
    """One backward stage through fa_bwd_stage on the current stream."""
    import torch
    _check_inputs(q, k, v, do)
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    _check(f"fa_bwd_stage({stage})",
           fa_bwd_stage(stage, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr() if o is not None else 0,
                        lse.data_ptr(),
                        do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                        B, H, N, d, scale, int(bool(causal)), _stream_handle(q.device)))


def sync_status(device=None) -> None:
    """Synchronise the current stream and raise if a kernel reported a failure."""
    status = fa_sync_status(_stream_handle(device))
    if status != FA_OK:
        detail = fa_last_failure() if status == FA_ERR_TIMEOUT else None
        raise FAError("fa_sync_status", status, fa_status_string(status) + (f" {detail}" if detail else ""))
