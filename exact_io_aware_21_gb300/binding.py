"""Thin ctypes binding of libfa_gb300.so (C ABI in include/fa.h).

Argument marshalling only: torch tensors are turned into (pointer, strides)
descriptors, the workspace and outputs are allocated with torch on the tensors'
device, and the current torch CUDA stream is passed down.  Every step of the
attention computation runs in the library's kernels; if the library is not
built, every call raises ``FAError`` (there is no fallback).
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

FA_OK = 0


class FAError(RuntimeError):
    """An error code returned by the C ABI (message from fa_strerror)."""

    def __init__(self, code, msg):
        super().__init__(f"fa error {code}: {msg}")
        self.code = code


class FaTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64), ("stride_n", ctypes.c_int64),
                ("stride_h", ctypes.c_int64)]


class FaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Nq", ctypes.c_int),
                ("Nk", ctypes.c_int), ("d", ctypes.c_int), ("scale", ctypes.c_float), ("causal", ctypes.c_int),
                ("window", ctypes.c_int), ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("rescale_threshold", ctypes.c_float)]


# name -> (restype, argtypes); mirrors include/fa.h
_PT = ctypes.POINTER(FaTensor)
_PS = ctypes.POINTER(FaShape)
_VP = ctypes.c_void_p
_I = ctypes.c_int
_PI = ctypes.POINTER(ctypes.c_int)
_SZ = ctypes.c_size_t
SIGNATURES = {
    "fa_fwd_workspace_size": (_SZ, [_PS]),
    "fa_fwd": (_I, [_PT, _PT, _PT, _PT, _VP, _PT, _PS, _VP, _SZ, _VP]),
    "fa_bwd_workspace_size": (_SZ, [_PS]),
    "fa_bwd": (_I, [_PT, _PT, _PT, _PT, _VP, _PT, _PT, _PT, _PT, _PT, _PS, _VP, _SZ, _VP]),
    "fa_bwd_part": (_I, [_I, _PT, _PT, _PT, _PT, _VP, _PT, _PT, _PT, _PT, _PT, _PS, _VP, _SZ, _VP]),
    "fa_decode_num_splits": (_I, [_PS, _I]),
    "fa_decode_workspace_size": (_SZ, [_PS, _I]),
    "fa_decode": (_I, [_PT, _PT, _PT, _PT, _VP, _PS, _I, _VP, _SZ, _VP]),
    "fa_decode_partials_layout": (_I, [_PS, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "fa_decode_paged": (_I, [_PT, _PT, _PT, _VP, _I, _VP, _I, _I, _PT, _VP, _PS, _I, _VP, _SZ, _VP]),
    "fa_decode_paged_workspace_size": (_SZ, [_PS, _I, _I]),
    "fa_decode_noalloc_max_bytes": (_SZ, []),
    "fa_decode_noalloc": (_I, [_PT, _PT, _PT, _PT, _VP, _PS, _I, _VP]),
    "fa_decode_noalloc_status": (_I, [_VP, _PI]),
    "fa_get_device_status": (_I, [_VP, _VP, _PI]),
    "fa_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "fa_set_trace": (None, [_VP, _SZ]),
    "fa_test_withhold_arrive": (None, []),
    "fa_strerror": (ctypes.c_char_p, [_I]),
    "fa_last_cuda_error": (_I, []),
    "fa_tile_class": (_I, [_PS, _I, _I]),
    "fa_fwd_num_units": (_I, [_PS]),
    "fa_fwd_unit": (_I, [_PS, _I, _PI, _PI, _PI]),
    "fa_dkdv_num_units": (_I, [_PS]),
    "fa_dkdv_unit": (_I, [_PS, _I, _PI, _PI, _PI]),
    "fa_dq_num_units": (_I, [_PS]),
    "fa_dq_unit": (_I, [_PS, _I, _PI, _PI, _PI]),
    "fa_decode_split_range": (_I, [_PS, _I, _I, _PI, _PI]),
    "fa_fwd_schedule": (_I, [_PS, _I, _PI, _PI]),
    "fa_fwd_split_plan": (_I, [_PS, _I, _PI, _PI]),
    "fa_selftest_mma": (_I, [_I, _I, _VP, _VP, _VP, _VP, _VP]),
    "fa_fwd_blocksparse": (_I, [_PT, _PT, _PT, _VP, _VP, _I, _PT, _VP, _PT, _PS, _VP, _SZ, _VP]),
    "fa_bwd_blocksparse_workspace_size": (_SZ, [_PS, _I]),
    "fa_bwd_blocksparse": (_I, [_PT, _PT, _PT, _VP, _VP, _I, _PT, _VP, _PT, _PT, _PT, _PT, _PT, _PS, _VP, _SZ, _VP]),
    "fa_fwd_varlen_workspace_size": (_SZ, [_PS, _I]),
    "fa_fwd_varlen": (_I, [_PT, _PT, _PT, _VP, _VP, _I, _I, _PT, _VP, _PT, _PS, _VP, _SZ, _VP]),
    "fa_bwd_varlen_workspace_size": (_SZ, [_PS, _I]),
    "fa_bwd_varlen": (_I, [_PT, _PT, _PT, _VP, _VP, _I, _I, _PT, _VP, _PT, _PT, _PT, _PT, _PT, _PS, _VP, _SZ, _VP]),
    "fa_quantize_fp8_workspace_size": (_SZ, [_I, _I]),
    "fa_quantize_fp8": (_I, [_PT, _I, _I, _I, _I, _I, _VP, _PT, _VP, _VP, _SZ, _VP]),
    "fa_fwd_fp8": (_I, [_PT, _PT, _PT, _VP, _VP, _VP, _PT, _VP, _PS, _VP, _SZ, _VP]),
}


def library_path():
    return os.path.join(_HERE, "_build", "libfa_gb300.so")


def library():
    """Load libfa_gb300.so (once).  Raises FAError if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise FAError(-1, f"{path} is missing: build it with `python -m exact_io_aware_21_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def check(rc):
    if rc != FA_OK:
        lib = library()
        msg = lib.fa_strerror(rc).decode()
        if rc in (5, 7):
            msg += f" (cuda error {lib.fa_last_cuda_error()})"
        raise FAError(rc, msg)


def shape(B, Hq, Hkv, Nq, Nk, d, scale=None, causal=False, window=None, rescale_threshold=0.0):
    """window = (left, right): query i sees keys i - left .. i + right (negative: unbounded).
    rescale_threshold: conditional rescaling of the forward, log2 units (0 = exact running max)."""
    w = (0, -1, -1) if window is None else (1, int(window[0]), int(window[1]))
    return FaShape(B, Hq, Hkv, Nq, Nk, d, 1.0 / math.sqrt(d) if scale is None else float(scale), int(bool(causal)),
                   *w, float(rescale_threshold))


def tdesc(t):
    """[B, N, H, d] bf16 CUDA tensor -> FaTensor (strides in elements)."""
    if t.dim() != 4 or t.dtype != torch.bfloat16 or not t.is_cuda or t.stride(-1) != 1:
        raise FAError(1, "expected a 4-D bf16 CUDA tensor [B, N, H, d] with unit head-dim stride")
    return FaTensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def tdesc_packed(t):
    """[total, H, d] bf16 CUDA tensor (packed sequences) -> FaTensor (stride_b unused)."""
    if t.dim() != 3 or t.dtype != torch.bfloat16 or not t.is_cuda or t.stride(-1) != 1:
        raise FAError(1, "expected a 3-D bf16 CUDA tensor [total, H, d] with unit head-dim stride")
    return FaTensor(t.data_ptr(), 0, t.stride(0), t.stride(1))


def _cu(t):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 1:
        raise FAError(1, "cu_seqlens must be contiguous 1-D int32 CUDA tensors")
    return t.data_ptr()


def tdesc_u8(t):
    """[B, N, H, d] uint8 (E4M3 codes) CUDA tensor -> FaTensor (strides in bytes)."""
    if t.dim() != 4 or t.dtype != torch.uint8 or not t.is_cuda or t.stride(-1) != 1:
        raise FAError(1, "expected a 4-D uint8 CUDA tensor [B, N, H, d] with unit head-dim stride")
    return FaTensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


# Tests set OUTPUT_CANARY to NaN so that any output element a kernel leaves
# unwritten shows up (E4M3 code outputs then start as 0xFF, a NaN code); the
# default leaves outputs uninitialised, as torch.empty does.
OUTPUT_CANARY = None


def _out(shape, dtype, device):
    if OUTPUT_CANARY is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return torch.full(shape, 0xFF if dtype == torch.uint8 else OUTPUT_CANARY, dtype=dtype, device=device)


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- C-ABI mirrors
def _opt(t):
    return None if t is None else ctypes.byref(tdesc(t))


def fa_fwd(q, k, v, o, lse, s, workspace, o_res=None):
    lib = library()
    check(lib.fa_fwd(tdesc(q), tdesc(k), tdesc(v), tdesc(o), lse.data_ptr(), _opt(o_res), ctypes.byref(s),
                     workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, s, workspace, o_res=None):
    lib = library()
    check(lib.fa_bwd(tdesc(q), tdesc(k), tdesc(v), tdesc(o), lse.data_ptr(), _opt(o_res), tdesc(do), tdesc(dq),
                     tdesc(dk), tdesc(dv), ctypes.byref(s), workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_bwd_part(part, q, k, v, o, lse, do, dq, dk, dv, s, workspace, o_res=None):
    lib = library()
    check(lib.fa_bwd_part(int(part), tdesc(q), tdesc(k), tdesc(v), tdesc(o), lse.data_ptr(), _opt(o_res),
                          tdesc(do), tdesc(dq), tdesc(dk), tdesc(dv), ctypes.byref(s), workspace.data_ptr(),
                          workspace.numel(), _stream(q)))


def fa_decode(q, kc, vc, o, lse, s, num_splits, workspace):
    lib = library()
    check(lib.fa_decode(tdesc(q), tdesc(kc), tdesc(vc), tdesc(o), lse.data_ptr(), ctypes.byref(s), int(num_splits),
                        workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_decode_paged(q, kc, vc, block_table, seqlens_k, o, lse, s, num_splits, workspace):
    """kc, vc: [num_pages, page_size, Hkv, d] bf16; block_table [B, max_pages] and
    seqlens_k [B] int32 CUDA tensors (contiguous)."""
    lib = library()
    if block_table.dtype != torch.int32 or seqlens_k.dtype != torch.int32 or not block_table.is_contiguous():
        raise FAError(1, "block_table and seqlens_k must be contiguous int32 CUDA tensors")
    check(lib.fa_decode_paged(tdesc(q), tdesc(kc), tdesc(vc), block_table.data_ptr(), block_table.shape[1],
                              seqlens_k.data_ptr(), kc.shape[0], kc.shape[1], tdesc(o), lse.data_ptr(),
                              ctypes.byref(s), int(num_splits), workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_fwd_blocksparse(q, k, v, row_ptr, col_idx, o, lse, s, workspace, o_res=None):
    """row_ptr [ceil(Nq/128) + 1], col_idx [nnz]: contiguous int32 CUDA tensors (the CSR block table)."""
    lib = library()
    for t in (row_ptr, col_idx):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise FAError(1, "row_ptr and col_idx must be contiguous int32 CUDA tensors")
    check(lib.fa_fwd_blocksparse(tdesc(q), tdesc(k), tdesc(v), row_ptr.data_ptr(),
                                 col_idx.data_ptr() if col_idx.numel() else None, col_idx.numel(), tdesc(o),
                                 lse.data_ptr(), _opt(o_res), ctypes.byref(s), workspace.data_ptr(),
                                 workspace.numel(), _stream(q)))


def fa_bwd_blocksparse(q, k, v, row_ptr, col_idx, o, lse, do, dq, dk, dv, s, workspace, o_res=None):
    lib = library()
    for t in (row_ptr, col_idx):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise FAError(1, "row_ptr and col_idx must be contiguous int32 CUDA tensors")
    check(lib.fa_bwd_blocksparse(tdesc(q), tdesc(k), tdesc(v), row_ptr.data_ptr(),
                                 col_idx.data_ptr() if col_idx.numel() else None, col_idx.numel(), tdesc(o),
                                 lse.data_ptr(), _opt(o_res), tdesc(do), tdesc(dq), tdesc(dk), tdesc(dv),
                                 ctypes.byref(s), workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_fwd_varlen(q, k, v, cu_q, cu_k, max_q, max_k, o, lse, s, workspace, o_res=None):
    lib = library()
    check(lib.fa_fwd_varlen(tdesc_packed(q), tdesc_packed(k), tdesc_packed(v), _cu(cu_q), _cu(cu_k), int(max_q),
                            int(max_k), tdesc_packed(o), lse.data_ptr(),
                            None if o_res is None else ctypes.byref(tdesc_packed(o_res)), ctypes.byref(s),
                            workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_bwd_varlen(q, k, v, cu_q, cu_k, max_q, max_k, o, lse, do, dq, dk, dv, s, workspace, o_res=None):
    lib = library()
    check(lib.fa_bwd_varlen(tdesc_packed(q), tdesc_packed(k), tdesc_packed(v), _cu(cu_q), _cu(cu_k), int(max_q),
                            int(max_k), tdesc_packed(o), lse.data_ptr(),
                            None if o_res is None else ctypes.byref(tdesc_packed(o_res)), tdesc_packed(do),
                            tdesc_packed(dq), tdesc_packed(dk), tdesc_packed(dv), ctypes.byref(s),
                            workspace.data_ptr(), workspace.numel(), _stream(q)))


def fa_quantize_fp8(x, block_rows, signs, out, scales, workspace):
    """x [B, N, H, d] bf16 -> out uint8 codes and fp32 scales (see fa_quantize_fp8 in include/fa.h)."""
    lib = library()
    B, N, H, d = x.shape
    if signs is not None and (signs.dtype != torch.float32 or not signs.is_cuda or signs.numel() != d):
        raise FAError(1, "signs must be a float32 CUDA tensor of d values")
    check(lib.fa_quantize_fp8(tdesc(x), B, N, H, d, int(block_rows), None if signs is None else signs.data_ptr(),
                              tdesc_u8(out), scales.data_ptr(), workspace.data_ptr(), workspace.numel(),
                              _stream(x)))


def fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, s, workspace):
    lib = library()
    check(lib.fa_fwd_fp8(tdesc_u8(q8), tdesc_u8(k8), tdesc_u8(v8), q_scale.data_ptr(), k_scale.data_ptr(),
                         v_scale.data_ptr(), tdesc(o), lse.data_ptr(), ctypes.byref(s), workspace.data_ptr(),
                         workspace.numel(), _stream(q8)))


def device_status(workspace):
    """Synchronise and return (rc, status bits) recorded in the workspace."""
    lib = library()
    st = ctypes.c_int(0)
    rc = lib.fa_get_device_status(workspace.data_ptr(), _stream(workspace), ctypes.byref(st))
    return rc, st.value


TRACE_MAX_CTAS, TRACE_UNIT0, TRACE_UNIT_WORDS = 1024, 4096, 16


def set_trace(buf):
    """Record the dense forward's timestamps into ``buf`` (a CUDA int64 tensor of at
    least TRACE_UNIT0 + TRACE_UNIT_WORDS * units elements), or stop (None)."""
    lib = library()
    if buf is None:
        lib.fa_set_trace(None, 0)
    else:
        lib.fa_set_trace(buf.data_ptr(), buf.numel() * buf.element_size())


# ---------------------------------------------------------------- convenience API
def _dims(q, k, scale, causal, window=None, rescale_threshold=0.0):
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    return shape(B, Hq, Hkv, Nq, Nk, d, scale, causal, window, rescale_threshold)


def forward(q, k, v, causal=False, scale=None, residual=False, window=None, rescale_threshold=0.0):
    """O, LSE = attention(q, k, v).  q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] bf16 on CUDA.

    With ``residual=True`` also returns O's bf16 rounding residual, which
    ``backward`` uses to form D accurately (see fa_bwd in include/fa.h).
    ``window=(left, right)`` restricts query i to keys i - left .. i + right.
    ``rescale_threshold`` > 0 turns on conditional rescaling (fa_shape_t in include/fa.h).
    """
    s = _dims(q, k, scale, causal, window, rescale_threshold)
    o = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = _out((s.B, s.Hq, s.Nq), dtype=torch.float32, device=q.device)
    res = _out(q.shape, dtype=torch.bfloat16, device=q.device) if residual else None
    ws = _ws(library().fa_fwd_workspace_size(ctypes.byref(s)), q.device)
    fa_fwd(q, k, v, o, lse, s, ws, res)
    return (o, lse, res) if residual else (o, lse)


def backward(q, k, v, o, lse, do, causal=False, scale=None, o_residual=None, window=None):
    """dQ, dK, dV of attention given O, LSE (and optionally O's residual) from ``forward``."""
    s = _dims(q, k, scale, causal, window)
    dq = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    dk = _out(k.shape, dtype=torch.bfloat16, device=q.device)
    dv = _out(v.shape, dtype=torch.bfloat16, device=q.device)
    ws = _ws(library().fa_bwd_workspace_size(ctypes.byref(s)), q.device)
    fa_bwd(q, k, v, o, lse, do, dq, dk, dv, s, ws, o_residual)
    return dq, dk, dv


def decode(q, k_cache, v_cache, scale=None, num_splits=0):
    """Split-KV decode: O, LSE for a short query q [B,Nq,Hq,d] against the cache."""
    s = _dims(q, k_cache, scale, False)
    o = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = _out((s.B, s.Hq, s.Nq), dtype=torch.float32, device=q.device)
    ws = _ws(library().fa_decode_workspace_size(ctypes.byref(s), int(num_splits)), q.device)
    fa_decode(q, k_cache, v_cache, o, lse, s, num_splits, ws)
    return o, lse


def decode_paged(q, k_cache, v_cache, block_table, seqlens_k, max_seqlen=None, scale=None, num_splits=0):
    """Decode against a paged, variable-length cache (see fa_decode_paged in include/fa.h).

    q [B,Nq,Hq,d]; k_cache/v_cache [num_pages, page_size, Hkv, d]; block_table
    [B, max_pages] int32; seqlens_k [B] int32.  ``max_seqlen`` bounds the
    lengths (defaults to seqlens_k.max(), which reads it back to the host).
    """
    B, Nq, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    if max_seqlen is None:
        max_seqlen = int(seqlens_k.max().item())
    s = shape(B, Hq, Hkv, Nq, int(max_seqlen), d, scale, False)
    o = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = _out((B, Hq, Nq), dtype=torch.float32, device=q.device)
    ws = _ws(library().fa_decode_paged_workspace_size(ctypes.byref(s), int(num_splits), k_cache.shape[1]), q.device)
    fa_decode_paged(q, k_cache, v_cache, block_table, seqlens_k, o, lse, s, num_splits, ws)
    return o, lse


def quantize_fp8(x, block_rows=128, signs=None):
    """E4M3 codes and scales of x [B, N, H, d] bf16: per 128-row block (``block_rows``
    = 128, scales [B, H, ceil(N/128)]) or per head (0, scales [B, H]); ``signs``
    (d float32 +-1 on the device) rotates the rows by the random Hadamard matrix first."""
    B, N, H, d = x.shape
    out = _out((B, N, H, d), dtype=torch.uint8, device=x.device)
    nblk = -(-N // 128)
    scales = _out((B, H, nblk) if block_rows else (B, H), dtype=torch.float32, device=x.device)
    ws = _ws(library().fa_quantize_fp8_workspace_size(B, H), x.device)
    fa_quantize_fp8(x, block_rows, signs, out, scales, ws)
    return out, scales


def forward_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=None, window=None, rescale_threshold=0.0):
    """O (bf16), LSE from E4M3 operands made by ``quantize_fp8`` (Q, K per block, V per head)."""
    s = _dims(q8, k8, scale, causal, window, rescale_threshold)
    o = _out(q8.shape, dtype=torch.bfloat16, device=q8.device)
    lse = _out((s.B, s.Hq, s.Nq), dtype=torch.float32, device=q8.device)
    ws = _ws(library().fa_fwd_workspace_size(ctypes.byref(s)), q8.device)
    fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, s, ws)
    return o, lse


def _varlen_shape(q, k, cu_q, scale, causal, rescale_threshold=0.0):
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    return shape(cu_q.numel() - 1, Hq, Hkv, total_q, total_k, d, scale, causal, None, rescale_threshold)


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False, scale=None,
                   residual=False, rescale_threshold=0.0):
    """Packed variable-length forward (see fa_fwd_varlen in include/fa.h): q [total_q, Hq, d],
    k/v [total_k, Hkv, d] bf16, cu_seqlens int32 [B + 1] on the device.  Returns O, LSE
    [Hq, total_q] (and O's residual with ``residual=True``)."""
    s = _varlen_shape(q, k, cu_seqlens_q, scale, causal, rescale_threshold)
    o = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = _out((s.Hq, s.Nq), dtype=torch.float32, device=q.device)
    res = _out(q.shape, dtype=torch.bfloat16, device=q.device) if residual else None
    ws = _ws(library().fa_fwd_varlen_workspace_size(ctypes.byref(s), int(max_seqlen_q)), q.device)
    fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, o, lse, s, ws, res)
    return (o, lse, res) if residual else (o, lse)


def backward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, o, lse, do, causal=False,
                    scale=None, o_residual=None):
    """dQ, dK, dV of the packed forward."""
    s = _varlen_shape(q, k, cu_seqlens_q, scale, causal)
    dq = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    dk = _out(k.shape, dtype=torch.bfloat16, device=q.device)
    dv = _out(v.shape, dtype=torch.bfloat16, device=q.device)
    ws = _ws(library().fa_bwd_varlen_workspace_size(ctypes.byref(s), int(max_seqlen_q)), q.device)
    fa_bwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, o, lse, do, dq, dk, dv, s, ws,
                  o_residual)
    return dq, dk, dv


def forward_blocksparse(q, k, v, row_ptr, col_idx, causal=False, scale=None, residual=False,
                        rescale_threshold=0.0):
    """Block-sparse forward (see fa_fwd_blocksparse in include/fa.h): q [B,Nq,Hq,d], k/v
    [B,Nk,Hkv,d] bf16; row_ptr / col_idx the CSR table of 128-key tiles per 128-row query tile."""
    s = _dims(q, k, scale, causal, None, rescale_threshold)
    o = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = _out((s.B, s.Hq, s.Nq), dtype=torch.float32, device=q.device)
    res = _out(q.shape, dtype=torch.bfloat16, device=q.device) if residual else None
    ws = _ws(library().fa_fwd_workspace_size(ctypes.byref(s)), q.device)
    fa_fwd_blocksparse(q, k, v, row_ptr, col_idx, o, lse, s, ws, res)
    return (o, lse, res) if residual else (o, lse)


def backward_blocksparse(q, k, v, row_ptr, col_idx, o, lse, do, causal=False, scale=None, o_residual=None):
    """dQ, dK, dV of ``forward_blocksparse`` (same table)."""
    s = _dims(q, k, scale, causal)
    dq = _out(q.shape, dtype=torch.bfloat16, device=q.device)
    dk = _out(k.shape, dtype=torch.bfloat16, device=q.device)
    dv = _out(v.shape, dtype=torch.bfloat16, device=q.device)
    ws = _ws(library().fa_bwd_blocksparse_workspace_size(ctypes.byref(s), col_idx.numel()), q.device)
    fa_bwd_blocksparse(q, k, v, row_ptr, col_idx, o, lse, do, dq, dk, dv, s, ws, o_residual)
    return dq, dk, dv
