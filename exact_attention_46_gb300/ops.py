"""Python binding of the attention library: torch tensors in, C-ABI calls out.

Argument marshalling only -- every step of the computation runs in the CUDA
kernels behind include/attn46.h.  torch supplies device memory and the current
stream.  Tensors are [B, S, H, D] contiguous on the current CUDA device.
"""

import torch

from . import _lib

__all__ = ["attn_fwd", "attn_fwd_fp8", "attn_fwd_varlen", "attn_bwd", "attn_fwd_gqa", "attn_decode", "hadamard_rotate_quant_fp8", "rope_cos_sin_table",
           "rope_hadamard_rotate_quant_fp8", "check",
           "set_spin_limit", "selftest_bounded_wait", "block_count", "ATTN_BF16", "ATTN_FP8_E4M3"]

ATTN_BF16 = 0
ATTN_FP8_E4M3 = 1
TOKEN_BLOCK = 128


def block_count(S):
    """Number of 128-token scale blocks for sequence length S."""
    return (S + TOKEN_BLOCK - 1) // TOKEN_BLOCK


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _check4(*ts):
    for t in ts:
        if not (t.is_cuda and t.is_contiguous() and t.dim() == 4):
            raise ValueError("expected contiguous 4-D CUDA tensors [B, S, H, D]")


def attn_fwd(q, k, v, causal=False, scale=0.0, out=None, lse=None, want_lse=True, stream=None):
    """O (bf16) and lse (fp32 [B, H, S], or None) for bf16 or E4M3 q, k, v.

    E4M3 inputs (torch.float8_e4m3fn or uint8) are taken with unit scales.
    """
    _check4(q, k, v)
    B, S, H, D = q.shape
    dtype = ATTN_FP8_E4M3 if q.element_size() == 1 else ATTN_BF16
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    _lib.call("attn_fwd", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, D,
              int(bool(causal)), float(scale), dtype, _stream(stream))
    return out, lse


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=0.0, out=None,
                 lse=None, want_lse=True, stream=None):
    """O (bf16) and lse for E4M3 inputs with per-(b, h, 128-token block) fp32 scales."""
    _check4(q8, k8, v8)
    B, S, H, D = q8.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q8.device)
    _lib.call("attn_fwd_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale),
              _ptr(v_scale), _ptr(out), _ptr(lse), B, H, S, D, int(bool(causal)), float(scale),
              _stream(stream))
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen=None, causal=False, scale=0.0, out=None, lse=None,
                    want_lse=True, stream=None):
    """Attention over a packed batch: q, k, v bf16 [total, H, D]; cu_seqlens int32 CUDA
    tensor [n_seq + 1]; max_seqlen bounds every sequence's length (None: read it from
    cu_seqlens, which synchronises).  Returns (o [total, H, D] bf16, lse [H, total] fp32 or
    None)."""
    for t in (q, k, v):
        if t.dim() != 3 or not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors [total, H, D]")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    total, H, D = q.shape
    if max_seqlen is None:
        max_seqlen = max(1, int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()))
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    _lib.call("attn_fwd_varlen", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
              int(cu_seqlens.numel() - 1), total, int(max_seqlen), H, D, int(bool(causal)), float(scale),
              _stream(stream))
    return out, lse


def _check_cu(cu_seqlens):
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")


def varlen_scale_blocks(total, n_seq):
    """Scale entries per head of a packed batch's block scales: total // 128 + n_seq + 1."""
    return int(_lib.load().attn_varlen_scale_blocks(int(total), int(n_seq)))


def hadamard_rotate_quant_fp8_varlen(x, cu_seqlens, signs=None, out=None, scale=None, stream=None):
    """E4M3 codes (uint8 [total, H, D]) and block scales (fp32 [H, varlen_scale_blocks]) of a
    packed bf16 batch x [total, H, D]; the blocks restart at every sequence's first token."""
    if x.dim() != 3 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [total, H, D]")
    _check_cu(cu_seqlens)
    total, H, D = x.shape
    n_seq = int(cu_seqlens.numel() - 1)
    if out is None:
        out = torch.empty((total, H, D), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((H, varlen_scale_blocks(total, n_seq)), dtype=torch.float32, device=x.device)
    _lib.call("hadamard_rotate_quant_fp8_varlen", _ptr(x), _ptr(out), _ptr(scale), _ptr(signs), _ptr(cu_seqlens),
              n_seq, total, H, D, _stream(stream))
    return out, scale


def rope_hadamard_rotate_quant_fp8_varlen(x, rope_cs, cu_seqlens, signs=None, out=None, scale=None, stream=None):
    """Rotary embedding (positions restarting at every sequence), then
    ``hadamard_rotate_quant_fp8_varlen``, in one kernel.  ``rope_cs``: a table from
    ``rope_cos_sin_table`` with at least 128 * ceil(len / 128) rows for the longest sequence."""
    if x.dim() != 3 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [total, H, D]")
    _check_cu(cu_seqlens)
    total, H, D = x.shape
    n_seq = int(cu_seqlens.numel() - 1)
    if out is None:
        out = torch.empty((total, H, D), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((H, varlen_scale_blocks(total, n_seq)), dtype=torch.float32, device=x.device)
    _lib.call("rope_hadamard_rotate_quant_fp8_varlen", _ptr(x), _ptr(rope_cs), int(rope_cs.shape[0]), _ptr(out),
              _ptr(scale), _ptr(signs), _ptr(cu_seqlens), n_seq, total, H, D, _stream(stream))
    return out, scale


def attn_fwd_varlen_fp8(q8, k8, v8, q_scale, k_scale, v_scale, cu_seqlens, max_seqlen=None, causal=False,
                        scale=0.0, out=None, lse=None, want_lse=True, stream=None):
    """attn_fwd_varlen on E4M3 codes [total, H, D] with the block scales of
    hadamard_rotate_quant_fp8_varlen -> (o [total, H, D] bf16, lse [H, total] fp32 or None)."""
    for t in (q8, k8, v8):
        if t.dim() != 3 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q8, k8, v8 must be contiguous CUDA tensors [total, H, D]")
    _check_cu(cu_seqlens)
    total, H, D = q8.shape
    if max_seqlen is None:
        max_seqlen = max(1, int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()))
    if out is None:
        out = torch.empty((total, H, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((H, total), dtype=torch.float32, device=q8.device)
    _lib.call("attn_fwd_varlen_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), _ptr(cu_seqlens), int(cu_seqlens.numel() - 1), total, int(max_seqlen), H, D,
              int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_fwd_gqa(q, k, v, causal=False, scale=0.0, out=None, lse=None, want_lse=True, stream=None):
    """Grouped-query attention: q [B, S, Hq, D], k, v [B, S, Hkv, D] bf16 -> (o, lse [B, Hq, S])."""
    _check4(q, k, v)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _lib.call("attn_fwd_gqa", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D,
              int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_fwd_gqa_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=0.0, out=None, lse=None,
                     want_lse=True, stream=None):
    """Grouped-query attention on E4M3 codes: q8 [B, S, Hq, D], k8, v8 [B, S, Hkv, D] with fp32
    block scales [B, Hq, ceil(S/128)] and [B, Hkv, ceil(S/128)] -> (o bf16, lse [B, Hq, S])."""
    _check4(q8, k8, v8)
    B, S, Hq, D = q8.shape
    Hkv = k8.shape[2]
    if out is None:
        out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q8.device)
    _lib.call("attn_fwd_gqa_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_decode(q, k, v, causal=False, scale=0.0, out=None, lse=None, want_lse=True, workspace=None, stream=None):
    """Decoding: q [B, Sq, Hq, D] against k, v [B, Sk, Hkv, D] bf16 -> (o, lse [B, Hq, Sq])."""
    _check4(q, k, v)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    nbytes = _lib.load().attn_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.call("attn_decode", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), wsb, B, Hq, Hkv,
              Sq, Sk, D, int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_decode_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=0.0, out=None, lse=None,
                    want_lse=True, workspace=None, stream=None):
    """Decoding on E4M3 codes: q8 [B, Sq, Hq, D], k8, v8 [B, Sk, Hkv, D] (uint8 or float8_e4m3fn)
    with fp32 block scales [B, Hq, ceil(Sq/128)] and [B, Hkv, ceil(Sk/128)] -> (o bf16, lse)."""
    _check4(q8, k8, v8)
    B, Sq, Hq, D = q8.shape
    Sk, Hkv = k8.shape[1], k8.shape[2]
    nbytes = _lib.load().attn_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=q8.device)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q8.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.call("attn_decode_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), _ptr(workspace), wsb, B, Hq, Hkv, Sq, Sk, D, int(bool(causal)), float(scale),
              _stream(stream))
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, causal=False, scale=0.0, dq=None, dk=None, dv=None, workspace=None,
             stream=None):
    """Gradients (dq, dk, dv) bf16 [B, S, H, D] of attn_fwd from its output o and lse."""
    _check4(q, k, v, o, dout)
    B, S, H, D = q.shape
    nbytes = _lib.load().attn_bwd_workspace_bytes(B, H, S)
    if workspace is None:
        workspace = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _lib.call("attn_bwd", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
              _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, S, D, int(bool(causal)),
              float(scale), _stream(stream))
    return dq, dk, dv


def hadamard_rotate_quant_fp8(x, signs=None, out=None, scale=None, stream=None):
    """E4M3 codes (uint8 [B, S, H, D]) and block scales (fp32 [B, H, ceil(S/128)]) of bf16 x.

    ``signs``: fp32 CUDA tensor of D values +-1 (rotate), or None (quantise only).
    """
    _check4(x)
    B, S, H, D = x.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((B, H, block_count(S)), dtype=torch.float32, device=x.device)
    _lib.call("hadamard_rotate_quant_fp8", _ptr(x), _ptr(out), _ptr(scale), _ptr(signs), B, H, S,
              D, _stream(stream))
    return out, scale


def rope_cos_sin_table(n_pos, D, base=10000.0, device="cuda", out=None, stream=None):
    """Rotary table fp32 [n_pos, D/2, 2]: (cos, sin) of p * base^(-2i/D), built on the GPU."""
    if out is None:
        out = torch.empty((n_pos, D // 2, 2), dtype=torch.float32, device=device)
    _lib.call("rope_cos_sin_table", _ptr(out), int(n_pos), int(D), float(base), _stream(stream))
    return out


def rope_hadamard_rotate_quant_fp8(x, rope_cs, signs=None, out=None, scale=None, stream=None):
    """Rotary embedding, then ``hadamard_rotate_quant_fp8``, in one kernel.

    ``rope_cs``: the table from ``rope_cos_sin_table`` with at least 128 * ceil(S/128) rows.
    """
    _check4(x)
    B, S, H, D = x.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((B, H, block_count(S)), dtype=torch.float32, device=x.device)
    _lib.call("rope_hadamard_rotate_quant_fp8", _ptr(x), _ptr(rope_cs), int(rope_cs.shape[0]), _ptr(out),
              _ptr(scale), _ptr(signs), B, H, S, D, _stream(stream))
    return out, scale


def check(stream=None):
    """Synchronise the stream and raise AttnError if a kernel's bounded wait ran out."""
    _lib.call("attn_check", _stream(stream))


def set_spin_limit(cycles):
    _lib.load().attn_set_spin_limit(int(cycles))


def selftest_bounded_wait(cycles, stream=None):
    _lib.call("attn_selftest_bounded_wait", int(cycles), _stream(stream))
