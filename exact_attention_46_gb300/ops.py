"""Python binding of the attention library: torch tensors in, C-ABI calls out.

Argument marshalling only -- every step of the computation runs in the CUDA
kernels behind include/attn46.h.  torch supplies device memory and the current
stream.  Each function checks its tensors (type, dtype, shape, contiguity, one
CUDA device) before it calls the library, which checks sizes, alignment and
overlaps again and launches nothing on a bad argument.
"""

import torch

from . import _lib

__all__ = ["attn_fwd", "attn_fwd_fp8", "attn_fwd_varlen", "attn_fwd_varlen_fp8", "attn_fwd_gqa",
           "attn_fwd_gqa_fp8", "attn_decode", "attn_decode_fp8", "attn_bwd", "attn_bwd_gqa",
           "hadamard_rotate_quant_fp8",
           "hadamard_rotate_quant_fp8_varlen", "rope_cos_sin_table", "rope_hadamard_rotate_quant_fp8",
           "rope_hadamard_rotate_quant_fp8_varlen", "varlen_scale_blocks", "block_count", "check",
           "set_spin_limit", "set_key_split", "key_split_plan", "attn_fwd_split", "split_workspace_bytes",
           "selftest_bounded_wait", "ATTN_BF16", "ATTN_FP8_E4M3"]

ATTN_BF16 = 0
ATTN_FP8_E4M3 = 1
TOKEN_BLOCK = 128

_BF16 = (torch.bfloat16,)
_CODES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())
_F32 = (torch.float32,)
_I32 = (torch.int32,)


def block_count(S):
    """Number of 128-token scale blocks for sequence length S."""
    return (S + TOKEN_BLOCK - 1) // TOKEN_BLOCK


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _arg(t, name, dtypes, shape=None, dim=None, device=None):
    """Check one tensor argument: dtype, rank or exact shape, contiguity, a CUDA device (the
    one of the other arguments when given).  Returns t."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected " + " or ".join(str(d) for d in dtypes))
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name}: expected {dim} dimensions, got shape {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other arguments on {device}")
    return t


def _opt(t, *args, **kwargs):
    return None if t is None else _arg(t, *args, **kwargs)


def _inputs(names, ts, dtypes, dim):
    """q, k, v-like inputs: same dtype family and rank, one device; returns that device."""
    dev = None
    for n, t in zip(names, ts):
        _arg(t, n, dtypes, dim=dim, device=dev)
        dev = t.device
    if len({t.dtype for t in ts}) != 1:
        raise ValueError(f"{', '.join(names)} must share one dtype")
    return dev


def attn_fwd(q, k, v, causal=False, scale=0.0, out=None, lse=None, want_lse=True, stream=None):
    """O (bf16) and lse (fp32 [B, H, S], or None) for bf16 or E4M3 q, k, v.

    E4M3 inputs (torch.float8_e4m3fn or uint8) are taken with unit scales.
    """
    dev = _inputs(("q", "k", "v"), (q, k, v), _BF16 + _CODES, 4)
    B, S, H, D = q.shape
    for n, t in (("k", k), ("v", v)):
        _arg(t, n, (q.dtype,), shape=q.shape)
    dtype = ATTN_FP8_E4M3 if q.element_size() == 1 else ATTN_BF16
    _opt(out, "out", _BF16, shape=(B, S, H, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, H, S), device=dev)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    _lib.call("attn_fwd", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, D,
              int(bool(causal)), float(scale), dtype, _stream(stream))
    return out, lse


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=0.0, out=None,
                 lse=None, want_lse=True, stream=None):
    """O (bf16) and lse for E4M3 inputs with per-(b, h, 128-token block) fp32 scales."""
    dev = _inputs(("q8", "k8", "v8"), (q8, k8, v8), _CODES, 4)
    B, S, H, D = q8.shape
    for n, t in (("k8", k8), ("v8", v8)):
        _arg(t, n, _CODES, shape=q8.shape)
    for n, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _arg(t, n, _F32, shape=(B, H, block_count(S)), device=dev)
    _opt(out, "out", _BF16, shape=(B, S, H, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, H, S), device=dev)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
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
    dev = _inputs(("q", "k", "v"), (q, k, v), _BF16, 3)
    total, H, D = q.shape
    for n, t in (("k", k), ("v", v)):
        _arg(t, n, _BF16, shape=q.shape)
    _arg(cu_seqlens, "cu_seqlens", _I32, dim=1, device=dev)
    _opt(out, "out", _BF16, shape=(total, H, D), device=dev)
    _opt(lse, "lse", _F32, shape=(H, total), device=dev)
    if max_seqlen is None:
        max_seqlen = max(1, int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()))
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((H, total), dtype=torch.float32, device=dev)
    _lib.call("attn_fwd_varlen", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
              int(cu_seqlens.numel() - 1), total, int(max_seqlen), H, D, int(bool(causal)), float(scale),
              _stream(stream))
    return out, lse


def varlen_scale_blocks(total, n_seq):
    """Scale entries per head of a packed batch's block scales: total // 128 + n_seq + 1."""
    return int(_lib.load().attn_varlen_scale_blocks(int(total), int(n_seq)))


def hadamard_rotate_quant_fp8_varlen(x, cu_seqlens, signs=None, out=None, scale=None, stream=None):
    """E4M3 codes (uint8 [total, H, D]) and block scales (fp32 [H, varlen_scale_blocks]) of a
    packed bf16 batch x [total, H, D]; the blocks restart at every sequence's first token."""
    dev = _arg(x, "x", _BF16, dim=3).device
    total, H, D = x.shape
    _arg(cu_seqlens, "cu_seqlens", _I32, dim=1, device=dev)
    _opt(signs, "signs", _F32, shape=(D,), device=dev)
    n_seq = int(cu_seqlens.numel() - 1)
    nb = varlen_scale_blocks(total, n_seq)
    _opt(out, "out", _CODES, shape=(total, H, D), device=dev)
    _opt(scale, "scale", _F32, shape=(H, nb), device=dev)
    if out is None:
        out = torch.empty((total, H, D), dtype=torch.uint8, device=dev)
    if scale is None:
        scale = torch.empty((H, nb), dtype=torch.float32, device=dev)
    _lib.call("hadamard_rotate_quant_fp8_varlen", _ptr(x), _ptr(out), _ptr(scale), _ptr(signs), _ptr(cu_seqlens),
              n_seq, total, H, D, _stream(stream))
    return out, scale


def rope_hadamard_rotate_quant_fp8_varlen(x, rope_cs, cu_seqlens, signs=None, out=None, scale=None, stream=None):
    """Rotary embedding (positions restarting at every sequence), then
    ``hadamard_rotate_quant_fp8_varlen``, in one kernel.  ``rope_cs``: a table from
    ``rope_cos_sin_table`` with at least 128 * ceil(len / 128) rows for the longest sequence."""
    dev = _arg(x, "x", _BF16, dim=3).device
    total, H, D = x.shape
    _arg(rope_cs, "rope_cs", _F32, dim=3, device=dev)
    if tuple(rope_cs.shape[1:]) != (D // 2, 2):
        raise ValueError(f"rope_cs: expected shape (n_pos, {D // 2}, 2), got {tuple(rope_cs.shape)}")
    _arg(cu_seqlens, "cu_seqlens", _I32, dim=1, device=dev)
    _opt(signs, "signs", _F32, shape=(D,), device=dev)
    n_seq = int(cu_seqlens.numel() - 1)
    nb = varlen_scale_blocks(total, n_seq)
    _opt(out, "out", _CODES, shape=(total, H, D), device=dev)
    _opt(scale, "scale", _F32, shape=(H, nb), device=dev)
    if out is None:
        out = torch.empty((total, H, D), dtype=torch.uint8, device=dev)
    if scale is None:
        scale = torch.empty((H, nb), dtype=torch.float32, device=dev)
    _lib.call("rope_hadamard_rotate_quant_fp8_varlen", _ptr(x), _ptr(rope_cs), int(rope_cs.shape[0]), _ptr(out),
              _ptr(scale), _ptr(signs), _ptr(cu_seqlens), n_seq, total, H, D, _stream(stream))
    return out, scale


def attn_fwd_varlen_fp8(q8, k8, v8, q_scale, k_scale, v_scale, cu_seqlens, max_seqlen=None, causal=False,
                        scale=0.0, out=None, lse=None, want_lse=True, stream=None):
    """attn_fwd_varlen on E4M3 codes [total, H, D] with the block scales of
    hadamard_rotate_quant_fp8_varlen -> (o [total, H, D] bf16, lse [H, total] fp32 or None)."""
    dev = _inputs(("q8", "k8", "v8"), (q8, k8, v8), _CODES, 3)
    total, H, D = q8.shape
    for n, t in (("k8", k8), ("v8", v8)):
        _arg(t, n, _CODES, shape=q8.shape)
    _arg(cu_seqlens, "cu_seqlens", _I32, dim=1, device=dev)
    nb = varlen_scale_blocks(total, int(cu_seqlens.numel() - 1))
    for n, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _arg(t, n, _F32, shape=(H, nb), device=dev)
    _opt(out, "out", _BF16, shape=(total, H, D), device=dev)
    _opt(lse, "lse", _F32, shape=(H, total), device=dev)
    if max_seqlen is None:
        max_seqlen = max(1, int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()))
    if out is None:
        out = torch.empty((total, H, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((H, total), dtype=torch.float32, device=dev)
    _lib.call("attn_fwd_varlen_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), _ptr(cu_seqlens), int(cu_seqlens.numel() - 1), total, int(max_seqlen), H, D,
              int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_fwd_gqa(q, k, v, causal=False, scale=0.0, out=None, lse=None, want_lse=True, stream=None):
    """Grouped-query attention: q [B, S, Hq, D], k, v [B, S, Hkv, D] bf16 -> (o, lse [B, Hq, S])."""
    dev = _inputs(("q", "k", "v"), (q, k, v), _BF16, 4)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    for n, t in (("k", k), ("v", v)):
        _arg(t, n, _BF16, shape=(B, S, Hkv, D))
    _opt(out, "out", _BF16, shape=(B, S, Hq, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, Hq, S), device=dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    _lib.call("attn_fwd_gqa", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D,
              int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_fwd_gqa_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=0.0, out=None, lse=None,
                     want_lse=True, stream=None):
    """Grouped-query attention on E4M3 codes: q8 [B, S, Hq, D], k8, v8 [B, S, Hkv, D] with fp32
    block scales [B, Hq, ceil(S/128)] and [B, Hkv, ceil(S/128)] -> (o bf16, lse [B, Hq, S])."""
    dev = _inputs(("q8", "k8", "v8"), (q8, k8, v8), _CODES, 4)
    B, S, Hq, D = q8.shape
    Hkv = k8.shape[2]
    for n, t in (("k8", k8), ("v8", v8)):
        _arg(t, n, _CODES, shape=(B, S, Hkv, D))
    _arg(q_scale, "q_scale", _F32, shape=(B, Hq, block_count(S)), device=dev)
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _arg(t, n, _F32, shape=(B, Hkv, block_count(S)), device=dev)
    _opt(out, "out", _BF16, shape=(B, S, Hq, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, Hq, S), device=dev)
    if out is None:
        out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    _lib.call("attn_fwd_gqa_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_decode(q, k, v, causal=False, scale=0.0, out=None, lse=None, want_lse=True, workspace=None, stream=None):
    """Decoding: q [B, Sq, Hq, D] against k, v [B, Sk, Hkv, D] bf16 -> (o, lse [B, Hq, Sq])."""
    dev = _inputs(("q", "k", "v"), (q, k, v), _BF16, 4)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    _arg(v, "v", _BF16, shape=k.shape)
    _opt(out, "out", _BF16, shape=(B, Sq, Hq, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, Hq, Sq), device=dev)
    _opt(workspace, "workspace", _F32, dim=1, device=dev)
    nbytes = _lib.load().attn_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.call("attn_decode", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), wsb, B, Hq, Hkv,
              Sq, Sk, D, int(bool(causal)), float(scale), _stream(stream))
    return out, lse


def attn_decode_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=0.0, out=None, lse=None,
                    want_lse=True, workspace=None, stream=None):
    """Decoding on E4M3 codes: q8 [B, Sq, Hq, D], k8, v8 [B, Sk, Hkv, D] (uint8 or float8_e4m3fn)
    with fp32 block scales [B, Hq, ceil(Sq/128)] and [B, Hkv, ceil(Sk/128)] -> (o bf16, lse)."""
    dev = _inputs(("q8", "k8", "v8"), (q8, k8, v8), _CODES, 4)
    B, Sq, Hq, D = q8.shape
    Sk, Hkv = k8.shape[1], k8.shape[2]
    _arg(v8, "v8", _CODES, shape=k8.shape)
    _arg(q_scale, "q_scale", _F32, shape=(B, Hq, block_count(Sq)), device=dev)
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _arg(t, n, _F32, shape=(B, Hkv, block_count(Sk)), device=dev)
    _opt(out, "out", _BF16, shape=(B, Sq, Hq, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, Hq, Sq), device=dev)
    _opt(workspace, "workspace", _F32, dim=1, device=dev)
    nbytes = _lib.load().attn_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.call("attn_decode_fp8", _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), _ptr(workspace), wsb, B, Hq, Hkv, Sq, Sk, D, int(bool(causal)), float(scale),
              _stream(stream))
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, causal=False, scale=0.0, dq=None, dk=None, dv=None, workspace=None,
             stream=None):
    """Gradients (dq, dk, dv) bf16 [B, S, H, D] of attn_fwd from its output o and lse."""
    dev = _inputs(("q", "k", "v", "o", "dout"), (q, k, v, o, dout), _BF16, 4)
    B, S, H, D = q.shape
    for n, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _arg(t, n, _BF16, shape=q.shape)
    _arg(lse, "lse", _F32, shape=(B, H, S), device=dev)
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _opt(t, n, _BF16, shape=q.shape, device=dev)
    _opt(workspace, "workspace", _F32, dim=1, device=dev)
    nbytes = _lib.load().attn_bwd_workspace_bytes(B, H, S)
    if workspace is None:
        workspace = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _lib.call("attn_bwd", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
              _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, S, D, int(bool(causal)),
              float(scale), _stream(stream))
    return dq, dk, dv


def attn_bwd_gqa(q, k, v, o, lse, dout, causal=False, scale=0.0, dq=None, dk=None, dv=None, workspace=None,
                 stream=None):
    """Gradients of attn_fwd_gqa: dq bf16 [B, S, Hq, D]; dk, dv bf16 [B, S, Hkv, D], summed over each group."""
    dev = _inputs(("q", "k", "v", "o", "dout"), (q, k, v, o, dout), _BF16, 4)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    for n, t in (("k", k), ("v", v)):
        _arg(t, n, _BF16, shape=(B, S, Hkv, D))
    for n, t in (("o", o), ("dout", dout)):
        _arg(t, n, _BF16, shape=q.shape)
    _arg(lse, "lse", _F32, shape=(B, Hq, S), device=dev)
    _opt(dq, "dq", _BF16, shape=q.shape, device=dev)
    for n, t in (("dk", dk), ("dv", dv)):
        _opt(t, n, _BF16, shape=k.shape, device=dev)
    _opt(workspace, "workspace", _F32, dim=1, device=dev)
    nbytes = _lib.load().attn_bwd_workspace_bytes(B, Hq, S)
    if workspace is None:
        workspace = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _lib.call("attn_bwd_gqa", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
              _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, Hq, Hkv, S, D,
              int(bool(causal)), float(scale), _stream(stream))
    return dq, dk, dv


def hadamard_rotate_quant_fp8(x, signs=None, out=None, scale=None, stream=None):
    """E4M3 codes (uint8 [B, S, H, D]) and block scales (fp32 [B, H, ceil(S/128)]) of bf16 x.

    ``signs``: fp32 CUDA tensor of D values +-1 (rotate), or None (quantise only).
    """
    dev = _arg(x, "x", _BF16, dim=4).device
    B, S, H, D = x.shape
    _opt(signs, "signs", _F32, shape=(D,), device=dev)
    _opt(out, "out", _CODES, shape=(B, S, H, D), device=dev)
    _opt(scale, "scale", _F32, shape=(B, H, block_count(S)), device=dev)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.uint8, device=dev)
    if scale is None:
        scale = torch.empty((B, H, block_count(S)), dtype=torch.float32, device=dev)
    _lib.call("hadamard_rotate_quant_fp8", _ptr(x), _ptr(out), _ptr(scale), _ptr(signs), B, H, S,
              D, _stream(stream))
    return out, scale


def hadamard_rotate_quant_fp8_qkv(q, k, v, signs=None, out=None, scale=None, stream=None):
    """``hadamard_rotate_quant_fp8`` of q and k (rotated by ``signs``) and of v (not rotated), in one
    launch.  Returns (q8, q_scale, k8, k_scale, v8, v_scale); bitwise what three separate calls give.
    ``out`` / ``scale``: optional sequences of three preallocated code / scale tensors (q, k, v).
    """
    dev = _arg(q, "q", _BF16, dim=4).device
    B, S, H, D = q.shape
    _arg(k, "k", _BF16, shape=(B, S, H, D), device=dev)
    _arg(v, "v", _BF16, shape=(B, S, H, D), device=dev)
    _opt(signs, "signs", _F32, shape=(D,), device=dev)
    codes = list(out) if out is not None else [None] * 3
    scales = list(scale) if scale is not None else [None] * 3
    if len(codes) != 3 or len(scales) != 3:
        raise ValueError("out and scale take three tensors each (q, k, v)")
    for i, n in enumerate("qkv"):
        _opt(codes[i], n + "8", _CODES, shape=(B, S, H, D), device=dev)
        _opt(scales[i], n + "_scale", _F32, shape=(B, H, block_count(S)), device=dev)
        if codes[i] is None:
            codes[i] = torch.empty((B, S, H, D), dtype=torch.uint8, device=dev)
        if scales[i] is None:
            scales[i] = torch.empty((B, H, block_count(S)), dtype=torch.float32, device=dev)
    _lib.call("hadamard_rotate_quant_fp8_qkv", _ptr(q), _ptr(k), _ptr(v), *[_ptr(c) for c in codes],
              *[_ptr(s_) for s_ in scales], _ptr(signs), B, H, S, D, _stream(stream))
    return codes[0], scales[0], codes[1], scales[1], codes[2], scales[2]


def rope_cos_sin_table(n_pos, D, base=10000.0, device="cuda", out=None, stream=None):
    """Rotary table fp32 [n_pos, D/2, 2]: (cos, sin) of p * base^(-2i/D), built on the GPU."""
    _opt(out, "out", _F32, shape=(n_pos, D // 2, 2))
    if out is None:
        out = torch.empty((n_pos, D // 2, 2), dtype=torch.float32, device=device)
    _lib.call("rope_cos_sin_table", _ptr(out), int(n_pos), int(D), float(base), _stream(stream))
    return out


def rope_hadamard_rotate_quant_fp8(x, rope_cs, signs=None, out=None, scale=None, stream=None):
    """Rotary embedding, then ``hadamard_rotate_quant_fp8``, in one kernel.

    ``rope_cs``: the table from ``rope_cos_sin_table`` with at least 128 * ceil(S/128) rows.
    """
    dev = _arg(x, "x", _BF16, dim=4).device
    B, S, H, D = x.shape
    _arg(rope_cs, "rope_cs", _F32, dim=3, device=dev)
    if tuple(rope_cs.shape[1:]) != (D // 2, 2):
        raise ValueError(f"rope_cs: expected shape (n_pos, {D // 2}, 2), got {tuple(rope_cs.shape)}")
    _opt(signs, "signs", _F32, shape=(D,), device=dev)
    _opt(out, "out", _CODES, shape=(B, S, H, D), device=dev)
    _opt(scale, "scale", _F32, shape=(B, H, block_count(S)), device=dev)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.uint8, device=dev)
    if scale is None:
        scale = torch.empty((B, H, block_count(S)), dtype=torch.float32, device=dev)
    _lib.call("rope_hadamard_rotate_quant_fp8", _ptr(x), _ptr(rope_cs), int(rope_cs.shape[0]), _ptr(out),
              _ptr(scale), _ptr(signs), B, H, S, D, _stream(stream))
    return out, scale


def check(stream=None):
    """Synchronise the stream and raise AttnError if a kernel's bounded wait ran out."""
    _lib.call("attn_check", _stream(stream))


def set_spin_limit(cycles):
    _lib.load().attn_set_spin_limit(int(cycles))


def set_key_split(max_parts):
    """Most key ranges a block of the last, partly filled round of a non-causal forward is cut
    into (1 = no split; default 4)."""
    _lib.load().attn_set_key_split(int(max_parts))


def key_split_plan(n_items, sms, key_tiles, max_parts=4):
    """(blocks run whole, blocks cut, ranges per cut block) for a non-causal forward; host only."""
    import ctypes
    out = (ctypes.c_longlong * 3)()
    _lib.call("attn_key_split_plan", int(n_items), int(sms), int(key_tiles), int(max_parts), ctypes.addressof(out))
    return tuple(int(x) for x in out)


def split_workspace_bytes(B, Hq, S, D, causal=False):
    """Bytes of workspace attn_fwd_split needs for this shape on the current device (0: no split)."""
    return int(_lib.load().attn_fwd_split_workspace_bytes(int(B), int(Hq), int(S), int(D), int(bool(causal))))


def attn_fwd_split(q, k, v, q_scale=None, k_scale=None, v_scale=None, causal=False, scale=0.0, out=None,
                   lse=None, want_lse=True, workspace=None, stream=None):
    """attn_fwd / attn_fwd_fp8 / attn_fwd_gqa(_fp8) with a workspace for the key-split tail.

    q [B, S, Hq, D], k, v [B, S, Hkv, D]: bf16, or E4M3 codes with all three block-scale arrays
    (or none: unit scales).  ``workspace``: a CUDA tensor of at least split_workspace_bytes(...)
    bytes, or None to allocate one here (torch's allocator) when the plan splits; an explicit
    empty tensor runs unsplit."""
    dev = _inputs(("q", "k", "v"), (q, k, v), _BF16 + _CODES, 4)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    for n, t in (("k", k), ("v", v)):
        _arg(t, n, (q.dtype,), shape=(B, S, Hkv, D))
    fp8 = q.element_size() == 1
    scales = (q_scale, k_scale, v_scale)
    if any(s is not None for s in scales):
        if not fp8 or any(s is None for s in scales):
            raise ValueError("block scales go with E4M3 inputs, all three or none")
        _arg(q_scale, "q_scale", _F32, shape=(B, Hq, block_count(S)), device=dev)
        for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
            _arg(t, n, _F32, shape=(B, Hkv, block_count(S)), device=dev)
    _opt(out, "out", _BF16, shape=(B, S, Hq, D), device=dev)
    _opt(lse, "lse", _F32, shape=(B, Hq, S), device=dev)
    if out is None:
        out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    if workspace is None:
        need = split_workspace_bytes(B, Hq, S, D, causal)
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev) if need else None
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _arg(workspace, "workspace", (workspace.dtype,), device=dev)
        ws_ptr, ws_bytes = (_ptr(workspace), workspace.numel() * workspace.element_size()) if workspace.numel() else (None, 0)
    _lib.call("attn_fwd_split", _ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
              _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, int(bool(causal)), float(scale),
              ATTN_FP8_E4M3 if fp8 else ATTN_BF16, ws_ptr, ws_bytes, _stream(stream))
    return out, lse


def selftest_bounded_wait(cycles, stream=None):
    _lib.call("attn_selftest_bounded_wait", int(cycles), _stream(stream))
