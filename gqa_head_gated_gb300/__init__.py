"""gqa_head_gated_gb300: gated causal GQA attention at head_dim 256 for GB300.

Thin PyTorch binding over the C ABI of libgqa_attn.so (include/gqa_attn.h).
It only checks and marshals arguments (pointers, sizes, the current CUDA
stream) and allocates outputs with torch; every step of the computation runs in
the library's CUDA kernels.  There is no CPU fallback: without the shared
library or a CUDA device the calls raise.  Every attention call takes bf16 or
fp16 tensors (one type per call) and picks the matching entry point.

    out = softmax(Q K^T / 16 + causal/offset mask) V * sigmoid(G)
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import GqaError, check, load  # noqa: F401

HEAD_DIM = 256

__all__ = ["prefill", "prefill_pair", "masked", "decode", "verify_tree", "kv_append", "kv_keep", "decode_plan", "decode_split", "lse_merge",
           "decode_workspace_size", "last_device_status", "set_wait_timeout_ns",
           "selftest_wait_timeout", "decode_noalloc", "launch_log", "GqaError",
           "load"]


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_ELEM = {torch.bfloat16: "", torch.float16: "_f16"}


def _elem(t, name):
    """Entry-point suffix for the element type of `t` (bf16 or fp16)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in _ELEM:
        raise TypeError(f"{name} must be bfloat16 or float16, got {t.dtype}")
    return _ELEM[t.dtype]


def _need(t, dtype, ndim, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or t.shape[-1] != HEAD_DIM and ndim >= 3:
        raise ValueError(f"{name} must be {ndim}-d with last dim {HEAD_DIM}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def prefill(q, k, v, g=None, kv_offset=0, out=None, return_lse=False):
    """Prompt rows.  q, g: [B,Hq,Lq,256] bf16; k, v: [B,Hkv,Lkv,256] bf16.
    Row i sits at position kv_offset + i and sees keys 0..kv_offset+i.
    Returns out [B,Hq,Lq,256] bf16 (and lse [B,Hq,Lq] fp32 if return_lse).
    fp16 inputs run the fp16 kernels and give an fp16 out."""
    sfx = _elem(q, "q")
    _need(q, q.dtype, 4, "q")
    _need(k, q.dtype, 4, "k")
    _need(v, q.dtype, 4, "v")
    if g is not None:
        _need(g, q.dtype, 4, "g")
    B, Hq, Lq, _ = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device) if return_lse else None
    _need(out, q.dtype, 4, "out")
    fn = getattr(load(), "gqa_attn_prefill" + sfx)
    code = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), _ptr(lse), B, Hq, Hkv, Lq, Lkv,
              int(kv_offset), _stream())
    check(code, "gqa_attn_prefill" + sfx)
    return (out, lse) if return_lse else out


def prefill_pair(q, k, v, g=None, kv_offset=0, out=None, return_lse=False):
    """prefill() through gqa_attn_prefill_pair (CTA pairs sharing each K/V tile);
    bf16 only."""
    if q.dtype != torch.bfloat16:
        raise TypeError("prefill_pair takes bf16 inputs")
    _need(q, q.dtype, 4, "q")
    _need(k, q.dtype, 4, "k")
    _need(v, q.dtype, 4, "v")
    if g is not None:
        _need(g, q.dtype, 4, "g")
    B, Hq, Lq, _ = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device) if return_lse else None
    _need(out, q.dtype, 4, "out")
    code = load().gqa_attn_prefill_pair(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), _ptr(lse),
                                        B, Hq, Hkv, Lq, Lkv, int(kv_offset), _stream())
    check(code, "gqa_attn_prefill_pair")
    return (out, lse) if return_lse else out


_MASK_KIND = {torch.bool: 1, torch.float32: 2, torch.bfloat16: 3, torch.float16: 4}


def masked(q, k, v, g=None, mask=None, causal=False, kv_offset=None, head_chunking=True,
           out=None, return_lse=False):
    """Gated attention with a general mask (the dense SDPA consumer's masks).

    q, g: [B,Hq,Lq,256]; k, v: [B,Hkv,Lkv,256]; bf16 or fp16.  mask: None, a bool
    tensor (True = attend) or a float32 / bf16 / fp16 tensor added to the scaled
    scores, of up to 4 dims broadcasting (trailing dims aligned) to [B, heads, Lq,
    Lkv]; any strides.  The head rule: with head_chunking, Lq <= 32 and Lq*GQA > 32
    the mask's head count must be 1 or the chunk size min(GQA, 32 // Lq) with no
    remainder chunk (chunk-local); otherwise 1 or Hq.  A mask that does not
    broadcast raises GqaError (GQA_ERR_INVALID_ARG) and launches nothing.
    causal: also hide keys j > kv_offset + i (kv_offset defaults to Lkv - Lq)."""
    sfx = _elem(q, "q")
    _need(q, q.dtype, 4, "q")
    _need(k, q.dtype, 4, "k")
    _need(v, q.dtype, 4, "v")
    if g is not None:
        _need(g, q.dtype, 4, "g")
    B, Hq, Lq, _ = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if kv_offset is None:
        kv_offset = Lkv - Lq
    kind, mptr = 0, None
    shape = (ctypes.c_longlong * 4)(1, 1, 1, 1)
    strides = (ctypes.c_longlong * 4)(0, 0, 0, 0)
    if mask is not None:
        if not isinstance(mask, torch.Tensor) or mask.dtype not in _MASK_KIND:
            raise TypeError("mask must be a bool, float32, bfloat16 or float16 tensor")
        if not mask.is_cuda:
            raise ValueError("mask must be a CUDA tensor")
        if mask.dim() > 4:
            raise GqaError(1, "gqa_attn_masked: mask has more than 4 dimensions")
        pad = 4 - mask.dim()
        for d in range(4):
            if d >= pad:
                shape[d] = mask.shape[d - pad]
                strides[d] = mask.stride(d - pad)
        kind, mptr = _MASK_KIND[mask.dtype], _ptr(mask)
    if out is None:
        out = torch.empty_like(q)
    _need(out, q.dtype, 4, "out")
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device) if return_lse else None
    fn = getattr(load(), "gqa_attn_masked" + sfx)
    code = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), mptr, kind, shape, strides, _ptr(out),
              _ptr(lse), B, Hq, Hkv, Lq, Lkv, int(bool(causal)), int(kv_offset),
              int(bool(head_chunking)), _stream())
    check(code, "gqa_attn_masked" + sfx)
    return (out, lse) if return_lse else out


def decode_plan(B, T, Hq, Hkv, max_rows, max_kv_len):
    """(num_splits, split_keys) that decode() uses for these sizes."""
    s, c = ctypes.c_int(0), ctypes.c_int(0)
    check(load().gqa_attn_decode_plan(B, T, Hq, Hkv, max_rows, max_kv_len, ctypes.byref(s),
                                      ctypes.byref(c)), "gqa_attn_decode_plan")
    return s.value, c.value


def decode_workspace_size(B, T, Hq, Hkv, max_rows, max_kv_len):
    return int(load().gqa_attn_decode_workspace_size(B, T, Hq, Hkv, max_rows, max_kv_len))


def _decode_sizes(q, k_cache, kv_lens, cu_rows, max_rows, max_kv_len):
    T, Hq, _ = q.shape
    B, Hkv, Lcap, _ = k_cache.shape
    if kv_lens.dtype != torch.int32 or not kv_lens.is_cuda or kv_lens.numel() != B:
        raise ValueError("kv_lens must be an int32 CUDA tensor of B entries")
    if cu_rows is not None and (cu_rows.dtype != torch.int32 or not cu_rows.is_cuda
                                or cu_rows.numel() != B + 1):
        raise ValueError("cu_rows must be an int32 CUDA tensor of B+1 entries")
    if max_kv_len is None:           # synchronises; pass it to avoid the copy
        max_kv_len = int(kv_lens.max().item())
    if max_rows is None:
        max_rows = 1 if cu_rows is None else int((cu_rows[1:] - cu_rows[:-1]).max().item())
    return T, Hq, B, Hkv, Lcap, int(max_rows), int(max_kv_len)


def decode(q, k_cache, v_cache, g, kv_lens, cu_rows=None, max_rows=None, max_kv_len=None,
           workspace=None, out=None, return_lse=False):
    """Decode / chain-verify rows.  q, g: [T,Hq,256] bf16 token-major; caches
    [B,Hkv,Lcap,256] bf16; kv_lens int32 [B] (counts the new rows); cu_rows int32
    [B+1] or None (one row per sequence).  Returns out [T,Hq,256] bf16 (fp16 for
    fp16 inputs)."""
    sfx = _elem(q, "q")
    _need(q, q.dtype, 3, "q")
    _need(k_cache, q.dtype, 4, "k_cache")
    _need(v_cache, q.dtype, 4, "v_cache")
    if g is not None:
        _need(g, q.dtype, 3, "g")
    T, Hq, B, Hkv, Lcap, max_rows, max_kv_len = _decode_sizes(q, k_cache, kv_lens, cu_rows,
                                                               max_rows, max_kv_len)
    if workspace is None:    # (a given workspace is checked by the library itself)
        need = decode_workspace_size(B, T, Hq, Hkv, max_rows, max_kv_len)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    _need(out, q.dtype, 3, "out")
    fn = getattr(load(), "gqa_attn_decode" + sfx)
    code = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(g), _ptr(kv_lens), _ptr(cu_rows),
              _ptr(out), _ptr(lse), B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, _ptr(workspace),
              workspace.numel() * workspace.element_size(), _stream())
    check(code, "gqa_attn_decode" + sfx)
    return (out, lse) if return_lse else out


def decode_noalloc(q, k_cache, v_cache, g, kv_lens, cu_rows=None, max_rows=None,
                   max_kv_len=None, out=None, return_lse=False):
    """decode() through gqa_attn_decode_noalloc: the library's fixed 16 MiB area is the
    workspace (bf16 only; calls whose workspace would not fit raise GQA_ERR_WORKSPACE).
    Same kernels, plan and results as decode()."""
    if q.dtype != torch.bfloat16:
        raise TypeError("decode_noalloc takes bf16 inputs")
    _need(q, q.dtype, 3, "q")
    _need(k_cache, q.dtype, 4, "k_cache")
    _need(v_cache, q.dtype, 4, "v_cache")
    if g is not None:
        _need(g, q.dtype, 3, "g")
    T, Hq, B, Hkv, Lcap, max_rows, max_kv_len = _decode_sizes(q, k_cache, kv_lens, cu_rows,
                                                               max_rows, max_kv_len)
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    _need(out, q.dtype, 3, "out")
    code = load().gqa_attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(g),
                                          _ptr(kv_lens), _ptr(cu_rows), _ptr(out), _ptr(lse), B,
                                          T, Hq, Hkv, Lcap, max_rows, max_kv_len, _stream())
    check(code, "gqa_attn_decode_noalloc")
    return (out, lse) if return_lse else out


def launch_log(n=64):
    """The library's record of its last kernel launches (at most 64), newest first:
    dicts of kernel, seq, grid, block, dynamic_smem, as the launches used them."""
    from ._lib import LaunchInfo
    buf = (LaunchInfo * n)()
    got = load().gqa_launch_log(buf, n)
    if got < 0:
        check(-got, "gqa_launch_log")
    return [{"kernel": r.kernel.decode(), "seq": int(r.seq), "grid": int(r.grid),
             "block": int(r.block), "dynamic_smem": int(r.dynamic_smem)} for r in buf[:got]]


def verify_tree(q, k_cache, v_cache, g, kv_lens, cu_rows, tree_mask, max_rows=None,
                max_kv_len=None, workspace=None, out=None, return_lse=False):
    """Draft verify over token trees.  As decode(), plus tree_mask: int64 [T] CUDA
    tensor, one mask per new row over its sequence's new rows (bit k: new row k
    visible; its ancestors and itself).  Rows per sequence <= 64.  bf16 or fp16."""
    sfx = _elem(q, "q")
    _need(q, q.dtype, 3, "q")
    _need(k_cache, q.dtype, 4, "k_cache")
    _need(v_cache, q.dtype, 4, "v_cache")
    if g is not None:
        _need(g, q.dtype, 3, "g")
    if cu_rows is None:
        raise ValueError("cu_rows is required for tree verify")
    if (tree_mask.dtype != torch.int64 or not tree_mask.is_cuda or not tree_mask.is_contiguous()
            or tree_mask.numel() != q.shape[0]):
        raise ValueError("tree_mask must be a contiguous int64 CUDA tensor of T entries")
    T, Hq, B, Hkv, Lcap, max_rows, max_kv_len = _decode_sizes(q, k_cache, kv_lens, cu_rows,
                                                               max_rows, max_kv_len)
    need = decode_workspace_size(B, T, Hq, Hkv, max_rows, max_kv_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    _need(out, q.dtype, 3, "out")
    fn = getattr(load(), "gqa_attn_verify_tree" + sfx)
    code = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(g), _ptr(kv_lens), _ptr(cu_rows),
              _ptr(tree_mask), _ptr(out), _ptr(lse), B, T, Hq, Hkv, Lcap, max_rows, max_kv_len,
              _ptr(workspace), workspace.numel() * workspace.element_size(), _stream())
    check(code, "gqa_attn_verify_tree" + sfx)
    return (out, lse) if return_lse else out


def kv_append(k_new, v_new, kv_lens, k_cache, v_cache, cu_rows=None):
    """Writes new rows ([T,Hkv,256] bf16) after the kv_lens[b] keys each sequence
    holds in the caches ([B,Hkv,Lcap,256]); kv_lens itself is not updated.  The
    copy moves 16-bit elements: bf16 or fp16, the same type throughout."""
    _elem(k_cache, "k_cache")
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, k_cache.dtype, 3, n)
    _need(k_cache, k_cache.dtype, 4, "k_cache")
    _need(v_cache, k_cache.dtype, 4, "v_cache")
    T, Hkv, _ = k_new.shape
    B, _, Lcap, _ = k_cache.shape
    check(load().gqa_kv_append(_ptr(k_new), _ptr(v_new), _ptr(cu_rows), _ptr(kv_lens),
                               _ptr(k_cache), _ptr(v_cache), B, T, Hkv, Lcap, _stream()),
          "gqa_kv_append")


def kv_keep(k_cache, v_cache, kv_lens, cu_rows, keep_idx, cu_keep, kv_lens_out=None):
    """Moves the accepted draft rows (keep_idx, per sequence via cu_keep, strictly
    increasing draft-row indices) to the front of each sequence's draft region, in
    place; writes the new lengths into kv_lens_out when given.  bf16 or fp16."""
    _elem(k_cache, "k_cache")
    _need(k_cache, k_cache.dtype, 4, "k_cache")
    _need(v_cache, k_cache.dtype, 4, "v_cache")
    B, Hkv, Lcap, _ = k_cache.shape
    check(load().gqa_kv_keep(_ptr(k_cache), _ptr(v_cache), _ptr(kv_lens), _ptr(cu_rows),
                             _ptr(keep_idx), _ptr(cu_keep), _ptr(kv_lens_out), B, Hkv, Lcap,
                             _stream()), "gqa_kv_keep")


def decode_split(q, k_cache, v_cache, kv_lens, cu_rows=None, max_rows=None, max_kv_len=None,
                 num_splits=None, split_keys=None, o_parts=None, lse_parts=None):
    """First half of decode: partial results (O/l [S,T*Hq,256] fp32, lse [S,T*Hq]).
    bf16 or fp16 inputs.  split_keys=0 selects balanced shares with num_splits part
    slots (the one-call decode's form on the mma.sync path)."""
    sfx = _elem(q, "q")
    _need(q, q.dtype, 3, "q")
    _need(k_cache, q.dtype, 4, "k_cache")
    _need(v_cache, q.dtype, 4, "v_cache")
    T, Hq, B, Hkv, Lcap, max_rows, max_kv_len = _decode_sizes(q, k_cache, kv_lens, cu_rows,
                                                               max_rows, max_kv_len)
    if num_splits is None or split_keys is None:
        num_splits, split_keys = decode_plan(B, T, Hq, Hkv, max_rows, max_kv_len)
    if o_parts is None:
        o_parts = torch.empty((num_splits, T * Hq, HEAD_DIM), dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((num_splits, T * Hq), dtype=torch.float32, device=q.device)
    fn = getattr(load(), "gqa_attn_decode_split" + sfx)
    code = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_lens), _ptr(cu_rows), _ptr(o_parts),
              _ptr(lse_parts), B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, num_splits, split_keys,
              _stream())
    check(code, "gqa_attn_decode_split" + sfx)
    return o_parts, lse_parts


def lse_merge(o_parts, lse_parts, g=None, out=None, return_lse=False, dtype=None):
    """Merge S partial results: o_parts [S,N,256] fp32, lse_parts [S,N] fp32,
    g None or [N,256] (any shape with N*256 elements).  Returns out [N,256] in the
    element type `dtype` (bf16 or fp16; default: that of g, else of out, else bf16)."""
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise TypeError("o_parts and lse_parts must be float32")
    if not (o_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("o_parts and lse_parts must be contiguous CUDA tensors")
    S, N, D = o_parts.shape
    if D != HEAD_DIM or tuple(lse_parts.shape) != (S, N):
        raise ValueError("shapes must be [S,N,256] and [S,N]")
    if dtype is None:
        dtype = g.dtype if g is not None else out.dtype if out is not None else torch.bfloat16
    if dtype not in _ELEM:
        raise TypeError(f"dtype must be bfloat16 or float16, got {dtype}")
    sfx = _ELEM[dtype]
    if g is not None and (g.dtype != dtype or g.numel() != N * HEAD_DIM
                          or not g.is_contiguous()):
        raise ValueError(f"g must be contiguous {dtype} with N*256 elements")
    if out is None:
        out = torch.empty((N, HEAD_DIM), dtype=dtype, device=o_parts.device)
    if out.dtype != dtype or out.numel() != N * HEAD_DIM or not out.is_contiguous():
        raise ValueError(f"out must be contiguous {dtype} with N*256 elements")
    lse = torch.empty(N, dtype=torch.float32, device=o_parts.device) if return_lse else None
    fn = getattr(load(), "attn_lse_merge" + sfx)
    code = fn(_ptr(o_parts), _ptr(lse_parts), S, N, _ptr(g), _ptr(out), _ptr(lse), _stream())
    check(code, "attn_lse_merge" + sfx)
    return (out, lse) if return_lse else out


def last_device_status():
    """Synchronises the current stream; returns and clears the device status code."""
    return load().gqa_last_device_status(_stream())


def set_wait_timeout_ns(ns):
    load().gqa_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout():
    """Runs the kernels' bounded wait on a barrier nothing completes.  Returns
    (device status, nanoseconds the wait took); the status should be
    GQA_ERR_TIMEOUT (4) and the time about the configured bound."""
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    check(load().gqa_selftest_wait_timeout(_ptr(el), _stream()), "gqa_selftest_wait_timeout")
    st = last_device_status()
    return st, int(el.item())
