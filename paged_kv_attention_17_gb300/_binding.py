"""ctypes binding of ``libpkv.so`` (the C ABI declared in ``include/pkv.h``).

Argument marshalling only: each wrapper reads pointers, shapes and the current
CUDA stream from torch tensors and calls the C entry point of the same name;
every step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpkv.so")
_lib = None

PKV_OK = 0
PKV_F32, PKV_BF16 = 0, 1
PKV_DECODE_MAX_QLEN = 4
FLAG_BAD_BLOCK, FLAG_BAD_SLOT, FLAG_BAD_LENGTHS, FLAG_TIMEOUT = 1, 2, 4, 8

# Every symbol include/pkv.h declares.
EXPORTS = ("pkv_write", "pkv_write_e4m3", "pkv_stage_inputs", "pkv_num_splits", "pkv_workspace_bytes",
           "pkv_attention_varlen", "pkv_write_attention_varlen", "pkv_attention_varlen_window",
           "pkv_attention_varlen_e4m3", "pkv_write_attention_varlen_e4m3",
           "pkv_attention_varlen_e4m3_window", "pkv_cascade_attention_e4m3",
           "pkv_attention_varlen_noalloc", "pkv_cascade_splits", "pkv_cascade_workspace_bytes",
           "pkv_cascade_attention", "pkv_build_metadata", "pkv_status_string")


class PkvError(RuntimeError):
    def __init__(self, func, code):
        super().__init__(f"{func} returned {code} ({status_string(code)})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"CUDA library not built: {_LIB_PATH} is missing "
                              "(run paged_kv_attention_17_gb300.build.build())")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.pkv_write.argtypes = [vp, vp, vp, i64, vp, vp, i64, i32, i32, i32, i32, vp, vp]
        L.pkv_write.restype = i32
        f32 = ctypes.c_float
        L.pkv_write_e4m3.argtypes = [vp, vp, vp, i64, vp, vp, i64, i32, i32, i32, i32, f32, f32,
                                     vp, vp]
        L.pkv_write_e4m3.restype = i32
        L.pkv_stage_inputs.argtypes = [vp, vp, i64, vp]
        L.pkv_stage_inputs.restype = i32
        L.pkv_num_splits.argtypes = [i32] * 7
        L.pkv_num_splits.restype = i32
        L.pkv_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.pkv_workspace_bytes.restype = sz
        L.pkv_attention_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32, i32,
                                           i32, i32, i32, i32, ctypes.c_float, i32, i32, vp, sz,
                                           vp, i64, i32, vp]
        L.pkv_attention_varlen.restype = i32
        L.pkv_write_attention_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                 i32, i64, i32, i32, i32, i32, i32, i32, f32,
                                                 i32, i32, vp, sz, vp, i64, i32, vp]
        L.pkv_write_attention_varlen.restype = i32
        L.pkv_write_attention_varlen_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                      i32, i32, i64, i32, i32, i32, i32, i32,
                                                      i32, f32, f32, f32, i32, i32, vp, sz, vp,
                                                      i64, vp]
        L.pkv_write_attention_varlen_e4m3.restype = i32
        L.pkv_attention_varlen_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64,
                                                  i32, i32, i32, i32, i32, i32, f32, i32, i32,
                                                  i32, vp, sz, vp, i64, i32, vp]
        L.pkv_attention_varlen_window.restype = i32
        L.pkv_attention_varlen_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32,
                                                i32, i32, i32, i32, i32, f32, f32, f32, i32, i32,
                                                vp, sz, vp, i64, vp]
        L.pkv_attention_varlen_e4m3.restype = i32
        L.pkv_attention_varlen_e4m3_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                                       i64, i32, i32, i32, i32, i32, i32, f32, f32,
                                                       f32, i32, i32, i32, vp, sz, vp, i64, vp]
        L.pkv_attention_varlen_e4m3_window.restype = i32
        L.pkv_attention_varlen_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64,
                                                   i32, i32, i32, i32, i32, i32, ctypes.c_float,
                                                   i32, i32, vp, i64, i32, vp]
        L.pkv_attention_varlen_noalloc.restype = i32
        L.pkv_cascade_splits.argtypes = [i64, i32, i32, i32, i32, i32, i32]
        L.pkv_cascade_splits.restype = i32
        L.pkv_cascade_workspace_bytes.argtypes = [i64, i32, i32, i32]
        L.pkv_cascade_workspace_bytes.restype = sz
        L.pkv_cascade_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i64,
                                            i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp,
                                            i64, i32, vp]
        L.pkv_cascade_attention.restype = i32
        L.pkv_cascade_attention_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                 i64, i32, i32, i32, i32, i32, i32, f32, f32, f32,
                                                 i32, vp, sz, vp, i64, vp]
        L.pkv_cascade_attention_e4m3.restype = i32
        L.pkv_build_metadata.argtypes = [i32, vp, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp, vp,
                                         vp, vp]
        L.pkv_build_metadata.restype = i32
        L.pkv_status_string.argtypes = [i32]
        L.pkv_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().pkv_status_string(int(code)).decode()


pkv_status_string = status_string


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return PKV_F32
    if t == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(func, code):
    if code != PKV_OK:
        raise PkvError(func, code)


def pkv_write(k_new, v_new, slot_mapping, k_cache, v_cache, error_flag=None, stream=None):
    """Store k_new[t] / v_new[t] ([N, Hkv, D]) at cache slot slot_mapping[t] (int64)."""
    nb, bs, hkv, d = k_cache.shape
    code = lib().pkv_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), int(slot_mapping.numel()),
                           _ptr(k_cache), _ptr(v_cache), int(nb), int(bs), int(hkv), int(d),
                           _dtype_code(k_cache.dtype), _ptr(error_flag), _stream(stream))
    _check("pkv_write", code)


def pkv_write_e4m3(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                   error_flag=None, stream=None):
    """pkv_write into uint8 caches of E4M3 codes: slot slot_mapping[t] gets the
    codes of k_new[t] / k_scale and v_new[t] / v_scale (inputs fp32 or bf16)."""
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 caches are uint8 tensors of codes")
    nb, bs, hkv, d = k_cache.shape
    code = lib().pkv_write_e4m3(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                int(slot_mapping.numel()), _ptr(k_cache), _ptr(v_cache), int(nb),
                                int(bs), int(hkv), int(d), _dtype_code(k_new.dtype),
                                float(k_scale), float(v_scale), _ptr(error_flag), _stream(stream))
    _check("pkv_write_e4m3", code)


def pkv_stage_inputs(dst, src, stream=None):
    """Copy the bytes of src (pinned host memory the device can address, or
    device memory) into the device tensor dst with one library kernel that
    lets the next kernel on the stream start at once.  Both contiguous, same
    byte size (a multiple of 16), 16-byte aligned."""
    if not dst.is_cuda:
        raise ValueError("dst must be a device tensor")
    if not src.is_cuda and not src.is_pinned():
        raise ValueError("src must be pinned host memory or a device tensor")
    if not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("dst and src must be contiguous")
    n = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != n:
        raise ValueError("dst and src differ in size")
    _check("pkv_stage_inputs", lib().pkv_stage_inputs(_ptr(dst), _ptr(src), int(n),
                                                      _stream(stream)))


def pkv_num_splits(num_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                   device=None) -> int:
    dev = torch.cuda.current_device() if device is None else int(device)
    return int(lib().pkv_num_splits(int(num_seqs), int(max_query_len), int(max_seq_len),
                                    int(num_q_heads), int(num_kv_heads), int(head_dim), dev))


def pkv_workspace_bytes(num_seqs, num_q_heads, head_dim, num_splits) -> int:
    return int(lib().pkv_workspace_bytes(int(num_seqs), int(num_q_heads), int(head_dim),
                                         int(num_splits)))


def _splits_and_workspace(q, hkv, num_seqs, max_query_len, span, num_splits, workspace):
    """The split count (pkv_num_splits for a context of ``span`` keys when
    num_splits is 0) and a workspace for its partials: the caller's, or one
    allocated with torch here when none is given and one is needed."""
    _, hq, d = q.shape
    splits = int(num_splits)
    if splits == 0 and num_seqs > 0:
        splits = pkv_num_splits(num_seqs, max_query_len, span, hq, hkv, d, q.device.index)
    need = pkv_workspace_bytes(num_seqs, hq, d, splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return splits, workspace, ws_bytes


def split_span(max_seq_len, window=0) -> int:
    """The context length the automatic split count is sized for: a window
    bounds the keys a decode row reads to window + PKV_DECODE_MAX_QLEN."""
    if 0 < window < max_seq_len - PKV_DECODE_MAX_QLEN:
        return int(window) + PKV_DECODE_MAX_QLEN
    return int(max_seq_len)


def pkv_attention_varlen(q, k_cache, v_cache, out, query_start_loc, seq_lens, block_table,
                         max_query_len, max_seq_len, softmax_scale, causal=True, num_splits=0,
                         workspace=None, lse_out=None, error_flag=None, stream=None, window=0):
    """Attention of the flat batch q [N, Hq, D] over the paged cache into out.

    Metadata tensors are int32 on the device.  ``workspace`` is a uint8 device
    tensor of at least ``pkv_workspace_bytes(...)`` bytes; if None and one is
    needed it is allocated with torch here (allocate it yourself to capture the
    call in a CUDA graph).  ``window`` > 0 calls pkv_attention_varlen_window:
    the row at position p sees keys j > p - window only.
    """
    n_tok, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    num_seqs = int(seq_lens.numel())
    splits, workspace, ws_bytes = _splits_and_workspace(
        q, hkv, num_seqs, max_query_len, split_span(max_seq_len, window), num_splits, workspace)
    if window:
        code = lib().pkv_attention_varlen_window(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out),
            _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]),
            num_seqs, int(n_tok), int(max_query_len), int(max_seq_len), int(hq), int(hkv), int(d),
            int(bs), float(softmax_scale), 1 if causal else 0, int(window), splits,
            _ptr(workspace), int(ws_bytes), _ptr(error_flag), int(nb), _dtype_code(q.dtype),
            _stream(stream))
        _check("pkv_attention_varlen_window", code)
        return out
    code = lib().pkv_attention_varlen(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out), _ptr(query_start_loc),
        _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]), num_seqs, int(n_tok),
        int(max_query_len), int(max_seq_len), int(hq), int(hkv), int(d), int(bs),
        float(softmax_scale), 1 if causal else 0, splits, _ptr(workspace), int(ws_bytes),
        _ptr(error_flag), int(nb), _dtype_code(q.dtype), _stream(stream))
    _check("pkv_attention_varlen", code)
    return out


def pkv_write_attention_varlen(k_new, v_new, slot_mapping, q, k_cache, v_cache, out,
                               query_start_loc, seq_lens, block_table, max_query_len,
                               max_seq_len, softmax_scale, causal=True, num_splits=0,
                               workspace=None, lse_out=None, error_flag=None, stream=None):
    """pkv_write of k_new / v_new at slot_mapping, then pkv_attention_varlen -
    one launch fewer when every request is decode-class (the decode kernel
    stores the rows it reads).  Workspace handling as pkv_attention_varlen."""
    n_tok, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    num_seqs = int(seq_lens.numel())
    splits, workspace, ws_bytes = _splits_and_workspace(
        q, hkv, num_seqs, max_query_len, max_seq_len, num_splits, workspace)
    code = lib().pkv_write_attention_varlen(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(out), _ptr(lse_out), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table),
        int(block_table.shape[1]), num_seqs, int(n_tok), int(max_query_len), int(max_seq_len),
        int(hq), int(hkv), int(d), int(bs), float(softmax_scale), 1 if causal else 0, splits,
        _ptr(workspace), int(ws_bytes), _ptr(error_flag), int(nb), _dtype_code(q.dtype),
        _stream(stream))
    _check("pkv_write_attention_varlen", code)
    return out


def pkv_write_attention_varlen_e4m3(k_new, v_new, slot_mapping, q, k_cache, v_cache, out,
                                    query_start_loc, seq_lens, block_table, max_query_len,
                                    max_seq_len, softmax_scale, k_scale, v_scale, causal=True,
                                    num_splits=0, workspace=None, lse_out=None, error_flag=None,
                                    stream=None):
    """pkv_write_e4m3 then pkv_attention_varlen_e4m3 in one call (the write
    rides in the decode kernel for decode-class steps)."""
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 caches are uint8 tensors of codes")
    if q.dtype != torch.bfloat16 or k_new.dtype != torch.bfloat16:
        raise TypeError("q and the new K/V are bf16 for E4M3 caches")
    n_tok, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    num_seqs = int(seq_lens.numel())
    splits, workspace, ws_bytes = _splits_and_workspace(
        q, hkv, num_seqs, max_query_len, max_seq_len, num_splits, workspace)
    code = lib().pkv_write_attention_varlen_e4m3(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(out), _ptr(lse_out), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table),
        int(block_table.shape[1]), num_seqs, int(n_tok), int(max_query_len), int(max_seq_len),
        int(hq), int(hkv), int(d), int(bs), float(softmax_scale), float(k_scale), float(v_scale),
        1 if causal else 0, splits, _ptr(workspace), int(ws_bytes), _ptr(error_flag), int(nb),
        _stream(stream))
    _check("pkv_write_attention_varlen_e4m3", code)
    return out


def pkv_attention_varlen_e4m3(q, k_cache, v_cache, out, query_start_loc, seq_lens, block_table,
                              max_query_len, max_seq_len, softmax_scale, k_scale, v_scale,
                              causal=True, num_splits=0, workspace=None, lse_out=None,
                              error_flag=None, stream=None, window=0):
    """pkv_attention_varlen over uint8 caches of E4M3 codes (key code c stands
    for k_scale * value(c), value code c for v_scale * value(c)); q and out
    are bf16.  Workspace handling as pkv_attention_varlen; ``window`` > 0
    calls pkv_attention_varlen_e4m3_window."""
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 caches are uint8 tensors of codes")
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("q and out are bf16 for E4M3 caches")
    n_tok, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    num_seqs = int(seq_lens.numel())
    splits, workspace, ws_bytes = _splits_and_workspace(
        q, hkv, num_seqs, max_query_len, split_span(max_seq_len, window), num_splits, workspace)
    if window:
        code = lib().pkv_attention_varlen_e4m3_window(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out),
            _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]),
            num_seqs, int(n_tok), int(max_query_len), int(max_seq_len), int(hq), int(hkv),
            int(d), int(bs), float(softmax_scale), float(k_scale), float(v_scale),
            1 if causal else 0, int(window), splits, _ptr(workspace), int(ws_bytes),
            _ptr(error_flag), int(nb), _stream(stream))
        _check("pkv_attention_varlen_e4m3_window", code)
        return out
    code = lib().pkv_attention_varlen_e4m3(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out), _ptr(query_start_loc),
        _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]), num_seqs, int(n_tok),
        int(max_query_len), int(max_seq_len), int(hq), int(hkv), int(d), int(bs),
        float(softmax_scale), float(k_scale), float(v_scale), 1 if causal else 0, splits,
        _ptr(workspace), int(ws_bytes), _ptr(error_flag), int(nb), _stream(stream))
    _check("pkv_attention_varlen_e4m3", code)
    return out


def pkv_attention_varlen_noalloc(q, k_cache, v_cache, out, query_start_loc, seq_lens, block_table,
                                 max_query_len, max_seq_len, softmax_scale, causal=True,
                                 num_splits=0, lse_out=None, error_flag=None, stream=None):
    """pkv_attention_varlen for callers that cannot allocate: the split-KV
    partials use the library's fixed 8 MiB device array instead of a
    workspace (automatic split counts are lowered to fit it; an explicit one
    that does not fit raises PkvError with PKV_ERR_WORKSPACE).  Calls whose
    kernels overlap on the GPU share that array and race; the first call on a
    device should come before any stream capture."""
    n_tok, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    code = lib().pkv_attention_varlen_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out), _ptr(query_start_loc),
        _ptr(seq_lens), _ptr(block_table), int(block_table.shape[1]), int(seq_lens.numel()),
        int(n_tok), int(max_query_len), int(max_seq_len), int(hq), int(hkv), int(d), int(bs),
        float(softmax_scale), 1 if causal else 0, int(num_splits), _ptr(error_flag), int(nb),
        _dtype_code(q.dtype), _stream(stream))
    _check("pkv_attention_varlen_noalloc", code)
    return out


def pkv_cascade_splits(num_tokens, shared_blocks, num_q_heads, num_kv_heads, head_dim,
                       dtype=torch.bfloat16, device=None) -> int:
    dev = torch.cuda.current_device() if device is None else int(device)
    return int(lib().pkv_cascade_splits(int(num_tokens), int(shared_blocks), int(num_q_heads),
                                        int(num_kv_heads), int(head_dim), _dtype_code(dtype),
                                        dev))


def pkv_cascade_workspace_bytes(num_tokens, num_q_heads, head_dim, prefix_splits) -> int:
    return int(lib().pkv_cascade_workspace_bytes(int(num_tokens), int(num_q_heads),
                                                 int(head_dim), int(prefix_splits)))


def pkv_cascade_attention(q, k_cache, v_cache, out, query_start_loc, suffix_lens,
                          suffix_block_table, shared_block_table, max_query_len, max_suffix_len,
                          softmax_scale, prefix_splits=0, workspace=None, lse_out=None,
                          error_flag=None, stream=None, kv_scales=None):
    """Attention of a batch whose requests share the blocks of
    ``shared_block_table`` (int32 [shared_blocks]) as a prefix, each followed
    by its own ``suffix_lens[r]`` keys in ``suffix_block_table`` row r.
    ``workspace`` (uint8, >= pkv_cascade_workspace_bytes) is allocated here
    if None.  uint8 caches of E4M3 codes take ``kv_scales`` = (k_scale,
    v_scale) and bf16 q / out (pkv_cascade_attention_e4m3)."""
    e4m3 = k_cache.dtype == torch.uint8
    if e4m3 and kv_scales is None:
        raise ValueError("an E4M3 (uint8) cache needs kv_scales=(k_scale, v_scale)")
    n_tok, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    num_seqs = int(suffix_lens.numel())
    shared = int(shared_block_table.numel()) if shared_block_table is not None else 0
    splits = int(prefix_splits)
    if shared == 0:
        splits = 0
    elif splits == 0 and n_tok > 0:
        # (an E4M3 prefix pass takes the tensor-core tiles where bf16 at
        # head_dim 128 would, else the CUDA-core tiles: the fp32 rule)
        rule = (torch.bfloat16 if d == 128 else torch.float32) if e4m3 else q.dtype
        splits = pkv_cascade_splits(n_tok, shared, hq, hkv, d, rule, q.device.index)
    need = pkv_cascade_workspace_bytes(n_tok, hq, d, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if e4m3:
        code = lib().pkv_cascade_attention_e4m3(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out),
            _ptr(query_start_loc), _ptr(suffix_lens), _ptr(suffix_block_table),
            int(suffix_block_table.shape[1]), _ptr(shared_block_table) if shared else None,
            shared, num_seqs, int(n_tok), int(max_query_len), int(max_suffix_len), int(hq),
            int(hkv), int(d), int(bs), float(softmax_scale), float(kv_scales[0]),
            float(kv_scales[1]), splits, _ptr(workspace), int(ws_bytes), _ptr(error_flag),
            int(nb), _stream(stream))
        _check("pkv_cascade_attention_e4m3", code)
        return out
    code = lib().pkv_cascade_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse_out), _ptr(query_start_loc),
        _ptr(suffix_lens), _ptr(suffix_block_table), int(suffix_block_table.shape[1]),
        _ptr(shared_block_table) if shared else None, shared, num_seqs, int(n_tok),
        int(max_query_len), int(max_suffix_len), int(hq), int(hkv), int(d), int(bs),
        float(softmax_scale), splits, _ptr(workspace), int(ws_bytes), _ptr(error_flag), int(nb),
        _dtype_code(q.dtype), _stream(stream))
    _check("pkv_cascade_attention", code)
    return out


def pkv_build_metadata(computed, scheduled, block_ids_per_request, block_size=16,
                       max_blocks_per_seq=None):
    """The step's flat-batch metadata from the library's host builder:
    ``computed`` / ``scheduled`` per request and each request's block ids.
    Returns numpy arrays query_start_loc, seq_lens, block_table (int32),
    slot_mapping, positions (int64) and the host scalars num_tokens,
    max_query_len, max_seq_len."""
    import numpy as np
    n = len(computed)
    c = np.ascontiguousarray(computed, dtype=np.int32)
    s = np.ascontiguousarray(scheduled, dtype=np.int32)
    counts = [len(b) for b in block_ids_per_request]
    offsets = np.zeros(n + 1, dtype=np.int32)
    np.cumsum(counts, out=offsets[1:])
    ids = np.ascontiguousarray(np.concatenate([np.asarray(b, dtype=np.int32)
                                               for b in block_ids_per_request])
                               if n and offsets[-1] else np.zeros(1, dtype=np.int32))
    width = int(max_blocks_per_seq or max(counts + [1]))
    num_tokens = int(s.sum()) if n else 0
    qsl = np.zeros(n + 1, dtype=np.int32)
    seq_lens = np.zeros(max(n, 1), dtype=np.int32)
    table = np.zeros((max(n, 1), width), dtype=np.int32)
    slots = np.zeros(max(num_tokens, 1), dtype=np.int64)
    pos = np.zeros(max(num_tokens, 1), dtype=np.int64)
    mq, ms = ctypes.c_int32(0), ctypes.c_int32(0)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)  # noqa: E731
    code = lib().pkv_build_metadata(n, p(c) if n else None, p(s) if n else None, p(offsets),
                                    p(ids), int(block_size), width, num_tokens, p(qsl),
                                    p(seq_lens), p(table), p(slots), p(pos),
                                    ctypes.byref(mq), ctypes.byref(ms))
    _check("pkv_build_metadata", code)
    return {"query_start_loc": qsl, "seq_lens": seq_lens[:n], "block_table": table[:n],
            "slot_mapping": slots[:num_tokens], "positions": pos[:num_tokens],
            "num_tokens": num_tokens, "max_query_len": int(mq.value),
            "max_seq_len": int(ms.value)}

