"""Python entry points with the C ABI's names (include/pagedattn.h).

Each function checks that tensors are on the GPU, contiguous and of the right
integer type, then calls the library on torch's current stream. Shapes and
sizes are validated by the library itself.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from ._lib import DTYPE_CODE, check, lib, ptr, stream_handle


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def pa_compute_slot_mapping(query_start_loc: torch.Tensor, positions: torch.Tensor,
                            block_table: torch.Tensor, block_size: int,
                            slot_mapping: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """slot[t] = block_table[r, pos // B] * B + pos % B for the tokens of each
    request r; -1 for tokens of no request. Returns int64 [num_tokens]."""
    _dev(query_start_loc, "query_start_loc", torch.int32)
    _dev(positions, "positions", torch.int64)
    _dev(block_table, "block_table", torch.int32)
    T = positions.numel()
    if slot_mapping is None:
        slot_mapping = torch.empty(T, dtype=torch.int64, device=positions.device)
    _dev(slot_mapping, "slot_mapping", torch.int64)
    stride = block_table.shape[1] if block_table.dim() == 2 else 0
    check("pa_compute_slot_mapping", lib().pa_compute_slot_mapping(
        ptr(query_start_loc), query_start_loc.numel() - 1, ptr(positions), T,
        ptr(block_table), stride, block_size, ptr(slot_mapping), stream_handle(stream)))
    return slot_mapping


def pa_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                         key_cache: torch.Tensor, value_cache: torch.Tensor,
                         stream=None) -> None:
    """Write k[t], v[t] ([T, Hkv, D]) into pool slot slot_mapping[t]; pools are
    [num_blocks, Hkv, B, D]."""
    for n, t in (("k", k), ("v", v), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(slot_mapping, "slot_mapping", torch.int64)
    NB, Hkv, B, D = key_cache.shape
    if value_cache.shape != key_cache.shape or k.shape != v.shape:
        raise ValueError("shape mismatch")
    if k.shape[1:] != (Hkv, D) or k.dtype != key_cache.dtype:
        raise ValueError("k/v must be [T, Hkv, D] in the cache dtype")
    check("pa_reshape_and_cache", lib().pa_reshape_and_cache(
        ptr(k), ptr(v), k.shape[0], Hkv, D, DTYPE_CODE[k.dtype], ptr(slot_mapping),
        ptr(key_cache), ptr(value_cache), NB, B, stream_handle(stream)))


def pa_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                              head_size: int, block_size: int, max_seq_len: int,
                              partition_size: int = 0) -> int:
    n = lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size,
                                        block_size, max_seq_len, partition_size)
    if n < 0:
        check("pa_decode_workspace_bytes", int(n))
    return int(n)


def pa_decode_partitioning(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                           block_size: int, max_seq_len: int, partition_size: int = 0):
    """(num_splits, partition_tokens) the attention call will use."""
    s, p = ctypes.c_int(0), ctypes.c_int(0)
    check("pa_decode_partitioning", lib().pa_decode_partitioning(
        num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, partition_size,
        ctypes.byref(s), ctypes.byref(p)))
    return s.value, p.value


def pa_decode_window_partitioning(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                  block_size: int, max_seq_len: int, window: int,
                                  partition_size: int = 0):
    """(num_splits, partition_tokens) the windowed attention calls will use."""
    s, p = ctypes.c_int(0), ctypes.c_int(0)
    check("pa_decode_window_partitioning", lib().pa_decode_window_partitioning(
        num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, window, partition_size,
        ctypes.byref(s), ctypes.byref(p)))
    return s.value, p.value


def pa_decode_fp8_partitioning(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                               head_size: int, block_size: int, dtype: torch.dtype,
                               max_seq_len: int, window: int = 0, partition_size: int = 0):
    """(num_splits, partition_tokens) the fp8-pool attention calls will use;
    dtype is the query type."""
    s, p = ctypes.c_int(0), ctypes.c_int(0)
    check("pa_decode_fp8_partitioning", lib().pa_decode_fp8_partitioning(
        num_seqs, num_q_heads, num_kv_heads, head_size, block_size, DTYPE_CODE[dtype],
        max_seq_len, window, partition_size, ctypes.byref(s), ctypes.byref(p)))
    return s.value, p.value


KV_FORMAT = {"16bit": 0, "fp8": 1, "fp8_block_scales": 2}


def pa_decode_even_ctas(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_size: int,
                        block_size: int, dtype: torch.dtype, kv_format: str, max_seq_len: int,
                        window: int = 0, partition_size: int = 0) -> int:
    """CTAs of the even schedule a decode call with these sizes runs (0: it
    uses fixed partitions); kv_format is "16bit", "fp8" or
    "fp8_block_scales", dtype the query type."""
    n = lib().pa_decode_even_ctas(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                  DTYPE_CODE[dtype], KV_FORMAT[kv_format], max_seq_len, window,
                                  partition_size)
    if n < 0:
        check("pa_decode_even_ctas", int(n))
    return int(n)


def pa_decode_fp8_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                  head_size: int, block_size: int, dtype: torch.dtype,
                                  max_seq_len: int, window: int = 0,
                                  partition_size: int = 0) -> int:
    """Scratch bytes of the fp8-pool decode calls; dtype is the query type."""
    n = lib().pa_decode_fp8_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size,
                                            block_size, DTYPE_CODE[dtype], max_seq_len, window,
                                            partition_size)
    if n < 0:
        check("pa_decode_fp8_workspace_bytes", int(n))
    return int(n)


def pa_decode_attention(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                        num_kv_heads: int, out: Optional[torch.Tensor] = None, *,
                        max_seq_len: int, partition_size: int = 0,
                        workspace: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Paged decode attention. q/out [S, Hq, D]; pools [NB, Hkv, B, D];
    block_tables int32 [S, max_blocks]; seq_lens int32 [S]; max_seq_len is a
    host upper bound of seq_lens."""
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = key_cache.shape
    if Hkv != num_kv_heads or Dk != D or value_cache.shape != key_cache.shape:
        raise ValueError("pool shape does not match q / num_kv_heads")
    if key_cache.dtype != q.dtype or value_cache.dtype != q.dtype:
        raise ValueError("q and pools must share a dtype")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out")
    need = pa_decode_workspace_bytes(S, Hq, Hkv, D, B, max_seq_len, partition_size)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention", lib().pa_decode_attention(
        ptr(q), ptr(key_cache), ptr(value_cache), ptr(block_tables), block_tables.shape[1],
        ptr(seq_lens), S, Hq, Hkv, D, B, NB, DTYPE_CODE[q.dtype], float(scale),
        int(max_seq_len), int(partition_size), ptr(out), ptr(workspace), ws_bytes,
        stream_handle(stream)))
    return out


def pa_copy_blocks(key_caches: Sequence[torch.Tensor], value_caches: Sequence[torch.Tensor],
                   src_dst_pairs: torch.Tensor,
                   src_dst_pairs_host: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy whole blocks src -> dst in every layer's K and V pool.
    src_dst_pairs: int64 [P, 2] on the GPU; src_dst_pairs_host: optional CPU
    copy, which enables the aliasing check before launch."""
    if len(key_caches) != len(value_caches) or not key_caches:
        raise ValueError("need one K and one V pool per layer")
    _dev(src_dst_pairs, "src_dst_pairs", torch.int64)
    kc0 = key_caches[0]
    for t in list(key_caches) + list(value_caches):
        _dev(t, "cache")
        if t.shape != kc0.shape or t.dtype != kc0.dtype:
            raise ValueError("all pools must share shape and dtype")
    nl = len(key_caches)
    kp = (ctypes.c_void_p * nl)(*[t.data_ptr() for t in key_caches])
    vp = (ctypes.c_void_p * nl)(*[t.data_ptr() for t in value_caches])
    host = None
    if src_dst_pairs_host is not None:
        host = src_dst_pairs_host.to(torch.int64).contiguous()
        if host.is_cuda or host.numel() != src_dst_pairs.numel():
            raise ValueError("src_dst_pairs_host must be a CPU copy of the pairs")
    NB = kc0.shape[0]
    block_bytes = kc0[0].numel() * kc0.element_size()
    check("pa_copy_blocks", lib().pa_copy_blocks(
        kp, vp, nl, ptr(src_dst_pairs), None if host is None else host.data_ptr(),
        src_dst_pairs.numel() // 2, NB, block_bytes, stream_handle(stream)))


def pa_get_device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the latched device error
    (0 = none)."""
    code = ctypes.c_int(0)
    check("pa_get_device_error", lib().pa_get_device_error(ctypes.byref(code),
                                                           stream_handle(stream)))
    return code.value


def pa_map_to_kernel_blocks(manager_table: torch.Tensor, blocks_per_kv_block: int,
                            kernel_table: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Expand an int32 [rows, cols] table of allocator block ids (each owning
    r = blocks_per_kv_block kernel blocks) into an int32 [rows, cols * r]
    table of kernel block ids."""
    _dev(manager_table, "manager_table", torch.int32)
    rows, cols = manager_table.shape
    r = int(blocks_per_kv_block)
    if kernel_table is None:
        kernel_table = torch.empty((rows, cols * r), dtype=torch.int32,
                                   device=manager_table.device)
    _dev(kernel_table, "kernel_table", torch.int32)
    check("pa_map_to_kernel_blocks", lib().pa_map_to_kernel_blocks(
        ptr(manager_table), rows, cols, cols, r, ptr(kernel_table), kernel_table.shape[1],
        stream_handle(stream)))
    return kernel_table


def pa_multi_query_workspace_bytes(num_tokens: int, num_seqs: int, num_q_heads: int,
                                   num_kv_heads: int, head_size: int, block_size: int,
                                   max_query_len: int, max_seq_len: int,
                                   partition_size: int = 0) -> int:
    n = lib().pa_multi_query_workspace_bytes(num_tokens, num_seqs, num_q_heads, num_kv_heads,
                                             head_size, block_size, max_query_len,
                                             max_seq_len, partition_size)
    if n < 0:
        check("pa_multi_query_workspace_bytes", int(n))
    return int(n)


def pa_multi_query_attention(q: torch.Tensor, query_start_loc: torch.Tensor,
                             key_cache: torch.Tensor, value_cache: torch.Tensor,
                             block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             num_kv_heads: int, out: Optional[torch.Tensor] = None, *,
                             max_query_len: int, max_seq_len: int, partition_size: int = 0,
                             workspace: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """Causal paged attention of several new tokens per sequence.
    q/out [T, Hq, D] with T = query_start_loc[-1]; pools [NB, Hkv, B, D]."""
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(query_start_loc, "query_start_loc", torch.int32)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    T, Hq, D = q.shape
    NB, Hkv, B, Dk = key_cache.shape
    if Hkv != num_kv_heads or Dk != D or value_cache.shape != key_cache.shape:
        raise ValueError("pool shape does not match q / num_kv_heads")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out")
    S = query_start_loc.numel() - 1
    need = pa_multi_query_workspace_bytes(T, S, Hq, Hkv, D, B, max_query_len, max_seq_len,
                                          partition_size)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_multi_query_attention", lib().pa_multi_query_attention(
        ptr(q), ptr(query_start_loc), S, T, ptr(key_cache), ptr(value_cache), ptr(block_tables),
        block_tables.shape[1], ptr(seq_lens), Hq, Hkv, D, B, NB, DTYPE_CODE[q.dtype],
        float(scale), int(max_query_len), int(max_seq_len), int(partition_size), ptr(out),
        ptr(workspace), ws_bytes, stream_handle(stream)))
    return out


def pa_reshape_and_cache_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                             key_cache: torch.Tensor, value_cache: torch.Tensor,
                             k_scale: float, v_scale: float, stream=None) -> None:
    """KV write into E4M3 pools (uint8 [NB, Hkv, B, D]): code = e4m3(x / scale)."""
    for n, t in (("k", k), ("v", v), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(slot_mapping, "slot_mapping", torch.int64)
    if key_cache.dtype != torch.uint8 or value_cache.dtype != torch.uint8:
        raise ValueError("fp8 pools are uint8 tensors of E4M3 codes")
    NB, Hkv, B, D = key_cache.shape
    check("pa_reshape_and_cache_fp8", lib().pa_reshape_and_cache_fp8(
        ptr(k), ptr(v), k.shape[0], Hkv, D, DTYPE_CODE[k.dtype], ptr(slot_mapping),
        ptr(key_cache), ptr(value_cache), NB, B, float(k_scale), float(v_scale),
        stream_handle(stream)))


def pa_decode_attention_fp8(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                            num_kv_heads: int, k_scale: float, v_scale: float,
                            out: Optional[torch.Tensor] = None, *, max_seq_len: int,
                            partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Decode attention over E4M3 pools; q/out in fp32/fp16/bf16."""
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = key_cache.shape
    if Hkv != num_kv_heads or Dk != D or key_cache.dtype != torch.uint8:
        raise ValueError("pools must be uint8 [NB, Hkv, B, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out")
    need = pa_decode_fp8_workspace_bytes(S, Hq, Hkv, D, B, q.dtype, max_seq_len, 0,
                                         partition_size)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention_fp8", lib().pa_decode_attention_fp8(
        ptr(q), ptr(key_cache), ptr(value_cache), ptr(block_tables), block_tables.shape[1],
        ptr(seq_lens), S, Hq, Hkv, D, B, NB, DTYPE_CODE[q.dtype], float(scale), float(k_scale),
        float(v_scale), int(max_seq_len), int(partition_size), ptr(out), ptr(workspace),
        ws_bytes, stream_handle(stream)))
    return out


def pa_reshape_and_cache_fp8_scaled(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                                    key_cache: torch.Tensor, value_cache: torch.Tensor,
                                    k_scales: torch.Tensor, v_scales: torch.Tensor,
                                    stream=None) -> None:
    """KV write into E4M3 pools whose blocks carry their own scales
    (k_scales / v_scales: float32 [NB, Hkv], updated where this write stores
    a block's first row)."""
    for n, t in (("k", k), ("v", v), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(slot_mapping, "slot_mapping", torch.int64)
    _dev(k_scales, "k_scales", torch.float32)
    _dev(v_scales, "v_scales", torch.float32)
    if key_cache.dtype != torch.uint8 or value_cache.dtype != torch.uint8:
        raise ValueError("fp8 pools are uint8 tensors of E4M3 codes")
    NB, Hkv, B, D = key_cache.shape
    if tuple(k_scales.shape) != (NB, Hkv) or tuple(v_scales.shape) != (NB, Hkv):
        raise ValueError("scales must be float32 [num_blocks, num_kv_heads]")
    check("pa_reshape_and_cache_fp8_scaled", lib().pa_reshape_and_cache_fp8_scaled(
        ptr(k), ptr(v), k.shape[0], Hkv, D, DTYPE_CODE[k.dtype], ptr(slot_mapping),
        ptr(key_cache), ptr(value_cache), ptr(k_scales), ptr(v_scales), NB, B,
        stream_handle(stream)))


def pa_decode_attention_fp8_scaled(q: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, k_scales: torch.Tensor,
                                   v_scales: torch.Tensor, block_tables: torch.Tensor,
                                   seq_lens: torch.Tensor, scale: float, num_kv_heads: int,
                                   out: Optional[torch.Tensor] = None, *, max_seq_len: int,
                                   window: int = 0, partition_size: int = 0,
                                   workspace: Optional[torch.Tensor] = None,
                                   stream=None) -> torch.Tensor:
    """Decode attention over E4M3 pools with per-(block, KV head) scales;
    window 0 attends the whole sequence."""
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(k_scales, "k_scales", torch.float32)
    _dev(v_scales, "v_scales", torch.float32)
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = key_cache.shape
    if Hkv != num_kv_heads or Dk != D or key_cache.dtype != torch.uint8:
        raise ValueError("pools must be uint8 [NB, Hkv, B, D] matching q")
    if tuple(k_scales.shape) != (NB, Hkv) or tuple(v_scales.shape) != (NB, Hkv):
        raise ValueError("scales must be float32 [num_blocks, num_kv_heads]")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out")
    need = pa_decode_fp8_workspace_bytes(S, Hq, Hkv, D, B, q.dtype, max_seq_len, window,
                                         partition_size)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention_fp8_scaled", lib().pa_decode_attention_fp8_scaled(
        ptr(q), ptr(key_cache), ptr(value_cache), ptr(k_scales), ptr(v_scales),
        ptr(block_tables), block_tables.shape[1], ptr(seq_lens), S, Hq, Hkv, D, B, NB,
        DTYPE_CODE[q.dtype], float(scale), int(window), int(max_seq_len), int(partition_size),
        ptr(out), ptr(workspace), ws_bytes, stream_handle(stream)))
    return out


def pa_decode_window_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                     head_size: int, block_size: int, max_seq_len: int,
                                     window: int, partition_size: int = 0) -> int:
    n = lib().pa_decode_window_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size,
                                               block_size, max_seq_len, window, partition_size)
    if n < 0:
        check("pa_decode_window_workspace_bytes", int(n))
    return int(n)


def _window_call(name, q, key_cache, value_cache, block_tables, seq_lens, scale, num_kv_heads,
                 scales, window, out, max_seq_len, partition_size, workspace, stream):
    for n, t in (("q", q), ("key_cache", key_cache), ("value_cache", value_cache)):
        _dev(t, n)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = key_cache.shape
    pool_dtype = torch.uint8 if scales else q.dtype
    if Hkv != num_kv_heads or Dk != D or value_cache.shape != key_cache.shape:
        raise ValueError("pool shape does not match q / num_kv_heads")
    if key_cache.dtype != pool_dtype or value_cache.dtype != pool_dtype:
        raise ValueError(f"pools must be {pool_dtype}")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out")
    if scales:       # fp8 pools: their own partitioning and scratch
        need = pa_decode_fp8_workspace_bytes(S, Hq, Hkv, D, B, q.dtype, max_seq_len, window,
                                             partition_size)
    else:
        need = pa_decode_window_workspace_bytes(S, Hq, Hkv, D, B, max_seq_len, window,
                                                partition_size)
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(name, getattr(lib(), name)(
        ptr(q), ptr(key_cache), ptr(value_cache), ptr(block_tables), block_tables.shape[1],
        ptr(seq_lens), S, Hq, Hkv, D, B, NB, DTYPE_CODE[q.dtype], float(scale),
        *[float(x) for x in scales], int(window), int(max_seq_len), int(partition_size),
        ptr(out), ptr(workspace), ws_bytes, stream_handle(stream)))
    return out


def pa_decode_attention_window(q: torch.Tensor, key_cache: torch.Tensor,
                               value_cache: torch.Tensor, block_tables: torch.Tensor,
                               seq_lens: torch.Tensor, scale: float, num_kv_heads: int,
                               window: int, out: Optional[torch.Tensor] = None, *,
                               max_seq_len: int, partition_size: int = 0,
                               workspace: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """Sliding-window decode: each query attends its sequence's last
    `window` tokens (0 = all); table entries of blocks wholly before the
    window are never read."""
    return _window_call("pa_decode_attention_window", q, key_cache, value_cache, block_tables,
                        seq_lens, scale, num_kv_heads, (), window, out, max_seq_len,
                        partition_size, workspace, stream)


def pa_decode_attention_fp8_window(q: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, block_tables: torch.Tensor,
                                   seq_lens: torch.Tensor, scale: float, num_kv_heads: int,
                                   k_scale: float, v_scale: float, window: int,
                                   out: Optional[torch.Tensor] = None, *, max_seq_len: int,
                                   partition_size: int = 0,
                                   workspace: Optional[torch.Tensor] = None,
                                   stream=None) -> torch.Tensor:
    """pa_decode_attention_window over E4M3 pools."""
    return _window_call("pa_decode_attention_fp8_window", q, key_cache, value_cache,
                        block_tables, seq_lens, scale, num_kv_heads, (k_scale, v_scale),
                        window, out, max_seq_len, partition_size, workspace, stream)


def pa_selftest_bounded_wait(timeout_cycles: int = 2_000_000, stream=None) -> list:
    """Run the bounded-wait self-test; returns [status of warp 0, status of
    warp 1, abort flag] (expected: [PA_ERR_TIMEOUT, PA_ERR_TIMEOUT, 1])."""
    status = torch.full((3,), 12345, dtype=torch.int32, device="cuda")
    check("pa_selftest_bounded_wait", lib().pa_selftest_bounded_wait(
        ptr(status), int(timeout_cycles), stream_handle(stream)))
    torch.cuda.synchronize()
    return status.cpu().tolist()
