"""fp64 / exact-integer oracle for slot mapping, the KV write, block copy and
paged decode attention.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Arrays are numpy. Stored KV
values keep their storage type: numpy float32, float16, or uint16 bit patterns
for bfloat16 (numpy has no bfloat16); `upcast` turns any of them into float64
exactly.

Pool layout (a reading; the pages only say a block holds the K/V vectors of B
tokens): key_cache and value_cache are [num_blocks, num_kv_heads, block_size,
head_size]. A slot id s names block s // B, row s % B of that block.
"""
from __future__ import annotations

import math

import numpy as np

PAD_SLOT = -1


# --------------------------------------------------------------------------
# dtype handling
# --------------------------------------------------------------------------
def upcast(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64.

    bf16 is the upper half of an IEEE fp32 word, so its value is the fp32
    whose high 16 bits are the stored pattern and low 16 bits are zero."""
    if dtype == "f32":
        assert a.dtype == np.float32
        return a.astype(np.float64)
    if dtype == "f16":
        assert a.dtype == np.float16
        return a.astype(np.float64)
    if dtype == "bf16":
        assert a.dtype in (np.uint16, np.int16)
        bits = a.view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# block arithmetic ([P4] "按 Block 分配"; [P2] block-size trade-off section)
# --------------------------------------------------------------------------
def blocks_needed(num_tokens: int, block_size: int) -> int:
    """A sequence of T tokens without sharing holds ceil(T / B) blocks
    ([P4] "按 Block 分配": 9 tokens, B=4 -> 3 blocks)."""
    assert num_tokens >= 0 and block_size >= 1
    return -(-num_tokens // block_size)


def slots_allocated(num_tokens: int, block_size: int) -> int:
    """B * ceil(T / B) token slots ([P4] "按 Block 分配": 12 slots)."""
    return block_size * blocks_needed(num_tokens, block_size)


def fragmentation(lengths, block_size: int):
    """Tail waste of a batch, as the block-size section of [P2] defines it:
    blocks = sum ceil(L/B), slots = blocks * B, empty = slots - sum L,
    rate = empty / slots. Returns (blocks, slots, empty, rate)."""
    blocks = sum(blocks_needed(L, block_size) for L in lengths)
    slots = blocks * block_size
    empty = slots - sum(lengths)
    return blocks, slots, empty, (empty / slots if slots else 0.0)


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_size: int,
                       dtype_bytes: int) -> int:
    """Per-token KV footprint: 2 (K and V) x layers x KV heads x head size x
    bytes per element ([P3] §2.1; [P1] §1.1 memory formula; [P2] OPT-13B
    example)."""
    return 2 * num_layers * num_kv_heads * head_size * dtype_bytes


def sharing_saving(tables) -> float:
    """Block saving of a set of block tables as [P2]'s Figure-8 simulator
    defines it: (logical mappings - distinct physical blocks) / logical
    mappings."""
    logical = sum(len(t) for t in tables)
    unique = len({b for t in tables for b in t})
    return (logical - unique) / logical if logical else 0.0


# --------------------------------------------------------------------------
# slot mapping ([P1] §2.3 BlockTable / slot-mapping kernel, single rank)
# --------------------------------------------------------------------------
def slot_mapping(query_start_loc, positions, block_table, block_size: int,
                 num_tokens: int | None = None) -> np.ndarray:
    """slot[t] for every token t of request r (query_start_loc[r] <= t <
    query_start_loc[r+1]):

        logical block  lb  = pos // B
        physical block pb  = block_table[r, lb]
        slot               = pb * B + (pos - lb * B)

    This is the context-parallel-free case of [P1] §2.3 (world size 1, so
    every token is local and no PAD is produced by the formula). Tokens that
    belong to no request keep PAD_SLOT (-1).

    Invalid input (negative position, logical block beyond the table row, or
    an unassigned (negative) table entry) raises ValueError."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    tab = np.asarray(block_table, dtype=np.int64)
    T = len(pos) if num_tokens is None else num_tokens
    out = np.full(T, PAD_SLOT, dtype=np.int64)
    B = int(block_size)
    for r in range(len(qsl) - 1):
        for t in range(int(qsl[r]), int(qsl[r + 1])):
            if t < 0 or t >= T:
                continue
            p = int(pos[t])
            if p < 0:
                raise ValueError(f"negative position at token {t}")
            lb = p // B
            if lb >= tab.shape[1]:
                raise ValueError(f"token {t}: logical block {lb} past the table")
            pb = int(tab[r, lb])
            if pb < 0:
                raise ValueError(f"token {t}: table entry {lb} unassigned")
            out[t] = pb * B + (p - lb * B)
    return out


# --------------------------------------------------------------------------
# KV write and block copy (byte copies)
# --------------------------------------------------------------------------
def reshape_and_cache(k, v, slots, key_cache, value_cache, block_size: int):
    """Write token t's K/V rows (every KV head) into the pool slot slots[t],
    in place. A negative slot (PAD) is skipped. The slot names block
    slot // B, row slot % B ([P1] §2.3: the slot mapping lets the attention
    kernel address the pool directly)."""
    B = int(block_size)
    nb = key_cache.shape[0]
    for t, s in enumerate(np.asarray(slots, dtype=np.int64)):
        s = int(s)
        if s < 0:
            continue
        blk, row = s // B, s % B
        if blk >= nb:
            raise ValueError(f"slot {s} outside the pool")
        key_cache[blk, :, row, :] = k[t]
        value_cache[blk, :, row, :] = v[t]


def copy_blocks(key_caches, value_caches, src_dst_pairs):
    """Block-level copy-on-write data movement: for each (src, dst) pair,
    every layer's K and V block src is copied whole into block dst ([P2]
    Figure 8: block 1's content is copied into block 3; [P4] COW figure:
    P0 copied into P4). Destinations must be distinct and no destination may
    also be a source."""
    pairs = [(int(a), int(b)) for a, b in np.asarray(src_dst_pairs).reshape(-1, 2)]
    dsts = [d for _, d in pairs]
    srcs = {s for s, _ in pairs}
    if len(set(dsts)) != len(dsts) or any(d in srcs for d in dsts):
        raise ValueError("aliasing copy pairs")
    for kc, vc in zip(key_caches, value_caches):
        for s, d in pairs:
            kc[d] = kc[s]
            vc[d] = vc[s]


# --------------------------------------------------------------------------
# paged decode attention
# --------------------------------------------------------------------------
def window_start(seq_len: int, window: int) -> int:
    """First token a decode query attends under a sliding window of `window`
    tokens (0 = no window). A reading: the window is the last `window`
    tokens of the sequence, the new token included, so token j is attended
    iff seq_len - window <= j < seq_len. The pages name the sliding window
    only through the blocks it lets the allocator release ([P1] §3.2
    allocate_slots, phase 1: blocks that fall wholly before the window are
    freed)."""
    if window <= 0 or seq_len <= window:
        return 0
    return seq_len - window


def skipped_blocks(seq_len: int, window: int, block_size: int) -> int:
    """Leading logical blocks that hold no attended token: the skipped
    tokens // B ([P1] §3.3.1 get_num_blocks_to_allocate: skipped blocks are
    the skipped tokens floor-divided by the block size). Their table entries
    are never read, so the allocator may free them."""
    return window_start(seq_len, window) // block_size


def gather_kv(cache, table_row, seq_len: int, kv_head: int, block_size: int,
              dtype: str, start: int = 0) -> np.ndarray:
    """Contiguous fp64 copy of one sequence's K (or V) rows start..seq_len-1
    for one KV head, token j read from physical block table_row[j // B], row
    j % B ([P4] "按 Block 分配": token 8 -> logical block 2 -> P4, row 0).
    Table entries of blocks before start // B are not read."""
    j = np.arange(start, seq_len, dtype=np.int64)
    blk = np.asarray(table_row, dtype=np.int64)[j // block_size]
    if len(j) and (blk.min() < 0 or blk.max() >= cache.shape[0]):
        raise ValueError("block id outside the pool")
    rows = cache[blk, kv_head, j % block_size, :]
    return upcast(np.ascontiguousarray(rows), dtype)


def decode_attention_one(q_vec64, K64, V64, scale: float) -> np.ndarray:
    """Textbook single-query softmax attention in fp64:
        x_j = scale * <q, k_j>;  m = max_j x_j;  p_j = exp(x_j - m)
        o   = sum_j p_j v_j / sum_j p_j
    An empty context gives the zero vector (a reading: the pages always
    attend over at least one token)."""
    if K64.shape[0] == 0:
        return np.zeros(V64.shape[1], dtype=np.float64)
    x = scale * (K64 @ q_vec64)
    m = x.max()
    p = np.exp(x - m)
    return (p @ V64) / p.sum()


def decode_attention(q, key_cache, value_cache, block_tables, seq_lens,
                     scale: float, num_kv_heads: int, block_size: int,
                     dtype: str, seqs=None, heads=None, window: int = 0) -> np.ndarray:
    """Paged decode attention for every (sequence, query head), or for the
    listed subsets. Query head h reads KV head h // (Hq / Hkv) (contiguous
    groups; [P3] §2.1: 64 query heads share 8 KV heads).

    The pages state that paging keeps dense attention semantics ([P4] last
    section; [P2]: the kernel reads block by block, so blocks need not be
    contiguous). The oracle therefore gathers each sequence's K and V through
    its block table into contiguous arrays and runs dense attention on them.

    window > 0: sliding-window attention over tokens window_start .. L-1.

    Returns float64 [S, Hq, D] (rows outside `seqs`/`heads` stay zero)."""
    S, Hq, D = q.shape
    assert Hq % num_kv_heads == 0
    g = Hq // num_kv_heads
    q64 = upcast(q, dtype)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    seqs = range(S) if seqs is None else seqs
    heads = range(Hq) if heads is None else heads
    for s in seqs:
        L = int(seq_lens[s])
        lo = window_start(L, window)
        by_kv = {}
        for h in heads:
            kvh = h // g
            if kvh not in by_kv:
                by_kv[kvh] = (
                    gather_kv(key_cache, block_tables[s], L, kvh, block_size, dtype, lo),
                    gather_kv(value_cache, block_tables[s], L, kvh, block_size, dtype, lo))
            K, V = by_kv[kvh]
            out[s, h] = decode_attention_one(q64[s, h], K, V, scale)
    return out


def decode_step(q, k_new, v_new, key_cache, value_cache, block_tables,
                context_lens, scale: float, num_kv_heads: int,
                block_size: int, dtype: str, seqs=None, heads=None):
    """One decode step as the build reads the pages' order: the new token's
    slot is computed from its position (= cached context length), its K/V are
    written there, then it attends over context + 1 tokens including itself.
    Mutates the caches (caller passes copies). Returns (slots, out fp64)."""
    S = q.shape[0]
    qsl = np.arange(S + 1, dtype=np.int64)
    pos = np.asarray(context_lens, dtype=np.int64)
    slots = slot_mapping(qsl, pos, block_tables, block_size)
    reshape_and_cache(k_new, v_new, slots, key_cache, value_cache, block_size)
    seq_lens = pos + 1
    out = decode_attention(q, key_cache, value_cache, block_tables, seq_lens,
                           scale, num_kv_heads, block_size, dtype, seqs, heads)
    return slots, out


# --------------------------------------------------------------------------
# hybrid block sizes ([P1] §3.4 map_to_kernel_blocks)
# --------------------------------------------------------------------------
def map_to_kernel_blocks(manager_ids, blocks_per_kv_block: int) -> np.ndarray:
    """Each allocator ("manager") block of r = blocks_per_kv_block kernel
    blocks expands to kernel ids k*r, k*r + 1, ..., k*r + r - 1, in order
    ([P1] §3.4: ids [0, 1, 2] with r = 2 give [0, 1, 2, 3, 4, 5]). A negative
    (unassigned) manager id expands to r entries of -1."""
    r = int(blocks_per_kv_block)
    assert r >= 1
    out = []
    for k in np.asarray(manager_ids, dtype=np.int64).reshape(-1):
        k = int(k)
        for i in range(r):
            out.append(-1 if k < 0 else k * r + i)
    return np.asarray(out, dtype=np.int64)


# --------------------------------------------------------------------------
# several new tokens per sequence (chunked prefill / speculative tokens)
# --------------------------------------------------------------------------
def multi_query_attention(q, key_cache, value_cache, block_tables, query_start_loc,
                          seq_lens, scale: float, num_kv_heads: int, block_size: int,
                          dtype: str) -> np.ndarray:
    """Causal paged attention for n_s = qsl[s+1] - qsl[s] new tokens of each
    sequence, whose K/V are already in the pool ([P3] §2.5: the scheduler
    gives each request a token budget that covers chunked prefill and
    speculative tokens alike; the slot mapping of [P1] §2.3 handles many
    tokens per request). Sequence s holds L_s = seq_lens[s] tokens including
    the new ones, so new token i sits at position L_s - n_s + i and attends to
    positions 0 .. L_s - n_s + i. With n_s = 1 this is decode attention.
    q: [T, Hq, D] with T = qsl[-1]. Returns float64 [T, Hq, D]."""
    T, Hq, D = q.shape
    g = Hq // num_kv_heads
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    q64 = upcast(q, dtype)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    for s in range(len(qsl) - 1):
        n = int(qsl[s + 1] - qsl[s])
        L = int(seq_lens[s])
        if n == 0:
            continue
        if n > L:
            raise ValueError(f"sequence {s}: {n} new tokens but length {L}")
        for kvh in range(num_kv_heads):
            K = gather_kv(key_cache, block_tables[s], L, kvh, block_size, dtype)
            V = gather_kv(value_cache, block_tables[s], L, kvh, block_size, dtype)
            for i in range(n):
                last = L - n + i
                for h in range(kvh * g, (kvh + 1) * g):
                    out[qsl[s] + i, h] = decode_attention_one(
                        q64[qsl[s] + i, h], K[:last + 1], V[:last + 1], scale)
    return out


# --------------------------------------------------------------------------
# fp8 (e4m3) KV blocks ([P1] §3.5 AttentionSpec.kv_quant_mode; §7 outlook on
# quantisation-aware blocks). The pages fix no format; the reading taken is
# OCP FP8 E4M3 codes with one fp32 scale per pool (K and V each):
#     code = e4m3(x / scale) with round-to-nearest-even and saturation to
#            +-448; value = decode(code) * scale.
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 is subnormal m * 2^-9; S.1111.111 is NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = sign * val
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(x32) -> np.ndarray:
    """Nearest E4M3 code of float32 values, ties to the even code, values
    beyond the largest finite magnitude (448) saturate to it, NaN -> 0x7F."""
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    flat, res = x.reshape(-1), out.reshape(-1)
    for idx, v in enumerate(flat):
        if np.isnan(v):
            res[idx] = 0x7F
            continue
        s = 0x80 if np.signbit(v) else 0
        a = abs(v)
        if a >= 448.0:
            res[idx] = s | 0x7E
            continue
        if a < 2.0 ** -6:                           # subnormal range
            q = int(np.rint(a / 2.0 ** -9))         # 8 becomes the smallest normal
            res[idx] = s | q
            continue
        mant, exp = np.frexp(a)                     # a = mant * 2^exp, mant in [0.5, 1)
        e = exp - 1                                 # a = (2 * mant) * 2^e
        q = int(np.rint((2.0 * mant - 1.0) * 8.0))
        if q == 8:
            e, q = e + 1, 0
        code = ((e + 7) << 3) | q
        res[idx] = s | min(code, 0x7E)
    return out


def quantize_e4m3(x, dtype: str, scale: float) -> np.ndarray:
    """Codes for stored values x: widened exactly to fp32, divided by the fp32
    scale with fp32 rounding, then encoded."""
    x32 = upcast(x, dtype).astype(np.float32)
    return e4m3_encode(x32 / np.float32(scale))


def reshape_and_cache_fp8(k, v, slots, key_cache8, value_cache8, block_size: int,
                          dtype: str, k_scale: float, v_scale: float):
    """KV write into e4m3 pools: quantise, then the same slot placement as
    reshape_and_cache."""
    reshape_and_cache(quantize_e4m3(k, dtype, k_scale), quantize_e4m3(v, dtype, v_scale),
                      slots, key_cache8, value_cache8, block_size)


def decode_attention_fp8(q, key_cache8, value_cache8, block_tables, seq_lens, scale: float,
                         num_kv_heads: int, block_size: int, dtype: str, k_scale: float,
                         v_scale: float, seqs=None, heads=None, window: int = 0) -> np.ndarray:
    """Decode attention over e4m3 pools: K = decode(code) * k_scale and
    V = decode(code) * v_scale exactly in fp64, then decode_attention
    (window as there)."""
    S, Hq, D = q.shape
    g = Hq // num_kv_heads
    q64 = upcast(q, dtype)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        L = int(seq_lens[s])
        j = np.arange(window_start(L, window), L)
        blk = np.asarray(block_tables[s], dtype=np.int64)[j // block_size]
        for h in (range(Hq) if heads is None else heads):
            kvh = h // g
            K = e4m3_decode(key_cache8[blk, kvh, j % block_size, :]) * np.float64(np.float32(k_scale))
            V = e4m3_decode(value_cache8[blk, kvh, j % block_size, :]) * np.float64(np.float32(v_scale))
            out[s, h] = decode_attention_one(q64[s, h], K, V, scale)
    return out


# --------------------------------------------------------------------------
# fp8 blocks that carry their own scales ([P1] §3.5 kv_quant_mode; §7.4 the
# compression-aware block: quantisation tied to the block). Readings (the
# pages fix no format): one scale per (physical block, KV head) for K and one
# for V, a power of two, fixed by the KV write that stores the block's first
# row from the largest magnitude among the tokens that this write puts into
# that block (row 0 and the rows right after it, in consecutive slots);
# every later write into the block quantises with the stored scale. The
# scale 2^k is the smallest power of two with amax / 2^k <= 128, i.e.
# k = ceil(log2(amax)) - 7, so the first tokens' largest magnitude lands in
# (64, 128] and later tokens have 3.5x headroom before the largest finite
# code (448). k is kept in [-126, 127] (normal fp32 powers of two); amax = 0
# gives 1. NaN elements are left out of the maximum.
# --------------------------------------------------------------------------
def block_scale_e4m3(amax: float) -> float:
    """Power-of-two scale for a block whose first tokens' largest magnitude
    is amax (>= 0; inf allowed)."""
    a = float(amax)
    assert a >= 0.0
    if a == 0.0:
        return 1.0
    if math.isinf(a):
        k = 127
    else:
        mant, exp = math.frexp(a)          # a = mant * 2^exp, mant in [0.5, 1)
        ceil_log2 = exp - 1 if mant == 0.5 else exp
        k = min(max(ceil_log2 - 7, -126), 127)
    return math.ldexp(1.0, k)


def reshape_and_cache_fp8_block_scaled(k, v, slots, key_cache8, value_cache8, k_scales,
                                       v_scales, block_size: int, dtype: str):
    """KV write into e4m3 pools whose blocks carry their own scales
    (k_scales / v_scales: float32 [num_blocks, num_kv_heads], updated in
    place). Two passes over the call's tokens:
      1. a token whose slot is row 0 of its block fixes that block's scales
         from the largest |value| over it and the tokens that follow it in
         this call in consecutive slots of the same block (at most B);
      2. every token (slot >= 0) is quantised with its block's scale, as in
         quantize_e4m3, at its slot."""
    B = block_size
    slots = np.asarray(slots, dtype=np.int64)
    T = len(slots)
    Hkv = key_cache8.shape[1]
    for t in range(T):
        s0 = int(slots[t])
        if s0 < 0 or s0 % B != 0:
            continue
        n = 1
        while n < B and t + n < T and int(slots[t + n]) == s0 + n:
            n += 1
        blk = s0 // B
        for h in range(Hkv):
            for src, dst in ((k, k_scales), (v, v_scales)):
                run = np.abs(upcast(np.ascontiguousarray(src[t:t + n, h]), dtype))
                amax = float(np.nanmax(run)) if not np.isnan(run).all() else 0.0
                dst[blk, h] = block_scale_e4m3(amax)
    for t in range(T):
        s = int(slots[t])
        if s < 0:
            continue
        blk, row = s // B, s % B
        for h in range(Hkv):
            key_cache8[blk, h, row] = quantize_e4m3(k[t, h], dtype, float(k_scales[blk, h]))
            value_cache8[blk, h, row] = quantize_e4m3(v[t, h], dtype, float(v_scales[blk, h]))


def decode_attention_fp8_block_scaled(q, key_cache8, value_cache8, k_scales, v_scales,
                                      block_tables, seq_lens, scale: float, num_kv_heads: int,
                                      block_size: int, dtype: str, seqs=None, heads=None,
                                      window: int = 0) -> np.ndarray:
    """Decode attention over e4m3 pools with per-(block, KV head) scales:
    K_s[j] = decode(code) * k_scales[block of j, kvh], likewise V, exactly in
    fp64; then decode_attention_one (window as in decode_attention)."""
    S, Hq, D = q.shape
    g = Hq // num_kv_heads
    q64 = upcast(q, dtype)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        L = int(seq_lens[s])
        j = np.arange(window_start(L, window), L)
        blk = np.asarray(block_tables[s], dtype=np.int64)[j // block_size]
        for h in (range(Hq) if heads is None else heads):
            kvh = h // g
            ks = np.asarray(k_scales, dtype=np.float64)[blk, kvh][:, None]
            vs = np.asarray(v_scales, dtype=np.float64)[blk, kvh][:, None]
            K = e4m3_decode(key_cache8[blk, kvh, j % block_size, :]) * ks
            V = e4m3_decode(value_cache8[blk, kvh, j % block_size, :]) * vs
            out[s, h] = decode_attention_one(q64[s, h], K, V, scale)
    return out
