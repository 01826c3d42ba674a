"""Seeded synthetic inputs for the paged-KV decode step.

This module only draws inputs: sequence lengths, a shuffled physical block
assignment, queries, new keys/values and the initial pool contents. It holds
none of the arithmetic the decode step performs (no slot computation, no
attention), so both the CUDA path and the CPU oracle can be fed from it.

Shapes follow the workloads the pages discuss: a Llama-7B-shaped layer
(32 heads, head size 128, fp16), a 72B-class GQA layer (64 query heads over 8
KV heads, "PagedAttention: 显存管理如何撑起大模型推理" §2.1), a shared-prefix
parallel-sampling batch and 32k long contexts. Values are N(0, 1) drawn in fp32
and rounded to the storage dtype; block ids come from a seeded permutation of
the pool, so logically adjacent blocks sit at unrelated physical places.

Pool layout used everywhere in this package:
    key_cache, value_cache : [num_blocks, num_kv_heads, block_size, head_size]
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


@dataclasses.dataclass
class DecodeConfig:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: str
    ctx_lo: int = 0               # cached context length range (inclusive)
    ctx_hi: int = 0
    ctx_fixed: Optional[list] = None
    pool_slack: float = 1.10      # pool = ceil(need * slack) blocks
    num_blocks: Optional[int] = None
    seed: int = 1000


# Named workloads. "context" = tokens already in the pool before the step; the
# step appends one token per sequence, so the attended length is context + 1.
CONFIGS: Dict[str, DecodeConfig] = {
    "tiny": DecodeConfig("tiny", 2, 4, 4, 64, 4, "f32", ctx_fixed=[7, 9],
                         num_blocks=8, seed=1000),
    "llama7b": DecodeConfig("llama7b", 64, 32, 32, 128, 16, "f16",
                            ctx_lo=128, ctx_hi=2048, seed=1001),
    "gqa72b": DecodeConfig("gqa72b", 128, 64, 8, 128, 16, "bf16",
                           ctx_lo=1024, ctx_hi=8192, seed=1002),
}
for _b in (8, 16, 32, 64, 128):
    CONFIGS[f"longctx_B{_b}"] = DecodeConfig(
        f"longctx_B{_b}", 16, 32, 8, 128, _b, "bf16",
        ctx_fixed=[32768] * 16, pool_slack=1.0, seed=1004)


@dataclasses.dataclass
class DecodeInputs:
    cfg: DecodeConfig
    context_lens: torch.Tensor    # int64 [S] tokens cached before the step
    seq_lens: torch.Tensor        # int32 [S] tokens attended (context + 1)
    num_blocks: int
    block_tables: torch.Tensor    # int32 [S, max_blocks]; -1 past the end
    positions: torch.Tensor       # int64 [S] position of the new token
    query_start_loc: torch.Tensor  # int32 [S + 1] (one new token per seq)
    q: torch.Tensor               # [S, Hq, D]
    k_new: torch.Tensor           # [S, Hkv, D]
    v_new: torch.Tensor           # [S, Hkv, D]
    key_cache: torch.Tensor       # [NB, Hkv, B, D]
    value_cache: torch.Tensor     # [NB, Hkv, B, D]
    scale: float

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0


def _blocks_for(length: int, block_size: int) -> int:
    # number of pool blocks a sequence of `length` tokens occupies; used only
    # to size the synthetic assignment, never as an expected value
    return -(-length // block_size)


def randn_into(out: torch.Tensor, gen: torch.Generator, chunk_rows: int = 1 << 14):
    """Fill `out` (any float dtype) with N(0,1) drawn in fp32, row chunk by
    row chunk along dim 0 so the fp32 staging stays small."""
    n = out.shape[0]
    for i in range(0, n, chunk_rows):
        j = min(n, i + chunk_rows)
        tmp = torch.randn((j - i,) + tuple(out.shape[1:]), generator=gen,
                          dtype=torch.float32, device=out.device)
        out[i:j].copy_(tmp.to(out.dtype))


def make_decode_inputs(cfg: DecodeConfig | str, device: str = "cpu",
                       seed: Optional[int] = None,
                       context_lens: Optional[list] = None) -> DecodeInputs:
    """Draw one decode step's inputs from torch.Generators seeded from the
    config (or `seed`). The batch's structure — context lengths and the
    block permutation — comes from a CPU generator, so it is the same on
    every device (the GPU bench and the CPU oracle time the same batch); the
    values (q, new K/V, pool contents) are drawn on `device`."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    seed = cfg.seed if seed is None else seed
    gcpu = torch.Generator().manual_seed(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1)
    S, B = cfg.num_seqs, cfg.block_size
    if context_lens is not None:
        ctx = torch.tensor(context_lens, dtype=torch.int64)
    elif cfg.ctx_fixed is not None:
        ctx = torch.tensor(cfg.ctx_fixed, dtype=torch.int64)
    else:
        ctx = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (S,), generator=gcpu,
                            dtype=torch.int64)
    seq_lens = (ctx + 1).to(torch.int32)
    nblk = [_blocks_for(int(x), B) for x in seq_lens.tolist()]
    need = sum(nblk)
    if cfg.num_blocks is not None:
        nb = cfg.num_blocks
    else:
        nb = max(need, int(math.ceil(need * cfg.pool_slack)))
    assert nb >= need, "pool too small for the drawn lengths"
    perm = torch.randperm(nb, generator=gcpu)
    mb = max(nblk) if nblk else 1
    tables = torch.full((S, mb), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[off:off + n].to(torch.int32)
        off += n
    dt = DTYPES[cfg.dtype]
    Hq, Hkv, D = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_size
    q = torch.empty((S, Hq, D), dtype=dt, device=device)
    k_new = torch.empty((S, Hkv, D), dtype=dt, device=device)
    v_new = torch.empty((S, Hkv, D), dtype=dt, device=device)
    randn_into(q, gen)
    randn_into(k_new, gen)
    randn_into(v_new, gen)
    kc = torch.empty((nb, Hkv, B, D), dtype=dt, device=device)
    vc = torch.empty((nb, Hkv, B, D), dtype=dt, device=device)
    rows = max(1, (1 << 24) // max(1, Hkv * B * D))
    randn_into(kc, gen, rows)
    randn_into(vc, gen, rows)
    return DecodeInputs(
        cfg=cfg, context_lens=ctx, seq_lens=seq_lens.to(device),
        num_blocks=nb, block_tables=tables.to(device),
        positions=ctx.clone().to(device),
        query_start_loc=torch.arange(S + 1, dtype=torch.int32).to(device),
        q=q, k_new=k_new, v_new=v_new, key_cache=kc, value_cache=vc,
        scale=1.0 / math.sqrt(D))


def make_random_prefill_batch(num_reqs: int, max_tokens_per_req: int,
                              block_size: int, num_blocks: int, seed: int,
                              max_blocks_per_req: Optional[int] = None):
    """A ragged multi-token batch for slot mapping: each request gets a random
    number of new tokens (0 allowed) at consecutive positions after a random
    number of cached tokens, and a table row drawn from a permutation.

    Returns (query_start_loc int32 [R+1], positions int64 [T],
    block_table int32 [R, MB]); all on CPU."""
    gen = torch.Generator().manual_seed(seed)
    n_new = torch.randint(0, max_tokens_per_req + 1, (num_reqs,), generator=gen)
    cached = torch.randint(0, 3 * max_tokens_per_req + 1, (num_reqs,),
                           generator=gen)
    total = cached + n_new
    nblk = [_blocks_for(int(x), block_size) for x in total.tolist()]
    mb = max_blocks_per_req or max(1, max(nblk) if nblk else 1)
    assert sum(nblk) <= num_blocks
    perm = torch.randperm(num_blocks, generator=gen)
    table = torch.full((num_reqs, mb), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(nblk):
        table[r, :n] = perm[off:off + n].to(torch.int32)
        off += n
    qsl = torch.zeros(num_reqs + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(n_new, 0).to(torch.int32)
    pos = []
    for r in range(num_reqs):
        c, n = int(cached[r]), int(n_new[r])
        pos.extend(range(c, c + n))
    positions = torch.tensor(pos, dtype=torch.int64)
    return qsl, positions, table
