"""A whole multi-layer decode step captured once as a CUDA graph and
replayed ("vLLM 的 PagedAttention：显存管理如何撑起大模型推理" §2.6: the decode
step is graph-captured to remove launch overhead). The C ABI calls allocate
nothing and never synchronise, so every kernel of the step is captured; the
replay must reproduce the eager step bit for bit and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 32, 8), ("f16", 8, 8)])
def test_multilayer_step_graph_replay(dtype, hq, hkv):
    layers = 4
    cfg = workloads.DecodeConfig("graph", 6, hq, hkv, 128, 16, dtype, ctx_lo=10, ctx_hi=900,
                                 seed=77)
    base = workloads.make_decode_inputs(cfg)
    pools = [workloads.make_decode_inputs(cfg, seed=100 + l,
                                         context_lens=base.context_lens.tolist())
             for l in range(layers)]
    assert all(p.num_blocks == base.num_blocks for p in pools)
    kcs = [p.key_cache.to(DEV) for p in pools]
    vcs = [p.value_cache.to(DEV) for p in pools]
    host_k = [np_(p.key_cache) for p in pools]
    host_v = [np_(p.value_cache) for p in pools]
    qs = [p.q.to(DEV) for p in pools]
    kn = [p.k_new.to(DEV) for p in pools]
    vn = [p.v_new.to(DEV) for p in pools]
    tables = base.block_tables.to(DEV)
    lens = base.seq_lens.to(DEV)
    pos = base.positions.to(DEV)
    qsl = base.query_start_loc.to(DEV)
    S = cfg.num_seqs
    slots = torch.empty(S, dtype=torch.int64, device=DEV)
    outs = [torch.empty_like(q) for q in qs]
    need = pa.pa_decode_workspace_bytes(S, hq, hkv, 128, 16, base.max_seq_len, 256)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=DEV)

    def step():
        pa.pa_compute_slot_mapping(qsl, pos, tables, 16, slot_mapping=slots)
        for l in range(layers):
            pa.pa_reshape_and_cache(kn[l], vn[l], slots, kcs[l], vcs[l])
            pa.pa_decode_attention(qs[l], kcs[l], vcs[l], tables, lens, base.scale, hkv,
                                   outs[l], max_seq_len=base.max_seq_len,
                                   partition_size=256, workspace=ws)

    step()                                   # eager (also first-call set-up)
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):                       # the KV write is idempotent
        g.replay()
    torch.cuda.synchronize()
    for l in range(layers):
        assert torch.equal(outs[l].view(torch.int16), eager[l].view(torch.int16)), l
    assert pa.pa_get_device_error() == 0
    # layer 0 against the oracle's own step
    _, want = oracle.decode_step(np_(pools[0].q), np_(pools[0].k_new), np_(pools[0].v_new),
                                 host_k[0], host_v[0], np_(base.block_tables),
                                 base.context_lens.numpy(), base.scale, hkv, 16, dtype)
    assert max_abs_err(outs[0], want) <= TOL[dtype]
