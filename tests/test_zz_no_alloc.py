"""pa_decode_attention_static: the decode attention entry point for callers
that cannot allocate device memory (an engine that gave nearly all of HBM to
its KV block pool up front, or a host that forbids cudaMalloc on the decode
path because it can stall the device). It takes its scratch from a fixed
array inside the library instead of a caller workspace.

These tests call it through the C ABI and compare it with
pa_decode_attention on the same inputs, on two calls in a row (the array is
shared by all calls and keeps the previous call's contents). The file is
named so pytest collects it last."""
import ctypes

import pytest
import torch

import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from paged_kv_cache_123_gb300._lib import DTYPE_CODE, lib
from tests.helpers import TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"
PA_STATIC_SCRATCH_BYTES = 32 << 20


def _static_call(g, cfg, inp, out, partition):
    stream = torch.cuda.current_stream().cuda_stream
    return lib().pa_decode_attention_static(
        g["q"].data_ptr(), g["kc"].data_ptr(), g["vc"].data_ptr(), g["tables"].data_ptr(),
        g["tables"].shape[1], g["lens"].data_ptr(), cfg.num_seqs, cfg.num_q_heads,
        cfg.num_kv_heads, cfg.head_size, cfg.block_size, inp.num_blocks,
        DTYPE_CODE[g["q"].dtype], ctypes.c_float(inp.scale), inp.max_seq_len, partition,
        out.data_ptr(), stream)


@pytest.mark.parametrize("dtype,partition", [("bf16", 256), ("f16", 0), ("f32", 64)])
def test_static_scratch_matches_workspace_entry_point(dtype, partition):
    cfg = workloads.DecodeConfig("noalloc", 6, 16, 2, 128, 16, dtype, ctx_lo=1,
                                 ctx_hi=3000, seed=404)
    inp = workloads.make_decode_inputs(cfg)
    g = {"q": inp.q.to(DEV), "kc": inp.key_cache.to(DEV), "vc": inp.value_cache.to(DEV),
         "tables": inp.block_tables.to(DEV), "lens": inp.seq_lens.to(DEV)}
    need = pa.pa_decode_workspace_bytes(cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads,
                                        cfg.head_size, cfg.block_size, inp.max_seq_len,
                                        partition)
    assert need <= PA_STATIC_SCRATCH_BYTES
    want = pa.pa_decode_attention(g["q"], g["kc"], g["vc"], g["tables"], g["lens"],
                                  inp.scale, cfg.num_kv_heads, max_seq_len=inp.max_seq_len,
                                  partition_size=partition).float()
    for call in range(2):
        out = torch.full_like(g["q"], float("nan"))
        assert _static_call(g, cfg, inp, out, partition) == 0
        torch.cuda.synchronize()
        err = (out.float() - want).abs().max().item()
        assert err <= TOL[dtype], (call, err)
    assert pa.pa_get_device_error() == 0


def test_static_scratch_refuses_oversized_problems():
    # 4096 sequences x 64 heads x 64 partitions of fp32 partials is far past
    # the fixed array; the call must refuse before launching anything
    cfg = workloads.DecodeConfig("big", 4096, 64, 8, 128, 16, "bf16")
    need = pa.pa_decode_workspace_bytes(4096, 64, 8, 128, 16, 64 * 64, 64)
    assert need > PA_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    p = dummy.data_ptr()
    st = lib().pa_decode_attention_static(p, p, p, p, 256, p, cfg.num_seqs, 64, 8, 128, 16,
                                          1, 2, ctypes.c_float(1.0), 64 * 64, 64, p,
                                          torch.cuda.current_stream().cuda_stream)
    assert st == -4
