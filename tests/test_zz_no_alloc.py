"""pa_decode_attention_static: the decode attention entry point for callers
that cannot allocate device memory (an engine that gave nearly all of HBM to
its KV block pool up front, or a host that forbids cudaMalloc on the decode
path because it can stall the device). It takes its scratch from a fixed
array inside the library instead of a caller workspace.

These tests call it through the C ABI and compare it with
pa_decode_attention on the same inputs, bit for bit (both calls resolve the
same partitioning, so the results must be identical), on two calls in a row,
and after a larger call has left many more partitions' partials in the shared
array than the checked call writes. One case is also checked against the
oracle. The file is named so pytest collects it last."""
import ctypes
import os
import re

import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from paged_kv_cache_123_gb300._lib import DTYPE_CODE, lib
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scratch_bytes_from_header():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "include", "pagedattn.h")
    m = re.search(r"#define\s+PA_STATIC_SCRATCH_BYTES\s+\((\d+)ll\s*<<\s*(\d+)\)",
                  open(path).read())
    assert m, "PA_STATIC_SCRATCH_BYTES not found in the header"
    return int(m.group(1)) << int(m.group(2))


PA_STATIC_SCRATCH_BYTES = _scratch_bytes_from_header()


def _inputs(cfg):
    inp = workloads.make_decode_inputs(cfg)
    g = {"q": inp.q.to(DEV), "kc": inp.key_cache.to(DEV), "vc": inp.value_cache.to(DEV),
         "tables": inp.block_tables.to(DEV), "lens": inp.seq_lens.to(DEV)}
    return inp, g


def _static_call(g, cfg, inp, out, partition):
    stream = torch.cuda.current_stream().cuda_stream
    return lib().pa_decode_attention_static(
        g["q"].data_ptr(), g["kc"].data_ptr(), g["vc"].data_ptr(), g["tables"].data_ptr(),
        g["tables"].shape[1], g["lens"].data_ptr(), cfg.num_seqs, cfg.num_q_heads,
        cfg.num_kv_heads, cfg.head_size, cfg.block_size, inp.num_blocks,
        DTYPE_CODE[g["q"].dtype], ctypes.c_float(inp.scale), inp.max_seq_len, partition,
        out.data_ptr(), stream)


def _with_workspace(g, cfg, inp, partition):
    # a caller-owned workspace full of garbage, like the shared array
    need = pa.pa_decode_workspace_bytes(cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads,
                                        cfg.head_size, cfg.block_size, inp.max_seq_len,
                                        partition)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device=DEV)
    return pa.pa_decode_attention(g["q"], g["kc"], g["vc"], g["tables"], g["lens"],
                                  inp.scale, cfg.num_kv_heads, max_seq_len=inp.max_seq_len,
                                  partition_size=partition, workspace=ws)


def _splits(cfg, inp, partition):
    return pa.pa_decode_partitioning(cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads,
                                     cfg.block_size, inp.max_seq_len, partition)[0]


@pytest.mark.parametrize("dtype,partition", [("bf16", 256), ("f16", 0), ("f32", 64)])
def test_static_scratch_matches_workspace_entry_point(dtype, partition):
    cfg = workloads.DecodeConfig("noalloc", 6, 16, 2, 128, 16, dtype, ctx_lo=1,
                                 ctx_hi=3000, seed=404)
    inp, g = _inputs(cfg)
    need = pa.pa_decode_workspace_bytes(cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads,
                                        cfg.head_size, cfg.block_size, inp.max_seq_len,
                                        partition)
    assert 0 < need <= PA_STATIC_SCRATCH_BYTES
    want = _with_workspace(g, cfg, inp, partition)
    for call in range(2):
        out = torch.full_like(g["q"], float("nan"))
        assert _static_call(g, cfg, inp, out, partition) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, want), call
    assert pa.pa_get_device_error() == 0
    if dtype == "bf16":
        ref = oracle.decode_attention(np_(inp.q), np_(inp.key_cache), np_(inp.value_cache),
                                      inp.block_tables.numpy(), inp.seq_lens.numpy(),
                                      inp.scale, cfg.num_kv_heads, cfg.block_size, dtype)
        assert max_abs_err(out, ref) <= TOL[dtype]


def test_leftovers_of_a_larger_call_do_not_leak():
    # the first call fills the shared array with the partials of many short
    # partitions; the second writes far fewer and must not read any of them
    big = workloads.DecodeConfig("noalloc_big", 8, 16, 4, 128, 16, "bf16", ctx_lo=5000,
                                 ctx_hi=6000, seed=405)
    small = workloads.DecodeConfig("noalloc_small", 5, 16, 4, 128, 16, "bf16", ctx_lo=300,
                                   ctx_hi=1500, seed=406)
    ib, gb = _inputs(big)
    isml, gs = _inputs(small)
    assert _splits(big, ib, 64) > 4 * _splits(small, isml, 512) > 4
    want_big = _with_workspace(gb, big, ib, 64)
    want_small = _with_workspace(gs, small, isml, 512)
    for _ in range(2):
        out_b = torch.full_like(gb["q"], float("nan"))
        assert _static_call(gb, big, ib, out_b, 64) == 0
        out_s = torch.full_like(gs["q"], float("nan"))
        assert _static_call(gs, small, isml, out_s, 512) == 0
        torch.cuda.synchronize()
        assert torch.equal(out_b, want_big)
        assert torch.equal(out_s, want_small)
    assert pa.pa_get_device_error() == 0
    ref = oracle.decode_attention(np_(isml.q), np_(isml.key_cache), np_(isml.value_cache),
                                  isml.block_tables.numpy(), isml.seq_lens.numpy(),
                                  isml.scale, small.num_kv_heads, small.block_size, "bf16")
    assert max_abs_err(out_s, ref) <= TOL["bf16"]


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
