"""Hybrid block sizes ("PagedAttention 核心创新深度分析" §3.4): allocator
blocks of r kernel blocks, expanded to a kernel-block table on the GPU and
read by the attention kernels with the kernel block size."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("r", [1, 2, 3, 8])
def test_expansion_bit_exact(r):
    rng = np.random.default_rng(r)
    tab = rng.integers(0, 5000, size=(37, 19)).astype(np.int32)
    tab[rng.random(tab.shape) < 0.2] = -1
    got = pa.pa_map_to_kernel_blocks(torch.from_numpy(tab).to(DEV), r).cpu().numpy()
    for i in range(tab.shape[0]):
        assert got[i].tolist() == oracle.map_to_kernel_blocks(tab[i], r).tolist()
    assert pa.pa_get_device_error() == 0


def test_pages_example_on_gpu():
    t = torch.tensor([[0, 1, 2]], dtype=torch.int32, device=DEV)
    assert pa.pa_map_to_kernel_blocks(t, 2).cpu().tolist() == [[0, 1, 2, 3, 4, 5]]


@pytest.mark.parametrize("dtype,G", [("bf16", 8), ("f16", 1)])
def test_attention_through_expanded_tables(dtype, G):
    """Sequences own allocator blocks of 64 tokens (r = 4 kernel blocks of 16);
    attention reads the expanded table and matches the oracle."""
    r, B, Hkv = 4, 16, 2
    lens = [1, 63, 64, 65, 300]
    nmgr = [-(-L // (B * r)) for L in lens]
    rng = np.random.default_rng(11)
    mgr_pool = 12
    ids = rng.permutation(mgr_pool)
    mtab = -np.ones((len(lens), max(nmgr)), dtype=np.int32)
    off = 0
    for s, n in enumerate(nmgr):
        mtab[s, :n] = ids[off:off + n]
        off += n
    NB = mgr_pool * r
    cfg = workloads.DecodeConfig("hyb", len(lens), Hkv * G, Hkv, 128, B, dtype, seed=12)
    gen = torch.Generator().manual_seed(12)
    dt = workloads.DTYPES[dtype]
    kc = torch.empty(NB, Hkv, B, 128, dtype=dt)
    vc = torch.empty_like(kc)
    q = torch.empty(len(lens), Hkv * G, 128, dtype=dt)
    for t in (kc, vc, q):
        workloads.randn_into(t, gen)
    ktab = pa.pa_map_to_kernel_blocks(torch.from_numpy(mtab).to(DEV), r)
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = pa.pa_decode_attention(q.to(DEV), kc.to(DEV), vc.to(DEV), ktab, seq_lens,
                                 128 ** -0.5, Hkv, max_seq_len=max(lens))
    otab = np.stack([oracle.map_to_kernel_blocks(row, r) for row in mtab])
    want = oracle.decode_attention(np_(q), np_(kc), np_(vc), otab, np.array(lens),
                                   128 ** -0.5, Hkv, B, dtype)
    assert max_abs_err(out, want) <= TOL[dtype]
    assert pa.pa_get_device_error() == 0
