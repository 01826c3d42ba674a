"""Full-size workloads in the launch configuration the benchmark times
(automatic partitioning): every slot and every written cache byte is checked,
and attention is checked element by element on sampled (sequence, head)
pairs that the oracle computes one by one."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, bytes_equal, max_abs_err, np_, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"

NAMES = ["llama7b", "gqa72b"] + [f"longctx_B{b}" for b in (8, 16, 32, 64, 128)]


@pytest.mark.parametrize("name", NAMES)
def test_full_size_step(name):
    pa.pa_get_device_error()
    inp = workloads.make_decode_inputs(name, device=DEV)
    cfg = inp.cfg
    # host copies of the pre-step inputs for the oracle
    host = {k: np_(getattr(inp, k)) for k in ("q", "k_new", "v_new", "key_cache",
                                              "value_cache", "block_tables")}
    g = to_dev(inp)
    slots = pa.pa_compute_slot_mapping(g["query_start_loc"], g["positions"],
                                       g["block_tables"], cfg.block_size)
    pa.pa_reshape_and_cache(g["k_new"], g["v_new"], slots, g["key_cache"], g["value_cache"])
    out = pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                                 g["seq_lens"], inp.scale, cfg.num_kv_heads,
                                 max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0

    lens = inp.seq_lens.cpu().numpy()
    rng = np.random.default_rng(0)
    seqs = sorted({int(lens.argmax()), int(lens.argmin()),
                   *rng.choice(cfg.num_seqs, size=min(4, cfg.num_seqs), replace=False).tolist()})
    heads = sorted({0, cfg.num_q_heads - 1,
                    *rng.choice(cfg.num_q_heads, size=2, replace=False).tolist()})
    kc, vc = host["key_cache"], host["value_cache"]
    slots_o, out_o = oracle.decode_step(host["q"], host["k_new"], host["v_new"], kc, vc,
                                        host["block_tables"], inp.context_lens.numpy(),
                                        inp.scale, cfg.num_kv_heads, cfg.block_size,
                                        cfg.dtype, seqs, heads)
    assert np.array_equal(slots.cpu().numpy(), slots_o)
    assert bytes_equal(g["key_cache"], kc) and bytes_equal(g["value_cache"], vc)
    err = max_abs_err(out, out_o, seqs, heads)
    assert err <= TOL[cfg.dtype], err
    # every output row is finite and every sequence produced something
    assert torch.isfinite(out.float()).all()
