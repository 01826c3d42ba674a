"""Failure detection without a GPU fault: a bounded wait on a barrier phase
nothing completes gives up after its limit, raises the CTA's abort flag and
lets the other waiter leave; the context stays usable and the next call is
exact."""
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import max_abs_err, np_

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cycles", [100_000, 2_000_000])
def test_bounded_wait_gives_up_and_the_context_stays_usable(cycles):
    assert pa.pa_selftest_bounded_wait(cycles) == [-10, -10, 1]
    # the device is still usable: a decode step right after is exact
    inp = workloads.make_decode_inputs("tiny")
    out = pa.pa_decode_attention(inp.q.cuda(), inp.key_cache.cuda(), inp.value_cache.cuda(),
                                 inp.block_tables.cuda(), inp.seq_lens.cuda(), inp.scale,
                                 inp.cfg.num_kv_heads, max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    want = oracle.decode_attention(np_(inp.q), np_(inp.key_cache), np_(inp.value_cache),
                                   inp.block_tables.numpy(), inp.seq_lens.numpy(), inp.scale,
                                   inp.cfg.num_kv_heads, inp.cfg.block_size, inp.cfg.dtype)
    assert max_abs_err(out, want) <= 1e-5
    assert pa.pa_get_device_error() == 0


def test_bounded_wait_rejects_bad_limits():
    for bad in (0, -5, 1 << 40):
        with pytest.raises(pa.PagedAttnError):
            pa.pa_selftest_bounded_wait(bad)
