"""Several new tokens per sequence (prefill chunks, speculative tokens):
slot mapping of all new tokens, their KV write, then causal paged attention
through the C ABI, element by element against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_batch(dtype, D, hq, hkv, B, ctx, n_new, seed):
    gen = torch.Generator().manual_seed(seed)
    dt = workloads.DTYPES[dtype]
    lens = [c + n for c, n in zip(ctx, n_new)]
    nblk = [-(-L // B) for L in lens]
    NB = sum(nblk) + 5
    perm = torch.randperm(NB, generator=gen)
    tables = torch.full((len(lens), max(nblk)), -1, dtype=torch.int32)
    off = 0
    for s, k in enumerate(nblk):
        tables[s, :k] = perm[off:off + k].to(torch.int32)
        off += k
    T = sum(n_new)
    kc = torch.empty(NB, hkv, B, D, dtype=dt)
    vc = torch.empty_like(kc)
    q = torch.empty(T, hq, D, dtype=dt)
    kn = torch.empty(T, hkv, D, dtype=dt)
    vn = torch.empty_like(kn)
    for t in (kc, vc, q, kn, vn):
        workloads.randn_into(t, gen)
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(n_new)]), dtype=torch.int32)
    pos = torch.tensor([p for c, n in zip(ctx, n_new) for p in range(c, c + n)],
                       dtype=torch.int64)
    return dict(kc=kc, vc=vc, q=q, kn=kn, vn=vn, qsl=qsl, pos=pos, tables=tables,
                lens=torch.tensor(lens, dtype=torch.int32), B=B, hkv=hkv, dtype=dtype,
                scale=D ** -0.5, max_q=max(n_new), max_len=max(lens))


def run_both(b, partition=0):
    kco, vco = np_(b["kc"]), np_(b["vc"])
    slots_o = oracle.slot_mapping(b["qsl"].numpy(), b["pos"].numpy(), b["tables"].numpy(), b["B"])
    oracle.reshape_and_cache(np_(b["kn"]), np_(b["vn"]), slots_o, kco, vco, b["B"])
    want = oracle.multi_query_attention(np_(b["q"]), kco, vco, b["tables"].numpy(),
                                        b["qsl"].numpy(), b["lens"].numpy(), b["scale"],
                                        b["hkv"], b["B"], b["dtype"])
    g = {k: v.to(DEV) for k, v in b.items() if isinstance(v, torch.Tensor)}
    slots = pa.pa_compute_slot_mapping(g["qsl"], g["pos"], g["tables"], b["B"])
    pa.pa_reshape_and_cache(g["kn"], g["vn"], slots, g["kc"], g["vc"])
    out = pa.pa_multi_query_attention(g["q"], g["qsl"], g["kc"], g["vc"], g["tables"], g["lens"],
                                      b["scale"], b["hkv"], max_query_len=b["max_q"],
                                      max_seq_len=b["max_len"], partition_size=partition)
    torch.cuda.synchronize()
    assert np.array_equal(slots.cpu().numpy(), slots_o)
    return out, want, g


CASES = []
for dtype in ("bf16", "f16"):
    for D in (64, 128):
        for G in (1, 2, 4, 8):
            CASES.append((dtype, D, G, 16))
for B in (8, 32, 64, 128, 256):
    CASES.append(("bf16", 128, 8, B))
    CASES.append(("f16", 128, 1, B))


@pytest.mark.parametrize("dtype,D,G,B", CASES)
def test_multi_query_matches_oracle(dtype, D, G, B):
    ctx = [0, 5, 100, 300, 0, 64]
    n_new = [1, 3, 17, 70, 130, 64]
    seed = 500 + 17 * D + 7 * G + B + (1000 if dtype == "f16" else 0)
    b = make_batch(dtype, D, 2 * G, 2, B, ctx, n_new, seed)
    out, want, _ = run_both(b)
    assert torch.isfinite(out.float()).all()
    err = max_abs_err(out, want)
    assert err <= TOL[dtype], err
    assert pa.pa_get_device_error() == 0


def test_one_new_token_matches_decode_kernel():
    b = make_batch("bf16", 128, 16, 2, 16, [10, 500, 2000], [1, 1, 1], 31)
    out, want, g = run_both(b)
    dec = pa.pa_decode_attention(g["q"], g["kc"], g["vc"], g["tables"], g["lens"], b["scale"], 2,
                                 max_seq_len=b["max_len"])
    assert (out.float() - dec.float()).abs().max().item() <= TOL["bf16"]
    assert max_abs_err(out, want) <= TOL["bf16"]


def test_garbage_pool_rows_do_not_leak():
    b = make_batch("bf16", 128, 16, 2, 16, [3, 40], [5, 9], 41)
    used = torch.zeros(b["kc"].shape[0], 16, dtype=torch.bool)
    for s, L in enumerate(b["lens"].tolist()):
        for j in range(L):
            used[int(b["tables"][s, j // 16]), j % 16] = True
    for cache in (b["kc"], b["vc"]):
        cache.permute(0, 2, 1, 3)[~used] = float("nan")
    out, want, _ = run_both(b)
    assert torch.isfinite(out.float()).all()
    assert max_abs_err(out, want) <= TOL["bf16"]


def test_more_new_tokens_than_length_is_rejected_on_device():
    b = make_batch("f16", 64, 4, 4, 16, [0, 8], [4, 4], 51)
    g = {k: v.to(DEV) for k, v in b.items() if isinstance(v, torch.Tensor)}
    g["lens"][0] = 2                          # 4 new tokens but length 2
    pa.pa_get_device_error()
    pa.pa_multi_query_attention(g["q"], g["qsl"], g["kc"], g["vc"], g["tables"], g["lens"],
                                b["scale"], 4, max_query_len=4, max_seq_len=12)
    assert pa.pa_get_device_error() == -5


def test_unsupported_dtype_and_block_are_refused():
    b = make_batch("f16", 64, 4, 4, 4, [0], [2], 61)
    g = {k: v.to(DEV) for k, v in b.items() if isinstance(v, torch.Tensor)}
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_multi_query_attention(g["q"], g["qsl"], g["kc"], g["vc"], g["tables"], g["lens"],
                                    b["scale"], 4, max_query_len=2, max_seq_len=2)
    assert e.value.status == -2               # block size 4 < 8


@pytest.mark.parametrize("partition", [64, 192, 1024])
@pytest.mark.parametrize("dtype,G,n_new", [("bf16", 8, [4, 1, 3, 2]), ("f16", 1, [7, 1, 30, 2]),
                                           ("bf16", 4, [40, 1, 100, 9])])
def test_split_partitions_with_combine(partition, dtype, G, n_new):
    """KV split into partitions, partials merged by log-sum-exp; rows whose
    visible keys fit one partition bypass the merge."""
    b = make_batch(dtype, 128, 2 * G, 2, 16, [900, 0, 2000, 63], n_new, 71)
    out, want, _ = run_both(b, partition)
    need = pa.pa_multi_query_workspace_bytes(sum(n_new), 4, 2 * G, 2, 128, 16, b["max_q"],
                                             b["max_len"], partition)
    assert need > 0
    assert max_abs_err(out, want) <= TOL[dtype]
    assert pa.pa_get_device_error() == 0


def test_short_query_runs_split_automatically():
    b = make_batch("bf16", 128, 16, 2, 16, [3000, 5000, 100], [4, 4, 4], 81)
    need = pa.pa_multi_query_workspace_bytes(12, 3, 16, 2, 128, 16, 4, b["max_len"], 0)
    assert need > 0                      # few CTAs without splits: the library splits
    out, want, _ = run_both(b)
    assert max_abs_err(out, want) <= TOL["bf16"]


SHORT = [(dt, D, G, B) for dt in ("bf16", "f16") for D in (64, 128) for G in (1, 2, 4, 8)
         for B in (16,)] + [("bf16", 128, 8, 8), ("bf16", 128, 4, 128), ("f16", 128, 1, 64)]


@pytest.mark.parametrize("rows", [16, 32, 96])
@pytest.mark.parametrize("dtype,D,G,B", SHORT)
def test_short_runs(dtype, D, G, B, rows):
    """Short runs, with and without KV partitions: at most 16 (token, head)
    rows per KV head go to the column kernel (KV tokens as M), longer ones to
    the tcgen05 kernel, whose row tile is then partly empty (warps without a
    row skip their work)."""
    n_max = max(1, rows // G)
    n_new = [1, n_max, max(1, n_max // 2), n_max]
    ctx = [0, 17, 700, 1500]
    b = make_batch(dtype, D, 2 * G, 2, B, ctx, n_new, 900 + 13 * G + D + B + rows)
    for partition in (0, 128):
        out, want, _ = run_both(b, partition)
        assert torch.isfinite(out.float()).all()
        err = max_abs_err(out, want)
        assert err <= TOL[dtype], (partition, err)
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("n,B", [(3, 16), (5, 8), (7, 64), (3, 128)])
def test_partial_warp_runs_with_garbage_pool(n, B):
    """Runs whose (token, head) rows leave a warp partly without tokens (3, 5
    or 7 tokens x 8 heads): those rows take no part in choosing the
    mask-free path and are not masked. Every pool row outside the sequences
    holds NaN, contexts are ragged (tiles with a tail and whole tiles), and
    all written outputs must match the oracle and be finite."""
    ctx = [0, 5, 130, 700, 1029]
    b = make_batch("bf16", 128, 16, 2, B, ctx, [n] * len(ctx), 1200 + 7 * n + B)
    used = torch.zeros(b["kc"].shape[0], B, dtype=torch.bool)
    for s, L in enumerate(b["lens"].tolist()):
        for j in range(L):
            used[int(b["tables"][s, j // B]), j % B] = True
    for cache in (b["kc"], b["vc"]):
        cache.permute(0, 2, 1, 3)[~used] = float("nan")
    for partition in (0, 256):
        out, want, _ = run_both(b, partition)
        assert torch.isfinite(out.float()).all(), partition
        assert max_abs_err(out, want) <= TOL["bf16"], partition
    assert pa.pa_get_device_error() == 0


def test_short_runs_with_garbage_rows():
    b = make_batch("bf16", 128, 16, 2, 16, [3, 40, 0], [2, 4, 1], 43)
    used = torch.zeros(b["kc"].shape[0], 16, dtype=torch.bool)
    for s, L in enumerate(b["lens"].tolist()):
        for j in range(L):
            used[int(b["tables"][s, j // 16]), j % 16] = True
    for cache in (b["kc"], b["vc"]):
        cache.permute(0, 2, 1, 3)[~used] = float("nan")
    out, want, _ = run_both(b)
    assert torch.isfinite(out.float()).all()
    assert max_abs_err(out, want) <= TOL["bf16"]


@pytest.mark.parametrize("n_new", [[2, 2, 2], [40, 40, 40]])
def test_bad_block_id_is_latched_and_other_sequences_are_exact(n_new):
    """A block id outside the pool in one sequence's table: the error is
    latched; sequences with valid tables still match the oracle (both the
    column kernel and the row kernel)."""
    b = make_batch("bf16", 128, 16, 2, 16, [100, 300, 50], n_new, 97)
    kco, vco = np_(b["kc"]), np_(b["vc"])
    slots_o = oracle.slot_mapping(b["qsl"].numpy(), b["pos"].numpy(), b["tables"].numpy(), 16)
    oracle.reshape_and_cache(np_(b["kn"]), np_(b["vn"]), slots_o, kco, vco, 16)
    want = oracle.multi_query_attention(np_(b["q"]), kco, vco, b["tables"].numpy(),
                                        b["qsl"].numpy(), b["lens"].numpy(), b["scale"], 2, 16,
                                        "bf16")
    g = {k: v.to(DEV) for k, v in b.items() if isinstance(v, torch.Tensor)}
    slots = pa.pa_compute_slot_mapping(g["qsl"], g["pos"], g["tables"], 16)
    pa.pa_reshape_and_cache(g["kn"], g["vn"], slots, g["kc"], g["vc"])
    pa.pa_get_device_error()
    g["tables"][1, 2] = b["kc"].shape[0] + 7           # sequence 1 now points outside
    out = pa.pa_multi_query_attention(g["q"], g["qsl"], g["kc"], g["vc"], g["tables"], g["lens"],
                                      b["scale"], 2, max_query_len=max(n_new),
                                      max_seq_len=b["max_len"])
    assert pa.pa_get_device_error() == -5
    q0, q1 = int(b["qsl"][1]), int(b["qsl"][2])
    keep = [t for t in range(out.shape[0]) if not (q0 <= t < q1)]
    assert max_abs_err(out[keep], want[keep]) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,G,D", [("bf16", 8, 128), ("f16", 1, 128), ("bf16", 4, 64)])
def test_long_prefill_with_growing_logits(dtype, G, D):
    """Keys scaled up along the sequence make each row's running maximum jump
    by far more than 2^8 across KV tiles, so the tensor-core kernel's output
    rescale runs many times; several 128-row tiles and KV tiles, ragged."""
    ctx, n_new = [700, 0, 37], [300, 257, 129]
    b = make_batch(dtype, D, 2 * G, 2, 16, ctx, n_new, 321 + G + D)
    f = lambda j: 1.0 + j / 40.0
    kc = b["kc"].float()
    for s, c in enumerate(ctx):
        for j in range(c):
            kc[int(b["tables"][s, j // 16]), :, j % 16, :] *= f(j)
    b["kc"] = kc.to(b["kc"].dtype)
    kn = b["kn"].float()
    for t, p in enumerate(b["pos"].tolist()):
        kn[t] *= f(p)
    b["kn"] = kn.to(b["kn"].dtype)
    out, want, _ = run_both(b)
    assert torch.isfinite(out.float()).all()
    assert max_abs_err(out, want) <= TOL[dtype]
    assert pa.pa_get_device_error() == 0


def test_long_prefill_many_tiles_against_oracle_sampled():
    """A 1024-token prefill chunk after 3000 cached tokens (GQA group 8):
    8 x 128-row tiles per KV head, 32 KV tiles; sampled rows vs the oracle."""
    b = make_batch("bf16", 128, 16, 2, 16, [3000], [1024], 404)
    kco, vco = np_(b["kc"]), np_(b["vc"])
    slots_o = oracle.slot_mapping(b["qsl"].numpy(), b["pos"].numpy(), b["tables"].numpy(), 16)
    oracle.reshape_and_cache(np_(b["kn"]), np_(b["vn"]), slots_o, kco, vco, 16)
    g = {k: v.to(DEV) for k, v in b.items() if isinstance(v, torch.Tensor)}
    slots = pa.pa_compute_slot_mapping(g["qsl"], g["pos"], g["tables"], 16)
    pa.pa_reshape_and_cache(g["kn"], g["vn"], slots, g["kc"], g["vc"])
    out = pa.pa_multi_query_attention(g["q"], g["qsl"], g["kc"], g["vc"], g["tables"], g["lens"],
                                      b["scale"], 2, max_query_len=1024, max_seq_len=4024)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    rows = [0, 1, 127, 128, 129, 500, 895, 1023]
    q = np_(b["q"])
    for i in rows:
        L_i = 3000 + i + 1
        for h in (0, 7, 8, 15):
            kvh = h // 8
            K = oracle.gather_kv(kco, b["tables"][0].numpy(), L_i, kvh, 16, "bf16")
            V = oracle.gather_kv(vco, b["tables"][0].numpy(), L_i, kvh, 16, "bf16")
            want = oracle.decode_attention_one(oracle.upcast(q[i, h], "bf16"), K, V, b["scale"])
            got = out[i, h].double().cpu().numpy()
            assert np.abs(got - want).max() <= TOL["bf16"], (i, h)
