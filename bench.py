"""Benchmark of the paged-KV decode step on GB300.

One step = the whole hot path over one batch: slot mapping of the new tokens,
the KV write (reshape_and_cache), and paged decode attention (with its split
combine when the partitioning uses more than one partition). Copy-on-write
block copies run only when a write hits a shared block, which the Llama-7B
batch never does; the shared-prefix workload exercises them (--config
shared_prefix).

Prints one JSON line (rank 0). `value` is KV-read GB/s over the whole step
(algorithmic bytes: sum_s L_s * 2 * Hkv * D * elt, valid tokens only) with
inputs resident in HBM; `e2e` is the same metric with the per-step inputs
copied from pinned host memory and the output copied back inside the timed
region; `roofline` is for the attention launch alone.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                       [--impl ours|reference]
For N > 1 launch under torch.distributed.run; each rank runs an independent
replica of the workload (the decode step shards by sequence with no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn: KV-read GB/s vs HBM peak; seq-tokens/s at Llama-7B shape"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ELT = {"f32": 4, "f16": 2, "bf16": 2}
CSRC = os.path.join(ROOT, "paged_kv_cache_123_gb300", "csrc")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", default="llama7b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels eagerly instead of replaying a CUDA graph")
    ap.add_argument("--partition", type=int, default=0,
                    help="tokens per context partition (0 = the library's choice)")
    ap.add_argument("--kv-dtype", default="model", choices=["model", "fp8"],
                    help="fp8: E4M3 pools (one new token per sequence)")
    ap.add_argument("--fp8-scales", default="pool", choices=["pool", "block"],
                    help="with --kv-dtype fp8: one scale per pool, or one power-of-two scale "
                         "per (block, KV head) fixed by the write of the block's first row")
    ap.add_argument("--new-tokens", type=int, default=1,
                    help="new tokens per sequence per step (>1: causal multi-query attention)")
    ap.add_argument("--layers", type=int, default=1,
                    help="decode layers per step, each with its own KV pools (one-token decode); "
                         "the whole multi-layer step is one CUDA graph")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window in tokens for one-new-token decode (0 = none); "
                         "blocks wholly before the window are released from the tables")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="use only the first N sequences (smaller profiling case)")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers
def kv_read_bytes(seq_lens, num_kv_heads, head_size, elt):
    """Algorithmic KV bytes one attention launch must read."""
    return int(sum(int(L) for L in seq_lens)) * 2 * num_kv_heads * head_size * elt


def block_scale_bytes(seq_lens, window, block_size, num_kv_heads):
    """Bytes of per-block fp8 scales one attention launch must read: a K and
    a V fp32 scale for every (block, KV head) that holds an attended token
    (tokens L - window .. L - 1 under a window, else all L)."""
    blocks = 0
    for L in seq_lens:
        L = int(L)
        if L <= 0:
            continue
        lo = L - window if 0 < window < L else 0
        blocks += (L - 1) // block_size - lo // block_size + 1
    return blocks * num_kv_heads * 2 * 4


def kernel_sources_digest():
    """Digest of every source the library is built from (kernels, shared
    device helpers, host dispatch and partitioning) and of the workload
    generator (the batches' lengths and tables): a profiled traffic row is
    used only while none of them has changed."""
    h = hashlib.sha256()
    paths = [os.path.join(CSRC, n) for n in sorted(os.listdir(CSRC))
             if n.endswith((".cu", ".cuh", ".h"))]
    paths.append(os.path.join(os.path.dirname(CSRC), "workloads.py"))
    for path in paths:
        if os.path.exists(path):
            with open(path, "rb") as f:
                h.update(os.path.basename(path).encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    try:
        rows = open(PROFILE_TRAFFIC).read().split("\n")
    except OSError:
        return None
    digest = kernel_sources_digest()
    for r in rows:
        parts = r.split()
        if len(parts) == 3 and parts[0] == config and parts[1] == digest:
            return int(parts[2])
    return None


def measured_peak(key="hbm_gbs", fallback=None):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return (FALLBACK_HBM_GBS if fallback is None else fallback), "fallback"


def attention_flops(ctx_lens, new_tokens, num_q_heads, head_size):
    """Algorithmic flops of causal multi-query attention: new token i of a
    sequence with c cached tokens sees c + i + 1 keys; 2 flops per
    multiply-add of q.k and of p.v over the head dim."""
    keys = sum((c + 1) * new_tokens + new_tokens * (new_tokens - 1) // 2 for c in ctx_lens)
    return 4 * head_size * num_q_heads * keys


class ClockSampler:
    """nvidia-smi samples tagged with host time, so the ones inside the timed
    window can be picked out."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id is not None:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed"
        if len(inside) < 2:
            inside = [s for t, s in self.samples if t <= t1]
            window = "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        mx = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------- oracle (CPU) timing
_ORC = {}


def _orc_init(spec):
    # runs in spawned worker processes: map the shared input files read-only
    import numpy as np
    for k, (path, shape, dt) in spec.items():
        _ORC[k] = np.memmap(path, dtype=np.dtype(dt), mode="r", shape=shape)


def _orc_run(job):
    import numpy as np

    import oracle
    kind, units, p = job
    A = _ORC
    if kind == "decode":
        oracle.decode_attention(A["q"], A["kc"], A["vc"], A["tables"], A["lens"], p["scale"],
                                p["hkv"], p["bs"], p["dtype"], seqs=units, window=p["window"])
    elif kind == "fp8":
        oracle.decode_attention_fp8(A["q"], A["kc"], A["vc"], A["tables"], A["lens"],
                                    p["scale"], p["hkv"], p["bs"], p["dtype"], p["ks"], p["vs"],
                                    seqs=units, window=p["window"])
    elif kind == "fp8b":
        oracle.decode_attention_fp8_block_scaled(A["q"], A["kc"], A["vc"], A["ks"], A["vs"],
                                                 A["tables"], A["lens"], p["scale"], p["hkv"],
                                                 p["bs"], p["dtype"], seqs=units,
                                                 window=p["window"])
    else:   # "mq": units are (sequence, KV head) pairs of N new tokens each
        N, g = p["N"], p["g"]
        for s, kvh in units:
            oracle.multi_query_attention(
                A["q"][s * N:(s + 1) * N, kvh * g:(kvh + 1) * g], A["kc"][:, kvh:kvh + 1],
                A["vc"][:, kvh:kvh + 1], A["tables"][s:s + 1], np.array([0, N]),
                A["lens"][s:s + 1], p["scale"], 1, p["bs"], p["dtype"])
    return len(units)


class OracleTimer:
    """The CPU oracle, as it stands, over a spawn pool of single-threaded
    workers that map the inputs from files in a temporary directory. `arrays`
    are numpy copies of the step's inputs taken before any kernel ran.
    kind "decode" (16-bit pools) or "fp8" (E4M3 pools, scales ks / vs) times
    decode attention, with a sliding window when window > 0, on whole
    sequences; kind "mq" times the causal attention of N new tokens per
    sequence on (sequence, KV head) units."""

    def __init__(self, arrays, cfg, scale, workers, kind="decode", window=0, ks=1.0, vs=1.0,
                 N=1):
        import multiprocessing as mp
        import tempfile

        import numpy as np
        self.cfg, self.scale, self.workers = cfg, scale, workers
        self.kind, self.window, self.N = kind, window, N
        self.params = {"scale": scale, "hkv": cfg.num_kv_heads, "bs": cfg.block_size,
                       "dtype": cfg.dtype, "window": window, "ks": ks, "vs": vs, "N": N,
                       "g": cfg.num_q_heads // cfg.num_kv_heads}
        lens = [int(x) for x in arrays["lens"].tolist()]
        self.lens = lens
        att = [min(L, window) if window > 0 else L for L in lens]
        if kind == "mq":
            self.units = [(s, h) for s in range(len(lens)) for h in range(cfg.num_kv_heads)]
            self.unit_tok = [lens[s] for s, _ in self.units]
            self.bytes_per_tok = 2 * cfg.head_size * ELT[cfg.dtype]
        else:
            self.units = list(range(len(lens)))
            self.unit_tok = att
            self.bytes_per_tok = 2 * cfg.num_kv_heads * cfg.head_size * (
                1 if kind in ("fp8", "fp8b") else ELT[cfg.dtype])
        self.dir = tempfile.mkdtemp(prefix="pa_oracle_")
        spec = {}
        for k, a in arrays.items():
            path = os.path.join(self.dir, k + ".bin")
            mm = np.memmap(path, dtype=a.dtype, mode="w+", shape=a.shape)
            mm[...] = a
            mm.flush()
            del mm
            spec[k] = (path, a.shape, a.dtype.str)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.pool = mp.get_context("spawn").Pool(workers, initializer=_orc_init, initargs=(spec,))
        self.sample = None

    def run(self, idx):
        chunks = [[self.units[i] for i in idx[k::self.workers]] for k in range(self.workers)]
        jobs = [(self.kind, c, self.params) for c in chunks if c]
        t0 = time.perf_counter()
        self.pool.map(_orc_run, jobs)
        return time.perf_counter() - t0

    def size_sample(self, budget_s):
        """A sample worth about budget_s of oracle time: the first n units,
        or the whole batch repeated when one pass is shorter."""
        tok, w = self.unit_tok, self.workers
        probe = list(range(min(len(tok), w)))
        self.run(probe)                      # warm the workers
        dt = self.run(probe)
        per_tok = dt * w / max(1, sum(tok[i] for i in probe))
        want_tok = budget_s * w / max(per_tok, 1e-12)
        n, t = 0, 0
        while n < len(tok) and (t < want_tok or n < w):
            t += tok[n]
            n += 1
        self.sample = list(range(n))
        self.repeats = 1
        if n == len(tok) and t < want_tok:
            self.repeats = max(1, int(round(want_tok / max(1, t))))
        return self.sample

    def measure(self):
        """(GB/s, seq-tokens/s, description, seconds) on the sized sample."""
        cfg = self.cfg
        dt = 0.0
        for _ in range(self.repeats):
            dt += self.run(self.sample)
        st = [self.unit_tok[i] for i in self.sample]
        byts = self.repeats * sum(st) * self.bytes_per_tok
        what = {"decode": "decode attention", "fp8": "decode attention over fp8 pools",
                "fp8b": "decode attention over fp8 pools with per-block scales",
                "mq": f"causal attention of {self.N} new tokens per sequence"}[self.kind]
        if self.window > 0:
            what += f", window {self.window}"
        if self.kind == "mq":
            seqs = sorted({self.units[i][0] for i in self.sample})
            desc = (f"{what}: first {len(self.sample)} of {len(self.units)} (sequence, KV head) "
                    f"units of the {cfg.name} batch ({len(seqs)} sequences)")
            toks = self.repeats * sum(st) / cfg.num_kv_heads
        else:
            desc = (f"{what}: first {len(st)} of {len(self.lens)} sequences of the {cfg.name} "
                    f"batch, all {cfg.num_q_heads} query heads ({sum(st)} context tokens)")
            toks = self.repeats * sum(st)
        if self.repeats > 1:
            desc += f", {self.repeats} passes"
        return byts / dt / 1e9, toks / dt, desc, dt

    def close(self):
        self.pool.close()
        self.pool.join()
        import shutil
        shutil.rmtree(self.dir, ignore_errors=True)


def np_(t):
    """Storage-typed numpy copy of a tensor (bf16 as uint16 bit patterns)."""
    import numpy as np
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def oracle_arrays(inp):
    return {"q": np_(inp.q), "kc": np_(inp.key_cache), "vc": np_(inp.value_cache),
            "tables": np_(inp.block_tables), "lens": np_(inp.seq_lens)}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------ distributed
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return dist.get_rank(), world
    return 0, 1


def max_over_ranks(x, world):
    """Max of a host float over ranks (a timing reduction; the decode data
    path itself has no exchange)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- arms
def reference_arm(args):
    """The oracle as the reference arm: CPU fp64, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_kv_cache_123_gb300 import workloads
    inp = workloads.make_decode_inputs(args.config, device="cpu")
    workers = host_cores()
    timer = OracleTimer(oracle_arrays(inp), inp.cfg, inp.scale, workers)
    try:
        # about two minutes of oracle work over the whole run, whatever K and W
        timer.size_sample(max(0.05, 120.0 / max(1, args.steps + args.warmup)))
        gbs_list, tps_list, dts = [], [], []
        desc = ""
        for i in range(args.warmup + args.steps):
            gbs, tps, desc, dt = timer.measure()
            if i >= args.warmup:
                gbs_list.append(gbs)
                tps_list.append(tps)
                dts.append(dt)
    finally:
        timer.close()
    value = statistics.median(gbs_list)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(dts), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "seq_tokens_per_s": round(statistics.median(tps_list), 1),
        "config": {"workload": args.config, "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": workers,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours_arm(args):
    import numpy as np
    import torch

    import paged_kv_cache_123_gb300 as pa
    from paged_kv_cache_123_gb300 import workloads

    rank, world = dist_setup(args)
    if world == 1:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    cfg = workloads.CONFIGS[args.config]
    if args.num_seqs:
        import dataclasses
        cfg = dataclasses.replace(cfg, num_seqs=args.num_seqs, name=f"{cfg.name}_s{args.num_seqs}",
                                  ctx_fixed=None if cfg.ctx_fixed is None
                                  else cfg.ctx_fixed[:args.num_seqs])
    inp = workloads.make_decode_inputs(cfg, device=str(dev), seed=cfg.seed + rank)
    B, Hkv, D = cfg.block_size, cfg.num_kv_heads, cfg.head_size
    S = cfg.num_seqs
    N = max(1, args.new_tokens)
    fp8 = args.kv_dtype == "fp8"
    if fp8 and N > 1:
        raise SystemExit("--kv-dtype fp8 runs one new token per sequence")
    W = max(0, args.window)
    if W and N > 1:
        raise SystemExit("--window runs one new token per sequence")
    LAYERS = max(1, args.layers)
    if LAYERS > 1 and N > 1:
        raise SystemExit("--layers runs one new token per sequence")
    kc, vc = inp.key_cache, inp.value_cache
    kscale = vscale = 1.0 / 48
    bscaled = fp8 and args.fp8_scales == "block"
    ksb = vsb = None
    if bscaled:
        # E4M3 pools holding the same N(0,1) draws, each (block, KV head) at
        # the power-of-two scale its write would fix had one call filled it:
        # 2^(ceil(log2(amax)) - 7)
        def block_scaled(x):
            amax = x.float().abs().amax(dim=(2, 3)).clamp_(min=2.0 ** -119)
            s_ = torch.exp2(torch.ceil(torch.log2(amax)) - 7)
            c_ = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
            for b0 in range(0, x.shape[0], 4096):
                c_[b0:b0 + 4096] = (x[b0:b0 + 4096].float() / s_[b0:b0 + 4096, :, None, None]
                                    ).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            return c_, s_.contiguous()
        kc, ksb = block_scaled(kc)
        vc, vsb = block_scaled(vc)
        del inp.key_cache, inp.value_cache
        torch.cuda.empty_cache()
    elif fp8:   # E4M3 pools holding the same N(0,1) draws at scale 1/48
        kc = (kc.float() / kscale).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        vc = (vc.float() / vscale).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        del inp.key_cache, inp.value_cache
        torch.cuda.empty_cache()
    # one pair of pools per layer (layer 0: the generated pools)
    kcs, vcs = [kc], [vc]
    kss, vss = [ksb], [vsb]
    for _ in range(LAYERS - 1):
        kcs.append(kc.clone())
        vcs.append(vc.clone())
        kss.append(None if ksb is None else ksb.clone())
        vss.append(None if vsb is None else vsb.clone())
    elt = 1 if fp8 else inp.q.element_size()
    lens = inp.seq_lens.cpu()
    if W:   # attended tokens per sequence; skipped blocks' table entries -> -1
        attended = [min(int(L), W) for L in lens.tolist()]
        tab = inp.block_tables.cpu()
        for s_, L in enumerate(lens.tolist()):
            tab[s_, :max(0, L - W) // B] = -1
        inp.block_tables.copy_(tab)
    else:
        attended = lens.tolist()
    kv_bytes = kv_read_bytes(attended, Hkv, D, elt)
    if bscaled:   # plus the K and V scale of every attended (block, KV head)
        kv_bytes += block_scale_bytes(lens.tolist(), W, B, Hkv)
    tokens = int(sum(attended))
    max_len = inp.max_seq_len
    P = args.partition
    g = dict(q=inp.q, k_new=inp.k_new, v_new=inp.v_new, tables=inp.block_tables,
             lens=inp.seq_lens, pos=inp.positions, qsl=inp.query_start_loc)
    if N > 1:   # the last N tokens of every sequence are new this step
        gen = torch.Generator(device=dev).manual_seed(cfg.seed + 77)
        for k, h in (("q", cfg.num_q_heads), ("k_new", Hkv), ("v_new", Hkv)):
            g[k] = torch.empty((S * N, h, D), dtype=inp.q.dtype, device=dev)
            workloads.randn_into(g[k], gen)
        g["qsl"] = torch.arange(S + 1, dtype=torch.int32, device=dev) * N
        g["pos"] = (inp.seq_lens.to(torch.int64)[:, None] - N +
                    torch.arange(N, device=dev)[None, :]).reshape(-1).contiguous()
        ws_bytes = pa.pa_multi_query_workspace_bytes(S * N, S, cfg.num_q_heads, Hkv, D, B, N,
                                                     max_len, P)
        splits = 1 if ws_bytes == 0 else 2
        ptoks = None
        even_ctas = 0
    else:
        if fp8:
            splits, ptoks = pa.pa_decode_fp8_partitioning(S, cfg.num_q_heads, Hkv, D, B,
                                                          inp.q.dtype, max_len, W, P)
        else:
            splits, ptoks = pa.pa_decode_window_partitioning(S, cfg.num_q_heads, Hkv, B,
                                                             max_len, W, P)
        # the even schedule (windowed tensor-core calls) instead of the
        # partitions: its CTA count, and a merge launch after the attention
        even_ctas = pa.pa_decode_even_ctas(S, cfg.num_q_heads, Hkv, D, B, inp.q.dtype,
                                           "fp8_block_scales" if bscaled else
                                           "fp8" if fp8 else "16bit", max_len, W, P)
        if even_ctas:
            splits, ptoks = None, None
        if fp8:
            ws_bytes = pa.pa_decode_fp8_workspace_bytes(S, cfg.num_q_heads, Hkv, D, B,
                                                        inp.q.dtype, max_len, W, P)
        else:
            ws_bytes = pa.pa_decode_window_workspace_bytes(S, cfg.num_q_heads, Hkv, D, B,
                                                           max_len, W, P)
    # host copies of the step's inputs for the CPU baseline, taken before any
    # kernel touches the pools (fp8 pools as codes, windowed tables with their
    # released entries, the N new tokens' queries)
    orc_arrays = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        orc_arrays = {"q": np_(g["q"]), "kc": np_(kc), "vc": np_(vc),
                      "tables": np_(g["tables"]), "lens": np_(g["lens"])}
        if bscaled:
            orc_arrays["ks"], orc_arrays["vs"] = np_(ksb), np_(vsb)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    out = torch.empty_like(g["q"])
    slots = torch.empty(S * N, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()

    def attention(t, kc=kc, vc=vc, ks=ksb, vs=vsb):
        o = t.get("out", out)
        if bscaled:
            pa.pa_decode_attention_fp8_scaled(t["q"], kc, vc, ks, vs, t["tables"], t["lens"],
                                              inp.scale, Hkv, o, max_seq_len=max_len, window=W,
                                              partition_size=P, workspace=ws)
        elif N > 1:
            pa.pa_multi_query_attention(t["q"], t["qsl"], kc, vc, t["tables"], t["lens"],
                                        inp.scale, Hkv, o, max_query_len=N, max_seq_len=max_len,
                                        partition_size=P, workspace=ws)
        elif fp8 and W:
            pa.pa_decode_attention_fp8_window(t["q"], kc, vc, t["tables"], t["lens"], inp.scale,
                                              Hkv, kscale, vscale, W, o, max_seq_len=max_len,
                                              partition_size=P, workspace=ws)
        elif W:
            pa.pa_decode_attention_window(t["q"], kc, vc, t["tables"], t["lens"], inp.scale, Hkv,
                                          W, o, max_seq_len=max_len, partition_size=P,
                                          workspace=ws)
        elif fp8:
            pa.pa_decode_attention_fp8(t["q"], kc, vc, t["tables"], t["lens"], inp.scale, Hkv,
                                       kscale, vscale, o, max_seq_len=max_len,
                                       partition_size=P, workspace=ws)
        else:
            pa.pa_decode_attention(t["q"], kc, vc, t["tables"], t["lens"], inp.scale, Hkv, o,
                                   max_seq_len=max_len, partition_size=P, workspace=ws)

    l2_small = kv_bytes <= 2 * 129e6
    l2_flush = torch.ones(256 << 20, dtype=torch.uint8, device=dev) if l2_small else None

    def step(t, ev=None):
        pa.pa_compute_slot_mapping(t["qsl"], t["pos"], t["tables"], B, slot_mapping=slots)
        for layer in range(LAYERS):
            kcl, vcl = kcs[layer], vcs[layer]
            if bscaled:
                pa.pa_reshape_and_cache_fp8_scaled(t["k_new"], t["v_new"], slots, kcl, vcl,
                                                   kss[layer], vss[layer])
            elif fp8:
                pa.pa_reshape_and_cache_fp8(t["k_new"], t["v_new"], slots, kcl, vcl, kscale,
                                            vscale)
            else:
                pa.pa_reshape_and_cache(t["k_new"], t["v_new"], slots, kcl, vcl)
            if ev is not None and layer == 0:
                # a workload that fits in twice L2 first reads a 256 MiB
                # buffer (L2 then holds clean lines of it, nothing of the
                # pools); then a ~20 us spin keeps the GPU busy while the host
                # launches the attention call, so no host time lands between
                # the events
                if l2_small:
                    l2_flush.sum(dtype=torch.int32)
                torch.cuda._sleep(40000)
                ev[0].record(stream)
            attention(t, kcl, vcl, kss[layer], vss[layer])
            if ev is not None and layer == 0:
                ev[1].record(stream)

    launches_per_step = 1 + LAYERS * (2 + (1 if bscaled else 0) +
                                      (1 if even_ctas or splits > 1 else 0))
    launch_label = (cfg.name + ("_fp8b" if bscaled else "_fp8" if fp8 else "") +
                    (f"_q{N}" if N > 1 else "") + (f"_w{W}" if W else ""))   # one attention launch
    label = launch_label + (f"_L{LAYERS}" if LAYERS > 1 else "")
    kernel_name = ("pa_decode_attention_fp8_scaled" if bscaled else
                   "pa_multi_query_attention" if N > 1 else
                   "pa_decode_attention_fp8" if fp8 else "pa_decode_attention") + (
                       "_window" if W and not bscaled else "")
    for _ in range(max(3, args.warmup)):
        step(g)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0

    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    # the step as one CUDA graph (the decode step is graph-captured in the
    # serving engine the pages describe); --no-graph launches it eagerly
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(g)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(g)
        graph.replay()
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_host0 = time.monotonic()
    start.record(stream)
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(g)
    stop.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.monotonic()
    barrier(world)
    ms_local = start.elapsed_time(stop)
    ms_total = max_over_ranks(ms_local, world)
    assert pa.pa_get_device_error() == 0

    # per-launch attention time: the same K steps launched eagerly, with
    # events on the launching stream around every attention call
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_host2 = time.monotonic()
    for i in range(args.steps):
        step(g, evs[i])
    torch.cuda.synchronize()
    t_host3 = time.monotonic()
    if sampler is not None:
        time.sleep(0.25)
        sampler.stop()
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    eager_ms = (t_host3 - t_host2) * 1e3
    assert pa.pa_get_device_error() == 0

    # e2e: per-step inputs from pinned host memory, output back to host.
    # Two device copies of the inputs and of the output, each with its own
    # captured step: step i+1's host-to-device copy (copy stream) runs under
    # step i's kernels, and step i's device-to-host read (a third stream)
    # under step i+1's. Every step still pays its own copies; only their
    # overlap with compute differs from a serial loop.
    e2e = None
    if not args.no_e2e:
        # every per-step input lives in one pinned staging buffer and one
        # device buffer, so a step costs one host-to-device copy
        names = list(g)
        offs, total = {}, 0
        for k in names:
            offs[k] = total
            total += (g[k].numel() * g[k].element_size() + 255) // 256 * 256
        host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()

        def view(buf, k):
            n = g[k].numel() * g[k].element_size()
            return buf[offs[k]:offs[k] + n].view(g[k].dtype).view(g[k].shape)
        for k in names:
            view(host_buf, k).copy_(g[k].cpu())
        dev_bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
        dbufs = []
        for db in dev_bufs:
            d = {k: view(db, k) for k in names}
            d["out"] = torch.empty_like(out)
            dbufs.append(d)
            db.copy_(host_buf)
        out_hosts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = total
        d2h = out_hosts[0].numel() * out_hosts[0].element_size()
        graphs_e2e = [None, None]
        if graph is not None:
            for j in range(2):
                step(dbufs[j])
                torch.cuda.synchronize()
                graphs_e2e[j] = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graphs_e2e[j]):
                    step(dbufs[j])
        torch.cuda.synchronize()
        copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}

        def h2d_copy(i):
            j = i % 2
            with torch.cuda.stream(copy_in):
                if i >= 2:   # step i-2's kernels have finished reading buffer j
                    copy_in.wait_event(ev["done"][j])
                dev_bufs[j].copy_(host_buf, non_blocking=True)
                ev["in"][j].record(copy_in)

        def e2e_run(n):
            h2d_copy(0)
            for i in range(n):
                j = i % 2
                stream.wait_event(ev["in"][j])
                if i >= 2:   # step i-2's output has reached the host
                    stream.wait_event(ev["out"][j])
                if graphs_e2e[j] is not None:
                    graphs_e2e[j].replay()
                else:
                    step(dbufs[j])
                ev["done"][j].record(stream)
                if i + 1 < n:
                    h2d_copy(i + 1)
                with torch.cuda.stream(copy_out):
                    copy_out.wait_event(ev["done"][j])
                    out_hosts[j].copy_(dbufs[j]["out"], non_blocking=True)
                    ev["out"][j].record(copy_out)

        e2e_run(3)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        barrier(world)
        t0 = time.perf_counter()
        e2e_run(args.steps)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(time.perf_counter() - t0, world)
        assert pa.pa_get_device_error() == 0
        e2e = {"value": round(world * LAYERS * kv_bytes * args.steps / e2e_s / 1e9, 2),
               "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "seq_tokens_per_s": round(world * LAYERS * tokens * args.steps / e2e_s, 1),
               "pipeline": "double-buffered inputs and output, copies on two side streams"}

    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    achieved = kv_bytes / (attn_ms * 1e-3) / 1e9
    # runs of more than 64 (token, head) rows per KV head go to the tcgen05
    # kernel: a dense contraction, judged against the tensor-core peak
    tensor_bound = N * (cfg.num_q_heads // Hkv) > 64
    if tensor_bound:
        ctx_lens = [int(L) - N for L in lens.tolist()]
        flops = attention_flops(ctx_lens, N, cfg.num_q_heads, D)
        t_peak, t_kind = measured_peak("bf16_tflops", FALLBACK_BF16_TFLOPS)
        roof = {"bound": "tensor", "kernel": kernel_name,
                "achieved": round(flops / (attn_ms * 1e-3) / 1e12, 1), "peak": t_peak,
                "peak_kind": f"bf16_tflops (burst) of {t_kind}", "unit": "TFLOP/s",
                "frac": round(flops / (attn_ms * 1e-3) / 1e12 / t_peak, 4),
                "traffic": profiled_traffic(launch_label),
                "avg_launch_us": round(attn_ms * 1e3, 2),
                "algorithmic_flops_per_launch": flops,
                "algorithmic_kv_bytes_per_launch": kv_bytes}
    step_s = ms_total * 1e-3 / args.steps
    value = world * LAYERS * kv_bytes / step_s / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * step_s, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "kv_dtype": ("e4m3, per-block scales" if bscaled else "e4m3")
        if fp8 else cfg.dtype, "accum_dtype": "f32",
        "data": "synthetic",
        "seq_tokens_per_s": round(world * LAYERS * tokens / step_s, 1),
        "config": {
            "workload": label,
            "new_tokens_per_seq": N,
            "layers": LAYERS,
            "shape": f"{S} seqs, ctx U[{cfg.ctx_lo},{cfg.ctx_hi}]+1 new token, "
                     f"{cfg.num_q_heads}q/{Hkv}kv heads, D={D}, B={B}, {cfg.dtype}"
            if cfg.ctx_fixed is None else f"{S} seqs x {cfg.ctx_fixed[0]}+1, "
                                          f"{cfg.num_q_heads}q/{Hkv}kv heads, D={D}, B={B}",
            "context_tokens": tokens, "kv_read_bytes_per_step": LAYERS * kv_bytes,
            **({"kv_bytes_note": "codes plus 8 B of scales per attended (block, KV head)"}
               if bscaled else {}),
            "pool_blocks": inp.num_blocks,
            **({"even_schedule_ctas": even_ctas} if even_ctas else
               {"partitions": splits, "partition_tokens": ptoks}),
            "l2": ("graph-replayed steps: inputs larger than L2 (KV read per step %.2f GB, "
                   "pool %.2f GB; 129 MB L2), no flush" % (kv_bytes / 1e9,
                                                           2 * kc.numel() * elt / 1e9)
                   if kv_bytes > 2 * 129e6 else
                   "graph-replayed steps: KV read per step %.3f GB fits in twice L2: L2-warm"
                   % (kv_bytes / 1e9)) +
                  ("; roofline launches each follow a 256 MiB read that evicts the pools "
                   "from L2" if kv_bytes <= 2 * 129e6 else
                   "; roofline launches: the same, eager, after a short spin kernel"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "roofline": roof if tensor_bound else {"bound": "hbm", "kernel": kernel_name,
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"hbm_gbs of {peak_kind}", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(launch_label),
                     "avg_launch_us": round(attn_ms * 1e3, 2),
                     "algorithmic_bytes_per_launch": kv_bytes},
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
        "clocks": sampler.summary(t_host0, t_host3) if sampler else None,
        "launch": "cuda graph per step" if graph is not None else "eager",
        "ms_per_step_eager_host": round(eager_ms / args.steps, 4),
        "device": props.name,
    }
    if orc_arrays is not None:
        workers = host_cores()
        timer = OracleTimer(orc_arrays, cfg, inp.scale, workers,
                            kind="mq" if N > 1 else ("fp8b" if bscaled else "fp8" if fp8
                                                      else "decode"), window=W,
                            ks=kscale, vs=vscale, N=N)
        try:
            timer.size_sample(args.cpu_baseline_seconds)
            gbs, tps, desc, dt = timer.measure()
        finally:
            timer.close()
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": workers,
                                "kind": "oracle", "sample": desc,
                                "seq_tokens_per_s": round(tps, 1), "seconds": round(dt, 2)}
    print(json.dumps(line), flush=True)


def shared_prefix_arm(args):
    """8 samples of one 1027-token prompt (64 full blocks of 16 + a 3-token
    tail), 32/32 heads, D=128, bf16, then 256 decode steps that append one
    token per sample. The timed region holds exactly those 256 steps, step 0
    included: there the first 7 samples to write find the shared tail block
    referenced 8 times and copy it (block-level copy-on-write, one
    pa_copy_blocks launch of 7 pairs) and the 8th writes in place. Every
    step the host BlockPool computes the positions, the copy pairs and the
    table rows, which go up in one copy from a pinned staging buffer (two
    buffers, reused behind events, so the host prepares step i+1 while the
    GPU runs step i); then slot mapping, KV write and decode attention run.
    Warm-up runs on 8 throw-away forks of the same prompt, freed before the
    timed steps. A second pass from a fresh fork of the prompt measures the
    same 256 steps end to end, with q and the new K/V copied up from pinned
    host memory and the output copied back every step.

    Reports logical KV-read GB/s (every sample's context, prefix counted once
    per sample) and unique-block GB/s (each physical block in use counted
    once per step) over the device time of the 256 steps."""
    import numpy as np
    import torch

    import paged_kv_cache_123_gb300 as pa
    from paged_kv_cache_123_gb300 import BlockPool, workloads

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    S, Hkv, D, B, P0 = 8, 32, 128, 16, 1027
    steps = args.steps if args.steps != 2000 else 256   # the workload's 256 decode steps
    warm = max(3, args.warmup)
    MB = (P0 + max(steps, warm) + B - 1) // B
    NB = 64 + 2 * S * (MB - 64 + 1) + 8                 # real samples and warm-up forks
    gen = torch.Generator(device=dev).manual_seed(1003)
    order = torch.randperm(NB, generator=gen, device=dev).tolist()
    kc = torch.empty(NB, Hkv, B, D, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    workloads.randn_into(kc, gen)
    workloads.randn_into(vc, gen)
    kp = torch.empty(P0, Hkv, D, dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    workloads.randn_into(kp, gen)
    workloads.randn_into(vp, gen)
    q = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device=dev)
    kn, vn = torch.empty_like(q), torch.empty_like(q)
    for t in (q, kn, vn):
        workloads.randn_into(t, gen)
    qsl = torch.arange(S + 1, dtype=torch.int32, device=dev)
    block_bytes = Hkv * B * D * 2
    stream = torch.cuda.current_stream()
    ws_bytes = pa.pa_decode_workspace_bytes(S, Hkv, Hkv, D, B, MB * B, 0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def fresh_prompt():
        """A pool holding the prompt as sequence 0 (its K/V written)."""
        pool = BlockPool(NB, B, order)
        pool.add_sequence(0, P0)
        row = torch.from_numpy(pool.table_rows([0], MB)).to(dev)
        sl = pa.pa_compute_slot_mapping(torch.tensor([0, P0], dtype=torch.int32, device=dev),
                                        torch.arange(P0, dtype=torch.int64, device=dev), row, B)
        pa.pa_reshape_and_cache(kp, vp, sl, kc, vc)
        return pool

    # per-step host staging: [tables S*MB | lens S] int32, [positions S |
    # pairs 2*S] int64; two of each, pinned, and the device buffers they feed
    class Stage:
        def __init__(self):
            self.h32 = torch.empty(S * MB + S, dtype=torch.int32).pin_memory()
            self.h64 = torch.empty(3 * S, dtype=torch.int64).pin_memory()
            self.d32 = torch.empty(S * MB + S, dtype=torch.int32, device=dev)
            self.d64 = torch.empty(3 * S, dtype=torch.int64, device=dev)
            self.hin = [torch.empty_like(x, device="cpu").pin_memory() for x in (q, kn, vn)]
            self.din = [torch.empty_like(x) for x in (q, kn, vn)]
            self.hout = torch.empty(q.shape, dtype=q.dtype).pin_memory()
            self.dout = torch.empty_like(q)
            self.up = torch.cuda.Event()      # the uploads from h32/h64/hin have run
            self.down = torch.cuda.Event()    # hout holds this buffer's last output
            self.used = False
    stages = [Stage(), Stage()]
    for st in stages:
        for h, x in zip(st.hin, (q, kn, vn)):
            h.copy_(x.cpu())

    slots_buf = [torch.empty(S, dtype=torch.int64, device=dev) for _ in range(2)]

    def kernels(j, e2e):
        """Slot mapping, KV write and attention of one step, reading staging
        buffer j's device copies (tables, lengths, positions)."""
        st = stages[j]
        qi, ki, vi = st.din if e2e else (q, kn, vn)
        tables, lens = st.d32[:S * MB].view(S, MB), st.d32[S * MB:]
        sl = pa.pa_compute_slot_mapping(qsl, st.d64[:S], tables, B, slot_mapping=slots_buf[j])
        pa.pa_reshape_and_cache(ki, vi, sl, kc, vc)
        pa.pa_decode_attention(qi, kc, vc, tables, lens, D ** -0.5, Hkv, st.dout,
                               max_seq_len=MB * B, workspace=ws)

    def capture(e2e):
        """One CUDA graph per staging buffer (the step's kernels read fixed
        device buffers; the copy-on-write launch, when a step has pairs, runs
        eagerly before the graph)."""
        out_graphs = []
        for j in range(2):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                kernels(j, e2e)
            out_graphs.append(g_)
        return out_graphs

    def run(pool, seqs, n, graphs, e2e=False, ev_copy=None):
        """n decode steps of `seqs`; returns (logical, unique, copy pairs)."""
        logical = unique = copies = 0
        for i in range(n):
            j = i % 2
            st = stages[j]
            positions, pairs = pool.prepare_decode_step(seqs)
            tabs = pool.table_rows(seqs, MB)
            if st.used:                         # this buffer's previous uploads have run
                st.up.synchronize()
            st.h32[:S * MB] = torch.from_numpy(tabs.reshape(-1))
            st.h32[S * MB:] = torch.from_numpy((positions + 1).astype(np.int32))
            st.h64[:S] = torch.from_numpy(positions)
            if pairs:
                st.h64[S:S + 2 * len(pairs)] = torch.from_numpy(
                    np.asarray(pairs, dtype=np.int64).reshape(-1))
            st.d32.copy_(st.h32, non_blocking=True)
            st.d64.copy_(st.h64, non_blocking=True)
            if e2e:
                for h, d in zip(st.hin, st.din):
                    d.copy_(h, non_blocking=True)
            st.up.record(stream)
            st.used = True
            if pairs:
                copies += len(pairs)
                if ev_copy is not None:
                    ev_copy[0].record(stream)
                pa.pa_copy_blocks([kc], [vc], st.d64[S:S + 2 * len(pairs)].view(-1, 2),
                                  st.h64[S:S + 2 * len(pairs)].view(-1, 2).clone())
                if ev_copy is not None:
                    ev_copy[1].record(stream)
            if graphs is None:
                kernels(j, e2e)
            else:
                graphs[j].replay()
            if e2e:
                if i >= 2:                      # step i-2's output has reached the host
                    st.down.synchronize()
                st.hout.copy_(st.dout, non_blocking=True)
                st.down.record(stream)
            logical += int((positions + 1).sum()) * 2 * Hkv * D * 2
            unique += (NB - pool.num_free()) * 2 * block_bytes
        return logical, unique, copies

    # warm-up on throw-away forks of the prompt (the timed samples are forked
    # after they are freed, so the timed step 0 still finds the tail shared 8x)
    pool = fresh_prompt()
    junk = list(range(100, 100 + S))
    for s_ in junk:
        pool.fork(0, s_)
    run(pool, junk, warm, None)
    torch.cuda.synchronize()
    graphs = None if args.no_graph else capture(False)
    if graphs is not None:
        run(pool, junk, 4, graphs)
    torch.cuda.synchronize()
    for s_ in junk:
        pool.release(s_)
    for s_ in range(1, S):
        pool.fork(0, s_)
    seqs = list(range(S))
    assert pa.pa_get_device_error() == 0

    sampler = ClockSampler("GPU-" + str(props.uuid)) if hasattr(props, "uuid") else None
    if sampler is not None:
        time.sleep(0.3)
    ev_copy = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_host0 = time.monotonic()
    start.record(stream)
    logical, unique, copies = run(pool, seqs, steps, graphs, ev_copy=ev_copy)
    stop.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.monotonic()
    dt = start.elapsed_time(stop) * 1e-3
    assert pa.pa_get_device_error() == 0
    in_use = NB - pool.num_free()
    copy_us_in_run = ev_copy[0].elapsed_time(ev_copy[1]) * 1e3

    # the kernels alone, from CUDA-graph replays so no host time is counted:
    # the attention launch of the final step (batch of 8 x 1283 tokens) and
    # the copy-on-write launch (7 pairs of scratch blocks)
    last = stages[(steps - 1) % 2]
    reps = 50

    def graph_time_us(fn):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_):
            for _ in range(reps):
                fn()
        g_.replay()
        torch.cuda.synchronize()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        g_.replay()
        b_.record(stream)
        torch.cuda.synchronize()
        return a_.elapsed_time(b_) * 1e3 / reps

    attn_us = graph_time_us(lambda: pa.pa_decode_attention(
        q, kc, vc, last.d32[:S * MB].view(S, MB), last.d32[S * MB:], D ** -0.5, Hkv, last.dout,
        max_seq_len=MB * B, workspace=ws))
    free_ids = list(pool._free)[:14]
    cpd = torch.tensor([[free_ids[2 * i], free_ids[2 * i + 1]] for i in range(7)],
                       dtype=torch.int64, device=dev)
    copy_us = graph_time_us(lambda: pa.pa_copy_blocks([kc], [vc], cpd))
    copy_bytes = 7 * 2 * 2 * block_bytes               # K and V, read + write
    final_logical = S * (P0 + steps) * 2 * Hkv * D * 2
    final_unique = in_use * 2 * block_bytes
    assert pa.pa_get_device_error() == 0

    # e2e: a fresh fork of the prompt, the same 256 steps with per-step
    # input and output copies
    e2e = None
    if not args.no_e2e:
        for s_ in seqs:
            pool.release(s_)
        pool2 = fresh_prompt()
        for s_ in range(1, S):
            pool2.fork(0, s_)
        graphs2 = None if args.no_graph else capture(True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        lg2, _, cp2 = run(pool2, seqs, steps, graphs2, e2e=True)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        assert pa.pa_get_device_error() == 0 and cp2 == copies
        stage = stages[0]
        h2d = (stage.h32.numel() * 4 + S * 8 + sum(h.numel() * 2 for h in stage.hin))
        e2e = {"value": round(lg2 / e2e_s / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": stage.hout.numel() * 2,
               "note": "host allocator, table upload, q/k/v up and output down every step; "
                       "copy-pair bytes (7 x 16 B at step 0) not in h2d"}
    if sampler is not None:
        time.sleep(0.25)
        sampler.stop()
    peak, peak_kind = measured_peak()
    line = {
        "metric": METRIC, "value": round(logical / dt / 1e9, 2), "unit": "GB/s",
        "n_gpus": 1, "steps": steps, "warmup": warm,
        "ms_per_step": round(1e3 * dt / steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "seq_tokens_per_s": round(logical / (2 * Hkv * D * 2) / dt, 1),
        "config": {"workload": "shared_prefix",
                   "shape": "8 samples x 1027-token prompt (64 full blocks + 3-token tail), "
                            "32/32 heads, D=128, B=16, bf16; 256 decode steps",
                   "timed": "all 256 steps, step 0's copy-on-write included; warm-up on "
                            "throw-away forks",
                   "unique_block_GBps": round(unique / dt / 1e9, 2),
                   "copy_on_write_pairs": copies,
                   "blocks_in_use": in_use,
                   "logical_kv_bytes_per_step_mean": round(logical / steps),
                   "unique_kv_bytes_per_step_mean": round(unique / steps),
                   "l2": "L2-warm: %.1f MB of blocks in use at the end, 129 MB L2; the "
                         "shared prefix is read 8x per step" % (in_use * 2 * block_bytes / 1e6),
                   "parallelism": "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "pa_decode_attention",
                     "achieved": round(final_unique / (attn_us * 1e-6) / 1e9, 1),
                     "achieved_logical": round(final_logical / (attn_us * 1e-6) / 1e9, 1),
                     "peak": peak, "peak_kind": f"hbm_gbs of {peak_kind}", "unit": "GB/s",
                     "frac": round(final_unique / (attn_us * 1e-6) / 1e9 / peak, 4),
                     "traffic": None, "avg_launch_us": round(attn_us, 2),
                     "algorithmic_bytes_per_launch": final_unique,
                     "launch": "the final step's attention (8 x 1283 tokens), 50 launches "
                               "replayed from a CUDA graph",
                     "note": "achieved counts each physical block once per launch (unique "
                             "bytes); the working set fits in L2, so this can pass the HBM peak"},
        "copy_blocks": {"pairs": 7, "bytes_per_launch": copy_bytes,
                        "avg_launch_us": round(copy_us, 2),
                        "GBps": round(copy_bytes / (copy_us * 1e-6) / 1e9, 1),
                        "launch_us_in_timed_step0": round(copy_us_in_run, 2)},
        "gpu_launches": steps * 3 + 1,
        "launch": "cuda graph per step (one per staging buffer), copy-on-write launch eager"
                  if graphs is not None else "eager",
        "e2e": e2e,
        "clocks": sampler.summary(t_host0, t_host1) if sampler else None,
        "device": props.name,
    }
    if not args.no_cpu_baseline:
        # the oracle on the final step's batch (8 samples of 1283 tokens,
        # the shared prefix read once per sample like the kernel)
        final = pool2 if e2e is not None else pool      # the pool whose blocks kc/vc hold
        tabs = final.table_rows(seqs, MB)
        lens_np = np.full(S, P0 + steps, dtype=np.int32)
        arrays = {"q": np_(q), "kc": np_(kc), "vc": np_(vc), "tables": tabs.astype(np.int32),
                  "lens": lens_np}
        cfg = workloads.DecodeConfig("shared_prefix", S, Hkv, Hkv, D, B, "bf16")
        workers = host_cores()
        timer = OracleTimer(arrays, cfg, D ** -0.5, workers)
        try:
            timer.size_sample(args.cpu_baseline_seconds)
            gbs, tps, desc, dt_o = timer.measure()
        finally:
            timer.close()
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": workers,
                                "kind": "oracle", "sample": desc,
                                "seq_tokens_per_s": round(tps, 1),
                                "seconds": round(dt_o, 2)}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    elif args.config == "shared_prefix":
        shared_prefix_arm(args)
    else:
        ours_arm(args)


if __name__ == "__main__":
    main()
