"""Shared test plumbing: tensor <-> numpy views and tolerances.

Holds no arithmetic of the method; the oracle lives in oracle/ and the CUDA
path behind the C ABI."""
import numpy as np
import torch

# max-abs-error bounds against the fp64 oracle (fp32 accumulation on the GPU)
TOL = {"f32": 1e-5, "f16": 1.5e-2, "bf16": 1.5e-2}


def np_(t: torch.Tensor) -> np.ndarray:
    """Storage-typed numpy copy of a tensor (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def bytes_equal(a: torch.Tensor, b: np.ndarray) -> bool:
    return np.array_equal(np_(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


def to_dev(inp, device="cuda"):
    """Device copies of a DecodeInputs' tensors, as a dict."""
    names = ("q", "k_new", "v_new", "key_cache", "value_cache", "block_tables",
             "seq_lens", "positions", "query_start_loc")
    return {n: getattr(inp, n).to(device).contiguous() for n in names}


def max_abs_err(gpu_out: torch.Tensor, oracle_out: np.ndarray, seqs=None, heads=None):
    got = gpu_out.double().cpu().numpy()
    if seqs is not None:
        got = got[np.ix_(seqs, heads)] if heads is not None else got[seqs]
        oracle_out = oracle_out[np.ix_(seqs, heads)] if heads is not None else oracle_out[seqs]
    return float(np.abs(got - oracle_out).max()) if got.size else 0.0
