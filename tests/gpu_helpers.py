"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, compare element by element."""
import numpy as np
import torch

import oracle
import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import build
from speculative_decoding_target_gb300 import workloads as wl

# bf16 KV: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise; FP8 KV: 5e-2
# absolute.  The bounds are the stated parity tolerances; a bf16 output
# rounding alone contributes up to 2^-9 |o|.
BF16_ATOL, BF16_RTOL = 2e-3, 1e-2
FP8_ATOL = 5e-2

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        sv.load()
        _built = True


def oracle_attention(inp, rows=None, threads=0):
    bits = wl.to_numpy_bits
    fp8 = inp["k_scales"] is not None
    return oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        num_kv_heads=inp["num_kv_heads"], scale=inp["scale"],
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None, rows=rows,
        threads=threads)


def gpu_attention(inp, checked=False, workspace=None):
    ensure_built()
    return sv.verify_attention(
        inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
        inp["seq_lens"], scale=inp["scale"], k_scales=inp["k_scales"],
        v_scales=inp["v_scales"], checked=checked, workspace=workspace)


def assert_attention_close(gpu_rows: np.ndarray, ref_rows: np.ndarray,
                           fp8: bool, what: str = ""):
    g = gpu_rows.astype(np.float64)
    assert g.shape == ref_rows.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref_rows)
    if fp8:
        bound = np.full_like(ref_rows, FP8_ATOL)
    else:
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref_rows)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
            f"max abs err {err.max():.3e}; first bad {idx.tolist()} "
            f"gpu {g[tuple(idx[0])]:.6f} ref {ref_rows[tuple(idx[0])]:.6f}")


def rows_of(out: torch.Tensor, rows=None) -> np.ndarray:
    flat = out.float().reshape(-1, out.shape[-1]).cpu().numpy()
    return flat if rows is None else flat[np.asarray(rows)]
