"""Shared test helpers: moving generated problems onto the GPU through the library's own
append, comparing results with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances (max-abs per dtype, relative L2) from the stated accuracy target: fp16 outputs within
# max-abs 2e-3, bf16 within 1e-2, relative L2 within 1e-3, with FP32 accumulation. An fp16 / bf16
# output cannot be closer to the exact value than its own rounding, so each bound adds what the
# path's roundings to that type contribute:
#   max-abs: + half an ulp of the oracle value in the output type (elementwise), times the number
#            of roundings to the input type on the path;
#   relL2:   + rho per rounding, rho = relL2(round_t(oracle), oracle) measured on the same data.
# Roundings on the path: the output (when out_dtype is fp16 / bf16) and, for the tensor-core
# prefill, the probabilities P rounded to the input type before the P.V contraction.
MAX_ABS = {"f16": 2e-3, "bf16": 1e-2}
REL_L2 = 1e-3
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the fp16 / bf16 grid at |x| (subnormal spacing near 0)."""
    ax = np.abs(x)
    mant = 10 if dtype == "f16" else 7
    emin = -14 if dtype == "f16" else -126
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** emin)))
    return 2.0 ** (e - mant)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32).to(TORCH_DT[dtype]).to(torch.float64).numpy()


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def check_close(got, ref: np.ndarray, dtype: str, roundings: int, what: str = "") -> dict:
    """got: torch tensor (any float dtype, any device); ref: float64 oracle values.
    roundings: number of roundings to `dtype` on the GPU path (output + P)."""
    g = got.detach().to(torch.float64).cpu().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    rho = rel_l2(round_to(ref, dtype), ref)
    err = np.abs(g - ref)
    bound = MAX_ABS[dtype] + roundings * 0.5 * ulp(ref, dtype)
    worst = float((err - bound).max()) if err.size else 0.0
    rl2 = rel_l2(g, ref)
    rl2_bound = REL_L2 + roundings * rho
    info = dict(max_abs=float(err.max()) if err.size else 0.0, rel_l2=rl2, rel_l2_bound=rl2_bound, rho=rho)
    assert worst <= 0, "%s: max-abs bound exceeded by %.3g (%s)" % (what, worst, info)
    assert rl2 <= rl2_bound, "%s: relative L2 %.3g > %.3g (%s)" % (what, rl2, rl2_bound, info)
    return info


def to_dev(t, dev="cuda"):
    return t.to(dev, non_blocking=False).contiguous()


def device_cache(problem, dev="cuda"):
    """Allocate the pool on the device, fill it with the problem's seeded noise, and append
    every context token through the library's kv_cache_append."""
    import paged_kv_flash_cache_gb300 as pkv
    shape = (problem.num_blocks, 2, problem.num_kv_heads, problem.block_size, problem.head_dim)
    if problem.pool_init is not None:
        cache = problem.pool_init.reshape(shape).to(dev)
    else:
        cache = torch.zeros(shape, dtype=TORCH_DT[problem.dtype], device=dev)
    if problem.k_ctx.shape[0]:
        pkv.kv_cache_append(cache, to_dev(problem.k_ctx, dev), to_dev(problem.v_ctx, dev),
                            to_dev(problem.cu_ctx_lens, dev), torch.zeros(problem.batch, dtype=torch.int32, device=dev),
                            to_dev(problem.block_tables, dev))
    return cache


def cache_bits(cache) -> np.ndarray:
    """Device cache -> host uint16 bits (the oracle's input format)."""
    return cache.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
