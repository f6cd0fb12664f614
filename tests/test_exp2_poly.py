"""The FMA-pipe exp2 used by the prefill softmax: the coefficients compiled into prefill.cu are
the ones the Remez script derives, and the kernel's float32 evaluation order stays within its
stated relative error against the exact 2^x (the GPU path itself is covered by prefill parity)."""
import importlib.util
import os
import re

import numpy as np
import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "paged_kv_flash_cache_gb300", "csrc")


def load_script():
    spec = importlib.util.spec_from_file_location("exp2_poly", os.path.join(CSRC, "exp2_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def kernel_coefficients():
    src = open(os.path.join(CSRC, "prefill.cu")).read()
    body = src[src.index("__device__ __forceinline__ float2 exp2_fma2"):src.index("p = ffma2(p, f, make_float2(1.f, 1.f));")]
    bf16_part, f16_part = body.split("} else {")[0], body.split("} else {")[1]
    grab = lambda t: [float(v) for v in re.findall(r"make_float2\(([-0-9.e+]+)f, \1f\)", t)]
    return grab(bf16_part), grab(f16_part)


@pytest.mark.parametrize("degree,bound", [(3, 4.4e-4), (4, 3.7e-6)])
def test_coefficients_match_remez_and_error_bound(degree, bound):
    mod = load_script()
    coef, err = mod.remez_exp2(degree)
    assert err < bound
    c_bf16, c_f16 = kernel_coefficients()
    kern = c_bf16 if degree == 3 else c_f16
    # kernel lists the Horner order: c_n, c_{n-1}, ..., c_1 (c_0 = 1 is the final FMA)
    np.testing.assert_allclose(kern, coef[1:][::-1].astype(np.float32), rtol=2e-7)
    xs = np.concatenate([np.linspace(-125, 8, 1000001), np.linspace(-1, 1, 100001)]).astype(np.float32)
    y = mod.emulate_f32(xs, coef.astype(np.float32)).astype(np.float64)
    rel = np.abs(y / np.exp2(xs.astype(np.float64)) - 1)
    assert rel.max() < bound * 1.05
    assert mod.emulate_f32(np.array([0.0], np.float32), coef.astype(np.float32))[0] == 1.0
