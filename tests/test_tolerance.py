"""The GEMM acceptance rule of the parity tests (helpers.py), checked on the host: the output-
rounding term is half a unit in the last place of fp16 / bf16 at the reference's magnitude, and a
result rounded once from an exact value always passes while one off by more than the bound fails."""
import numpy as np
import torch

from helpers import assert_gemm_close, out_half_ulp


def test_half_ulp_values():
    assert out_half_ulp(np.array([1058.98]), 0.0, torch.bfloat16)[0] == 4.0      # bf16 step 8 in [1024, 2048)
    assert out_half_ulp(np.array([1058.98]), 0.0, torch.float16)[0] == 0.5      # fp16 step 1 there
    assert out_half_ulp(np.array([0.75]), 0.0, torch.bfloat16)[0] == 2.0 ** -9
    assert out_half_ulp(np.array([0.0]), 1e-3, torch.float16)[0] == 2.0 ** -21   # 1e-3 in [2^-10, 2^-9)
    assert out_half_ulp(np.array([0.0]), 0.0, torch.float16)[0] == 2.0 ** -25    # subnormal spacing / 2


def test_one_rounding_passes_and_a_larger_error_fails():
    rng = np.random.default_rng(0)
    exact = (rng.standard_normal((4, 256)) * 3000).astype(np.float32)
    B = np.abs(exact).astype(np.float64)            # one dominant product: |C| == sum |a*w|
    for dt in (torch.float16, torch.bfloat16):
        C = torch.from_numpy(exact).to(dt)           # RN to the output dtype
        assert_gemm_close(C, exact, B, str(dt))
        bound = 2e-3 * B + 1e-3 + out_half_ulp(exact, 2e-3 * B + 1e-3, dt)
        off = torch.from_numpy((exact.astype(np.float64) + 1.5 * bound).astype(np.float32)).to(dt)
        try:
            assert_gemm_close(off, exact, B, str(dt))
        except AssertionError:
            pass
        else:
            raise AssertionError("an error of 1.5x the bound passed for %s" % dt)
