"""sv_map_pool_static: the MAP head for callers that cannot let the library
allocate device memory at call time (its scratch is a fixed array compiled
into the library). Its output must match the allocating sv_map_pool, call
after call, since both share the same array-free inputs and weights.

This file sorts last so that a run stopping at the first failure has run
every other test already; it initialises its own weights, so it also passes
when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev_f16, host

pytestmark = pytest.mark.gpu

RT = 2.0 ** -10


@pytest.mark.parametrize("gemm_dtype", [0, 1])
def test_static_scratch_matches_allocating_entry_point(sv, gemm_dtype):
    sv.sv_init_weights_dims(0, 729, 588, 1152, 16, 4304, 1)
    for call, B in enumerate((3, 5)):  # two calls in a row, different batches
        x = dev_f16(synth.normal(700 + call, 1, (B, 729, 1152)))
        want = torch.empty(B, 1, 1152, dtype=torch.float16, device="cuda")
        got = torch.empty(B, 1, 1152, dtype=torch.float16, device="cuda")
        sv.sv_map_pool(x, want, B, gemm_dtype)
        sv.sv_map_pool_static(x, got, B, gemm_dtype)
        sv.sv_sync()
        g, w = host(got).reshape(B, -1), host(want).reshape(B, -1)
        assert np.abs(g - w).max() <= 2e-2
        scale = float(np.sqrt(np.mean(w ** 2)))
        assert_close(g, w, 4 * RT, 4 * RT * scale, f"static vs allocating, call {call}")


def test_static_scratch_rejects_oversized_batch(sv):
    sv.sv_init_weights_dims(0, 729, 588, 1152, 16, 4304, 1)
    x = torch.zeros(8, dtype=torch.float16, device="cuda")
    with pytest.raises(sv.SvError) as e:
        sv.sv_map_pool_static(x, x, 257, 0)
    assert e.value.status == sv.SV_ERR_INVALID_ARG
    assert "static buffer" in str(e.value)
