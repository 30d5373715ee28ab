"""sv_map_pool_static: the MAP head for callers that cannot let the library
allocate device memory at call time (its scratch is a fixed array compiled
into the library). Its output must match the allocating sv_map_pool, call
after call, and the oracle's MAP head; calls allocate no device memory.

This file sorts last so that a run stopping at the first failure has run
every other test already; it initialises its own weights, so it also passes
when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, cosine_rows, dev_f16, host

pytestmark = pytest.mark.gpu

RT = 2.0 ** -10


def _scale(ref):
    return float(np.sqrt(np.mean(np.asarray(ref, dtype=np.float64) ** 2))) + 1e-12


@pytest.fixture(scope="module")
def model1(sv):
    sv.sv_init_weights_dims(0, 729, 588, 1152, 16, 4304, 1)
    return oracle.OracleModel.from_synth(0, synth.so400m(1))


def _static(sv, x, B, gemm_dtype):
    out = torch.full((B, 1, 1152), float("nan"), dtype=torch.float16, device="cuda")
    sv.sv_map_pool_static(x, out, B, gemm_dtype)
    sv.sv_sync()
    return host(out).reshape(B, 1152)


@pytest.mark.parametrize("gemm_dtype", [0, 1])
@pytest.mark.parametrize("B", [1, 3])
def test_static_scratch_matches_oracle(sv, model1, B, gemm_dtype):
    """Against the oracle's MAP head at the tolerances of the allocating entry
    point's tests (F16: max-abs 2e-2 and the MAP element tolerance; E4M3: cosine
    against the oracle's operand-rounding mode and the unquantised oracle)."""
    x = synth.normal(720 + B, 1, (B, 729, 1152))
    got = _static(sv, dev_f16(x), B, gemm_dtype)
    ref = model1.map_pool(x)
    if gemm_dtype == 0:
        assert np.abs(got - ref).max() <= 2e-2
        assert_close(got, ref, 4 * RT, 4 * RT * _scale(ref), f"static map_pool B{B}")
    else:
        assert cosine_rows(got, model1.map_pool(x, fp8=True)).min() > 0.999
        assert cosine_rows(got, ref).min() > 0.99


def test_static_scratch_at_its_maximum_batch(sv, model1):
    """256 images, the documented maximum: every image against the allocating entry
    point, two sampled images against the oracle."""
    B = 256
    x = synth.normal(730, 1, (B, 729, 1152))
    xd = dev_f16(x)
    want = torch.empty(B, 1, 1152, dtype=torch.float16, device="cuda")
    sv.sv_map_pool(xd, want, B, 0)
    got = _static(sv, xd, B, 0)
    w = host(want).reshape(B, -1)
    assert_close(got, w, 4 * RT, 4 * RT * _scale(w), "static vs allocating at B = 256")
    pick = [0, B - 1]
    ref = model1.map_pool(x[pick])
    assert np.abs(got[pick] - ref).max() <= 2e-2
    assert_close(got[pick], ref, 4 * RT, 4 * RT * _scale(ref), "static vs oracle at B = 256")


def test_static_scratch_allocates_nothing(sv, model1):
    """Device memory is unchanged across calls. The first call on a device may load
    the library's code holding the static array (lazy module loading), so the
    measurement starts after one call; the calls measured use other batch sizes
    than that one (which would need new workspaces on the allocating path)."""
    x = dev_f16(synth.normal(740, 1, (5, 729, 1152)))
    out = torch.empty(5, 1, 1152, dtype=torch.float16, device="cuda")
    sv.sv_map_pool_static(x, out, 2, 0)
    sv.sv_map_pool_static(x, out, 2, 1)
    sv.sv_sync()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for B, dt in ((1, 0), (5, 0), (3, 1), (5, 1)):
        sv.sv_map_pool_static(x, out, B, dt)
    sv.sv_sync()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


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
