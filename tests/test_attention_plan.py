"""Host logic of the attention kernel choice (CPU; no device needed), through
sv_debug_attention_plan on a 152-SM GB300. Items of one 128-query tile (the
three-score-slot kernel) run when all of them fit in the first round of the grid; items
of two tiles otherwise. The choices pinned here are the ones the measurements made: one
image of 729 tokens and 16 heads takes the slot kernel (2.00 -> 1.88 ms per encoder step),
two images and more the two-tile kernel (the slot kernel was 4% slower at two images)."""
import pytest

import vision_transformer_gb300 as vt

SMS = 152


@pytest.fixture(autouse=True)
def by_size():
    vt.sv_debug_attention_kernel(0)
    yield
    vt.sv_debug_attention_kernel(0)


def plan(B, T=729, H=16, sms=SMS):
    return vt.sv_debug_attention_plan(B, T, H, sms)


def test_one_image_takes_the_slot_kernel():
    assert plan(1) == {"kernel": 2, "grid": 96}  # 6 query tiles x 16 heads


@pytest.mark.parametrize("B,grid", [(2, 96), (8, 152), (32, 152), (128, 152)])
def test_larger_batches_take_two_tile_items(B, grid):
    assert plan(B) == {"kernel": 1, "grid": grid}  # 3 query pairs x 16 heads x B, capped at the SMs


def test_boundary_is_one_round():
    # one 128-token tile per head: B x H one-tile items
    assert plan(152, T=128, H=1) == {"kernel": 2, "grid": 152}
    assert plan(153, T=128, H=1) == {"kernel": 1, "grid": 152}
    assert plan(1, T=729, H=16, sms=95) == {"kernel": 1, "grid": 48}
    assert plan(1, T=1, H=1) == {"kernel": 2, "grid": 1}


def test_forced_choice():
    vt.sv_debug_attention_kernel(1)
    assert plan(1) == {"kernel": 1, "grid": 48}
    vt.sv_debug_attention_kernel(2)
    assert plan(128) == {"kernel": 2, "grid": 152}
    assert plan(1, T=300, H=4) == {"kernel": 2, "grid": 12}
    vt.sv_debug_attention_kernel(0)
    assert plan(1) == {"kernel": 2, "grid": 96}


def test_bad_arguments_rejected():
    lib = vt.load()
    import ctypes
    k, g = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.sv_debug_attention_kernel(3) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_attention_kernel(-1) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_attention_plan(0, 729, 16, SMS, ctypes.byref(k), ctypes.byref(g)) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_attention_plan(1, 729, 16, 0, ctypes.byref(k), ctypes.byref(g)) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_attention_plan(1, 729, 16, SMS, None, ctypes.byref(g)) == vt.SV_ERR_INVALID_ARG
