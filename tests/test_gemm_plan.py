"""Host logic of the GEMM launch plan (CPU; no device needed): tile width, CTA pairs,
K per pipeline stage and the split-K choices, through sv_debug_gemm_plan on a 152-SM
GB300. The decisions pinned here are the ones the measurements chose (the split of the
729-row MLP-down GEMM at one image, of the last round at 32 images, none for E4M3 at two
images), and the plan's invariants hold over a sweep of shapes."""
import itertools

import pytest

import vision_transformer_gb300 as vt

SMS = 152


def plan(M, N, K, fp8=0, max_splits=8, sms=SMS):
    return vt.sv_debug_gemm_plan(M, N, K, fp8, sms, max_splits)


def tile_items(p, M, N):
    mt = (M + 127) // 128
    units = (mt + 1) // 2 if p["pairs"] else mt
    return units * -(-N // p["bn"])


def test_one_image_mlp_down_splits_every_tile():
    p = plan(729, 1152, 4304)
    assert (p["bn"], p["pairs"], p["atoms"]) == (256, 1, 1)
    assert (p["k_splits"], p["kb_split"], p["n_main"]) == (5, 14, 0)  # 67 stages of 64 K
    # 15 pair tiles (3 pair rows x 5 column tiles) x 5 ranges of 256 x 256 F32
    assert p["ws_bytes"] == 15 * 5 * 256 * 256 * 4


def test_no_workspace_no_split():
    p = plan(729, 1152, 4304, max_splits=1)
    assert p["k_splits"] == 1 and p["ws_bytes"] == 0
    assert p["bn"] == 64 and p["pairs"] == 1  # the picker's choice without a split


def test_thirty_two_images_split_the_last_round():
    p = plan(32 * 729, 1152, 4304)
    # 92 pair rows x 5 = 460 tiles on 76 pairs: 456 in six full rounds, 4 left over
    assert tile_items(p, 32 * 729, 1152) == 460
    assert (p["n_main"], p["k_splits"], p["kb_split"]) == (456, 8, 9)
    assert p["ws_bytes"] == 4 * 8 * 256 * 256 * 4


@pytest.mark.parametrize("M,fp8", [(32 * 729, 1), (128 * 729, 0), (2 * 729, 1), (1 * 729, 1)])
def test_no_split_where_it_did_not_pay(M, fp8):
    """E4M3 last rounds (slower when split), a last round of one narrow tile (128 images),
    E4M3 at one and two images (their main loop is short against the reduction)."""
    assert plan(M, 1152, 4304, fp8)["k_splits"] == 1


@pytest.mark.parametrize("M", [1, 32, 128])
def test_map_head_second_projection_splits(M):
    """The MAP head's 4304 -> 1152 projection has one row tile: both dtypes split it."""
    for fp8 in (0, 1):
        p = plan(M, 1152, 4304, fp8)
        assert p["k_splits"] >= 7 and p["n_main"] == 0 and p["pairs"] == 0


def test_short_k_never_splits():
    for M in (729, 5832, 23328):
        for N, K in ((3456, 1152), (1152, 1152), (4304, 1152), (1152, 592)):
            assert plan(M, N, K)["k_splits"] == 1


def test_encoder_tiles():
    # QKV / MLP up at one image: 192-wide pairs; at 32 images 256-wide pairs with two rows of K
    assert (plan(729, 3456, 1152)["bn"], plan(729, 3456, 1152)["pairs"]) == (192, 1)
    big = plan(32 * 729, 3456, 1152)
    assert (big["bn"], big["pairs"], big["atoms"]) == (256, 1, 2)
    # the output projection pairs (K >= 1024); the patch embedding (K 592, N 1152) does not
    assert plan(32 * 729, 1152, 1152)["pairs"] == 1
    assert plan(32 * 729, 1152, 592)["pairs"] == 0
    # E4M3 operands never take two rows of K per stage
    assert plan(32 * 729, 3456, 1152, fp8=1)["atoms"] == 1


@pytest.mark.parametrize("fp8", [0, 1])
def test_plan_invariants(fp8):
    for M, N, K in itertools.product((1, 100, 729, 1458, 5832, 23328, 93312), (1152, 2304, 4304),
                                     (592, 1152, 2048, 4304)):
        p = plan(M, N, K, fp8)
        items = tile_items(p, M, N)
        bk = (128 if fp8 else 64) * p["atoms"]
        k_blocks = -(-K // bk)
        assert p["bn"] in (64, 128, 192, 256)
        assert p["tail_n"] == 0 or (p["tail_n"] < p["bn"] and p["tail_n"] % (32 if p["pairs"] else 16) == 0)
        if p["k_splits"] == 1:
            assert p["ws_bytes"] == 0 and p["n_main"] == 0
            continue
        # every range non-empty and together they cover K
        assert p["k_splits"] * p["kb_split"] >= k_blocks > (p["k_splits"] - 1) * p["kb_split"]
        assert p["k_splits"] <= 8 and p["bn"] == 256 and p["atoms"] == 1 and K >= 2048
        assert 0 <= p["n_main"] < items
        rows = 256 if p["pairs"] else 128
        assert p["ws_bytes"] == (items - p["n_main"]) * p["k_splits"] * rows * 256 * 4
        # split items fit one round of the CTAs (pairs) next to nothing else
        slots = SMS // 2 if p["pairs"] else SMS
        assert (items - p["n_main"]) * p["k_splits"] <= slots


def test_fewer_sms_change_the_rounds():
    """On 148 SMs (74 pairs) the 32-image MLP down has 460 % 74 = 16 tiles in its last round,
    more than an eighth of the pairs: no split."""
    assert plan(32 * 729, 1152, 4304, sms=148)["k_splits"] == 1


def test_bad_arguments_rejected():
    lib = vt.load()
    import ctypes
    out = (ctypes.c_int * 8)()
    assert lib.sv_debug_gemm_plan(0, 1152, 1152, 0, SMS, 8, out, None) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_gemm_plan(729, 1000, 1152, 0, SMS, 8, out, None) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_gemm_plan(729, 1152, 1152, 2, SMS, 8, out, None) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_debug_gemm_plan(729, 1152, 1152, 0, 0, 8, out, None) == vt.SV_ERR_INVALID_ARG
