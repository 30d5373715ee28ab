"""Per-op parity of the CUDA kernels (through the C ABI) with the CPU oracle.

Inputs are seeded synthetic F16 tensors from synth/; both sides read the same
values. Shapes cover several tiles with ragged tails and the full So400m/14
shapes at batch 8 (the single-layer batch-8 configuration's per-stage checks).

Tolerances (derived from the arithmetic): the kernels accumulate in F32 and
round the result once to F16 (relative 2^-11); the oracle accumulates in
double. An F16 result is accepted when |gpu - ref| <= 2^-10 |ref| + atol, with
atol a 2^-10 fraction of the output scale. Attention rounds P to F16 before
the PV product, adding at most 2^-11 of max|v|. An E4M3 result may differ from
the reference by one E4M3 step (2^-3 relative) where the two sides round a
value that sits within 2^-10 of a rounding boundary.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, decode_e4m3, dev_f16, host

pytestmark = pytest.mark.gpu

RT = 2.0 ** -10


def _gemm_inputs(seed, M, N, K):
    A = synth.normal(seed, 1, (M, K))
    W = synth.normal(seed, 2, (K, N), std=1.0 / np.sqrt(K))
    b = synth.normal(seed, 3, (N,), std=0.01)
    return A, W, b


def _scale(ref):
    return float(np.sqrt(np.mean(np.asarray(ref, dtype=np.float64) ** 2))) + 1e-12


@pytest.mark.parametrize("M,N,K", [
    (1, 1152, 1152),      # MAP probe projection (one row)
    (200, 48, 80),        # tiny, ragged M
    (729, 1152, 1152),    # out projection, one image
    (1458, 3456, 1152),   # fused QKV, two images
    (729, 4304, 1152),    # MLP up (N tail 4304 = 16*256 + 208)
    (729, 1152, 4304),    # MLP down (K = 4304)
    (729, 1152, 592),     # patch embedding (K 588 padded to 592)
    (5832, 3456, 1152),   # QKV at batch 8
    (333, 2304, 1152),    # MAP KV
])
def test_gemm_f16_bias(sv, M, N, K):
    A, W, b = _gemm_inputs(20 + M % 7, M, N, K)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, None, C, M, N, K)
    sv.sv_sync()
    ref = oracle.linear(A, W, b)
    assert_close(host(C), ref, RT, RT * _scale(ref), f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,act,res", [
    (5832, 4304, 1152, 1, False),  # MLP up + GELU at batch 8
    (5832, 1152, 4304, 0, True),   # MLP down + residual at batch 8
    (5832, 1152, 1152, 0, True),   # output projection + residual at batch 8
])
def test_gemm_batch8_mlp_shapes(sv, M, N, K, act, res):
    """The encoder's MLP and output-projection GEMMs at the single-layer batch-8
    configuration's size (5832 = 8 x 729 rows), element by element."""
    A, W, b = _gemm_inputs(25, M, N, K)
    R = synth.normal(25, 4, (M, N)) if res else None
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, dev_f16(R) if res else None, C, M, N, K,
                        act=act)
    sv.sv_sync()
    ref = oracle.linear(A, W, b, residual=R, act=act)
    assert_close(host(C), ref, RT, RT * _scale(ref), f"gemm {M}x{N}x{K} act {act} residual {res}")


def test_gemm_epilogues_gelu_residual_pos(sv):
    M, N, K = 777, 4304, 1152
    A, W, b = _gemm_inputs(31, M, N, K)
    R = synth.normal(31, 4, (M, N))
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, dev_f16(R), C, M, N, K, act=1)
    sv.sv_sync()
    ref = oracle.linear(A, W, b, residual=R, act=1)
    assert_close(host(C), ref, RT, RT * _scale(ref), "gelu+residual")
    # residual aliasing the output (the encoder's in-place residual stream)
    X = dev_f16(R)
    sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, X, X, M, N, K)
    sv.sv_sync()
    ref = oracle.linear(A, W, b, residual=R)
    assert_close(host(X), ref, RT, RT * _scale(ref), "in-place residual")
    # positional embedding by row m % T
    T = 729
    pos = synth.normal(31, 5, (T, 1152), std=1 / np.sqrt(1152))
    A2, W2, b2 = _gemm_inputs(32, 2 * T, 1152, 592)
    C2 = torch.empty(2 * T, 1152, dtype=torch.float16, device="cuda")
    sv.sv_gemm_bias_act(dev_f16(A2), dev_f16(W2.T), dev_f16(b2), dev_f16(pos), T, None, C2, 2 * T, 1152, 592)
    sv.sv_sync()
    ref = oracle.linear(A2, W2, b2) + np.tile(pos.astype(np.float32), (2, 1))
    assert_close(host(C2), ref, RT, RT * _scale(ref), "pos")


def test_quantize_e4m3_bit_exact(sv):
    x = synth.normal(40, 1, (4096, 64), std=8.0)
    x[0, :8] = np.array([0, -0.0, 1e-5, 30.0, -30.0, 27.9, 0.0625 / 16, 3e4], dtype=np.float16)
    y = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    sv.sv_quantize_e4m3(dev_f16(x), y, x.size)
    sv.sv_sync()
    got = decode_e4m3(y).reshape(x.shape)
    want = np.array([oracle.e4m3(16.0 * float(v)) for v in x.astype(np.float32).ravel()]).reshape(x.shape) / 16.0
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(729, 1152, 1152), (1458, 4304, 1152), (300, 1152, 4304), (1, 1152, 1152)])
def test_gemm_e4m3(sv, M, N, K):
    A, W, b = _gemm_inputs(50, M, N, K)
    A8 = torch.empty(M * K, dtype=torch.uint8, device="cuda")
    W8 = torch.empty(N * K, dtype=torch.uint8, device="cuda")
    sv.sv_quantize_e4m3(dev_f16(A), A8, M * K)
    sv.sv_quantize_e4m3(dev_f16(W.T), W8, N * K)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    sv.sv_gemm_bias_act(A8, W8, dev_f16(b), None, 1, None, C, M, N, K, in_dtype=1, scale_a=2.0 ** -4, scale_w=2.0 ** -4)
    sv.sv_sync()
    ref = oracle.linear(A, W, b, fp8=True)
    assert_close(host(C), ref, RT, RT * _scale(ref), f"e4m3 gemm {M}x{N}x{K}")


def test_gemm_e4m3_output(sv):
    M, N, K = 600, 4304, 1152
    A, W, b = _gemm_inputs(60, M, N, K)
    C = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, None, C, M, N, K, act=1, out_dtype=1)
    sv.sv_sync()
    ref = oracle.linear(A, W, b, act=1)
    got = decode_e4m3(C).reshape(M, N)
    assert_close(got, ref, 2.0 ** -3 + RT, 2.0 ** -10, "e4m3 out")
    # almost every code is the correctly rounded one
    want = np.vectorize(lambda v: oracle.e4m3(16.0 * v))(ref.astype(np.float32)) / 16.0
    assert (got != want).mean() < 0.01


@pytest.mark.parametrize("rows,width", [(1, 1152), (37, 144), (5832, 1152), (1000, 4096)])
def test_layernorm(sv, rows, width):
    x = (synth.normal(70, 1, (rows, width)).astype(np.float32) * 3 + 1.5).astype(np.float16)
    g = synth.normal(70, 2, (width,), mean=1.0, std=0.2)
    bt = synth.normal(70, 3, (width,), std=0.2)
    y = torch.empty(rows, width, dtype=torch.float16, device="cuda")
    sv.sv_layernorm(dev_f16(x), None, dev_f16(g), dev_f16(bt), y, rows, width)
    sv.sv_sync()
    ref = oracle.layernorm(x, g, bt)
    assert_close(host(y), ref, RT, RT, f"layernorm {rows}x{width}")
    y8 = torch.empty(rows, width, dtype=torch.uint8, device="cuda")
    sv.sv_layernorm(dev_f16(x), None, dev_f16(g), dev_f16(bt), y8, rows, width, out_dtype=1)
    sv.sv_sync()
    assert_close(decode_e4m3(y8).reshape(rows, width), ref, 2.0 ** -3 + RT, 2.0 ** -10, "layernorm e4m3")


@pytest.mark.parametrize("rows,width", [(1, 1152), (37, 144), (5832, 1152), (1000, 4096)])
def test_layernorm_residual(sv, rows, width):
    """y = LN(x + res) with the F16 sum written back to x ("SigLIP ViT benchmark",
    LayerNorm/Add paragraph). The sum is one F32 add of two F16 values rounded to
    F16, so the written-back x is bit-exact against the same rounding in numpy; y is
    checked against the oracle's LayerNorm of that sum at the LayerNorm tolerance."""
    x = (synth.normal(72, 1, (rows, width)).astype(np.float32) * 3 + 1.5).astype(np.float16)
    r = synth.normal(72, 4, (rows, width), std=2.0)
    g = synth.normal(72, 2, (width,), mean=1.0, std=0.2)
    bt = synth.normal(72, 3, (width,), std=0.2)
    xs = (x.astype(np.float32) + r.astype(np.float32)).astype(np.float16)
    xd = dev_f16(x)
    y = torch.empty(rows, width, dtype=torch.float16, device="cuda")
    sv.sv_layernorm(xd, dev_f16(r), dev_f16(g), dev_f16(bt), y, rows, width)
    sv.sv_sync()
    assert np.array_equal(xd.cpu().numpy().view(np.uint16), xs.view(np.uint16))
    ref = oracle.layernorm(xs, g, bt)
    assert_close(host(y), ref, RT, RT, f"layernorm+residual {rows}x{width}")
    # E4M3 output from the same sum (x now holds it; a zero residual leaves it unchanged)
    y8 = torch.empty(rows, width, dtype=torch.uint8, device="cuda")
    sv.sv_layernorm(xd, dev_f16(np.zeros_like(r)), dev_f16(g), dev_f16(bt), y8, rows, width, out_dtype=1)
    sv.sv_sync()
    assert np.array_equal(xd.cpu().numpy(), xs)
    assert_close(decode_e4m3(y8).reshape(rows, width), ref, 2.0 ** -3 + RT, 2.0 ** -10, "layernorm+residual e4m3")


@pytest.mark.parametrize("M,N,K,act", [(729, 3456, 1152, 0), (777, 4304, 1152, 1), (200, 48, 80, 0)])
def test_ln_gemm_folded(sv, M, N, K, act):
    """LayerNorm folded into the following GEMM (the encoder's F16 LN1->QKV and
    LN2->MLP-up pairs) against the oracle's LayerNorm followed by its linear map.
    Rows with a large mean (x*3 + 1.5) exercise the mean correction; the folded
    path keeps LN(x) in F32 where the unfolded one rounds it to F16, and rounds
    W*gamma to F16 instead, so the tolerance is two F16 roundings of the output scale."""
    x = (synth.normal(71, 1, (M, K)).astype(np.float32) * 3 + 1.5).astype(np.float16)
    g = synth.normal(71, 2, (K,), mean=1.0, std=0.2)
    bt = synth.normal(71, 3, (K,), std=0.2)
    W = synth.normal(71, 4, (K, N), std=1.0 / np.sqrt(K))
    b = synth.normal(71, 5, (N,), std=0.01)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    sv.sv_ln_gemm(dev_f16(x), dev_f16(g), dev_f16(bt), dev_f16(W.T), dev_f16(b), C, M, N, K, act=act)
    sv.sv_sync()
    ref = oracle.linear(oracle.layernorm(x, g, bt), W, b, act=act)
    assert_close(host(C), ref, RT, 2 * RT * _scale(ref), f"ln_gemm {M}x{N}x{K}")
    # the weights passed in are left unchanged (the call scales a private copy)
    C2 = torch.empty_like(C)
    sv.sv_ln_gemm(dev_f16(x), dev_f16(g), dev_f16(bt), dev_f16(W.T), dev_f16(b), C2, M, N, K, act=act)
    sv.sv_sync()
    assert torch.equal(C, C2)


@pytest.mark.parametrize("B,side,C,patch", [(2, 378, 3, 14), (1, 42, 3, 14), (3, 32, 4, 8)])
def test_pack_patches_bit_exact(sv, B, side, C, patch):
    """Image -> patch-row packing (image-binding paragraph) is a permutation of F16
    values: bit-exact against the oracle's packing."""
    img = synth.uniform(80, side, (B, side, side, C)).astype(np.float16)
    G = side // patch
    out = torch.full((B, G * G, patch * patch * C), float("nan"), dtype=torch.float16, device="cuda")
    sv.sv_pack_patches(dev_f16(img), out, B, side, C, patch)
    sv.sv_sync()
    ref = oracle.pack_patches(img.astype(np.float32), patch).astype(np.float16)
    assert np.array_equal(host(out).astype(np.float16).view(np.uint16), ref.view(np.uint16))


@pytest.fixture(params=[1, 2], ids=["two_tile_items", "score_slots"])
def attn_kernel(request, sv):
    """Runs the test on each attention kernel (1: items of two 128-query tiles, 2: one
    tile with three score slots in tensor memory); launches choose by size otherwise."""
    sv.sv_debug_attention_kernel(request.param)
    yield request.param
    sv.sv_debug_attention_kernel(0)


def _attn_ref(qkv, H):
    D = H * 72
    return oracle.attention(qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H, 72)


@pytest.mark.parametrize("B,H,T,sharp", [(1, 2, 4, 1.0), (2, 16, 729, 1.0), (1, 3, 200, 3.0), (8, 16, 729, 2.0),
                                         (1, 1, 129, 1.0), (1, 2, 1, 1.0), (3, 4, 300, 1.5)])
def test_attention(sv, attn_kernel, B, H, T, sharp):
    D = H * 72
    qkv = synth.normal(80 + T, 1, (B, T, 3 * D))
    qkv[..., :D] = (qkv[..., :D].astype(np.float32) * sharp).astype(np.float16)
    o = torch.empty(B, T, D, dtype=torch.float16, device="cuda")
    sv.sv_attention(dev_f16(qkv), o, B, H, T)
    sv.sv_sync()
    ref = _attn_ref(qkv, H)
    vmax = float(np.abs(qkv[..., 2 * D:].astype(np.float64)).max())
    assert_close(host(o), ref, RT, RT * vmax, f"attention B{B} H{H} T{T}")


@pytest.mark.parametrize("qk8", [0, 1])
def test_attention_repeats_bit_identical(sv, attn_kernel, qk8):
    """The attention kernels' products reuse tensor-memory columns in issue order (the
    next S product overwrites the P values the P V product reads); a race there would
    show up as outputs that differ between identical launches. 12 launches at the batch-32
    size (1536 or 3072 work items over the persistent CTAs) must give the same bits."""
    B, H, T = 32, 16, 729
    D = H * 72
    qkv = dev_f16(synth.normal(95, 1, (B, T, 3 * D)))
    first = torch.empty(B, T, D, dtype=torch.float16, device="cuda")
    sv.sv_attention_ex(qkv, first, B, H, T, flags=qk8)
    o = torch.empty_like(first)
    for _ in range(11):
        sv.sv_attention_ex(qkv, o, B, H, T, flags=qk8)
        sv.sv_sync()
        assert torch.equal(o, first)


@pytest.mark.parametrize("B,H,T,stride", [(2, 16, 729, 80), (1, 3, 200, 72), (3, 4, 300, 96), (1, 2, 1, 80)])
def test_attention_heads(sv, attn_kernel, B, H, T, stride):
    """Per-head Q, K, V [B, H, T, stride]: the columns past the head width are NaN and
    never read; the result equals the attention of the same values in the fused
    layout, and the default scale (0 -> 1/sqrt(72)) equals the explicit one."""
    D = H * 72
    qkv = synth.normal(280 + T, 1, (B, T, 3 * D))
    heads = []
    for j in range(3):
        a = np.full((B, H, T, stride), np.nan, dtype=np.float16)
        a[..., :72] = qkv[..., j * D:(j + 1) * D].reshape(B, T, H, 72).transpose(0, 2, 1, 3)
        heads.append(dev_f16(a))
    o = torch.full((B, T, D), float("nan"), dtype=torch.float16, device="cuda")
    sv.sv_attention_heads(heads[0], heads[1], heads[2], o, B, H, T, head_stride=stride)
    sv.sv_sync()
    ref = _attn_ref(qkv, H)
    vmax = float(np.abs(qkv[..., 2 * D:].astype(np.float64)).max())
    assert_close(host(o), ref, RT, RT * vmax, f"attention (per head) B{B} H{H} T{T} stride {stride}")
    o2 = torch.empty_like(o)
    s32 = float(np.float32(1.0) / np.sqrt(np.float32(72.0)))  # 1/sqrt(72) rounded as the library's F32 does
    sv.sv_attention_heads(heads[0], heads[1], heads[2], o2, B, H, T, head_stride=stride, scale=s32)
    sv.sv_sync()
    assert torch.equal(o, o2)


@pytest.mark.parametrize("B,H,T,sharp", [(1, 2, 4, 1.0), (2, 16, 729, 1.0), (1, 3, 200, 3.0), (3, 4, 300, 1.5),
                                         (1, 1, 129, 1.0), (1, 2, 1, 1.0)])
def test_attention_qk_e4m3(sv, attn_kernel, B, H, T, sharp):
    """FP8 score products ("FP8 attention and resident image/embedding transfers",
    Projected attention): both sides round the same F16 Q and K values to E4M3 at
    scale 2^-4, so the F16 attention tolerance holds against the oracle's QK-rounding
    mode, while the unrounded attention is measurably further away."""
    D = H * 72
    qkv = synth.normal(180 + T, 1, (B, T, 3 * D))
    qkv[..., :D] = (qkv[..., :D].astype(np.float32) * sharp).astype(np.float16)
    o = torch.empty(B, T, D, dtype=torch.float16, device="cuda")
    sv.sv_attention_ex(dev_f16(qkv), o, B, H, T, flags=sv.SV_ATTENTION_QK_E4M3)
    sv.sv_sync()
    ref = oracle.attention(qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H, 72, qk_fp8=True)
    vmax = float(np.abs(qkv[..., 2 * D:].astype(np.float64)).max())
    got = host(o)
    assert_close(got, ref, RT, RT * vmax, f"attention qk-e4m3 B{B} H{H} T{T}")
    if T >= 100:
        assert np.abs(got - _attn_ref(qkv, H)).max() > 4 * RT * vmax


def test_attention_e4m3_output_and_poisoned_neighbours(sv, attn_kernel):
    """Rows past an image's last token and columns outside a head are never
    read as data: the qkv buffer sits inside NaN-filled memory and the output
    buffer starts as NaN."""
    B, H, T = 2, 16, 729
    D = H * 72
    qkv = synth.normal(90, 1, (B, T, 3 * D))
    big = torch.full((B * T * 3 * D + 4096,), float("nan"), dtype=torch.float16, device="cuda")
    view = big[:B * T * 3 * D].view(B, T, 3 * D)
    view.copy_(dev_f16(qkv))
    o = torch.full((B, T, D), float("nan"), dtype=torch.float16, device="cuda")
    sv.sv_attention(view, o, B, H, T)
    sv.sv_sync()
    ref = _attn_ref(qkv, H)
    vmax = float(np.abs(qkv[..., 2 * D:].astype(np.float64)).max())
    assert_close(host(o), ref, RT, RT * vmax, "attention in NaN surroundings")
    o8 = torch.empty(B, T, D, dtype=torch.uint8, device="cuda")
    sv.sv_attention(view, o8, B, H, T, out_dtype=1)
    sv.sv_sync()
    assert_close(decode_e4m3(o8).reshape(B, T, D), ref, 2.0 ** -3 + RT, RT * vmax, "attention e4m3 out")


@pytest.fixture(scope="module")
def full1(sv):
    """Full-width weights with one encoder layer (the MAP head included), on both sides."""
    sv.sv_init_weights_dims(0, 729, 588, 1152, 16, 4304, 1)
    return oracle.OracleModel.from_synth(0, synth.so400m(1))


@pytest.mark.parametrize("B", [1, 3, 8])
def test_map_pool(sv, full1, B):
    x = synth.normal(100 + B, 1, (B, 729, 1152))
    out = torch.empty(B, 1, 1152, dtype=torch.float16, device="cuda")
    sv.sv_map_pool(dev_f16(x), out, B)
    sv.sv_sync()
    ref = full1.map_pool(x)
    got = host(out).reshape(B, 1152)
    assert np.abs(got - ref).max() <= 2e-2
    assert_close(got, ref, 4 * RT, 4 * RT * _scale(ref), f"map_pool B{B}")


def test_map_pool_e4m3(sv, full1):
    B = 2
    x = synth.normal(110, 1, (B, 729, 1152))
    out = torch.empty(B, 1, 1152, dtype=torch.float16, device="cuda")
    sv.sv_map_pool(dev_f16(x), out, B, gemm_dtype=1)
    sv.sv_sync()
    got = host(out).reshape(B, 1152)
    ref_q = full1.map_pool(x, fp8=True)
    ref = full1.map_pool(x)
    cos = (got * ref_q).sum(1) / np.linalg.norm(got, axis=1) / np.linalg.norm(ref_q, axis=1)
    assert cos.min() > 0.999
    cos_u = (got * ref).sum(1) / np.linalg.norm(got, axis=1) / np.linalg.norm(ref, axis=1)
    assert cos_u.min() > 0.99


def test_bounded_wait_reports_timeout_and_context_survives(sv):
    sv.sv_debug_wait_timeout(2000)
    with pytest.raises(sv.SvError) as e:
        sv.sv_sync()
    assert e.value.status == sv.SV_ERR_TIMEOUT
    sv.sv_sync()  # the error word was cleared; the context still works
    x = dev_f16(np.ones((8, 16), dtype=np.float16))
    y = torch.empty(8 * 16, dtype=torch.uint8, device="cuda")
    sv.sv_quantize_e4m3(x, y, 128)
    sv.sv_sync()
    assert np.all(decode_e4m3(y) == 1.0)


def test_gpu_argument_errors(sv):
    x = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(sv.SvError) as e:
        sv.sv_ln_gemm(x, x, x, x, None, x, 64, 64, 8000)
    assert e.value.status == sv.SV_ERR_INVALID_ARG
    with pytest.raises(sv.SvError) as e:
        sv.sv_gemm_bias_act(x, x, None, None, 1, None, x, 64, 60, 64)
    assert e.value.status == sv.SV_ERR_INVALID_ARG
    with pytest.raises(sv.SvError) as e:
        sv.sv_attention(x, x, 1, 1, 4, head_dim=64)
    assert e.value.status == sv.SV_ERR_UNSUPPORTED
