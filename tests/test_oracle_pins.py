"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks an oracle function against something other than itself: a
direct convolution, a library routine (torch / numpy in float64), an invariant,
a closed form, a brute-force restatement on a tiny input, or a degenerate case
with a known answer. Citations name the page and section of the SigLIP pages.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

PATCH = 14


def _pack_patches(img):
    """[H, W, 3] image -> [T, 588] rows in [patch_y, patch_x, y, x, channel] order
    ("SigLIP ViT benchmark" page, image-binding paragraph)."""
    H, W, C = img.shape
    py, px = H // PATCH, W // PATCH
    return (img.reshape(py, PATCH, px, PATCH, C).transpose(0, 2, 1, 3, 4).reshape(py * px, PATCH * PATCH * C))


@pytest.mark.parametrize("hw", [(28, 28), (42, 28)])
def test_patch_embed_is_valid_stride14_convolution(hw):
    """The 588->D GEMM on packed patches equals a 14x14 stride-14 VALID convolution
    (network paragraph: the embedding GEMM is the patch convolution)."""
    H, W = hw
    D = 16
    img = synth.uniform(5, 100, (H, W, 3)).astype(np.float64)
    Wp = synth.normal(5, 101, (588, D), std=0.05).astype(np.float64)
    bp = synth.normal(5, 102, (D,), std=0.01).astype(np.float64)
    pix = _pack_patches(img)[None]
    got = oracle.patch_embed(pix, Wp, bp, np.zeros((pix.shape[1], D)))[0]
    # brute-force direct convolution with HWIO kernel Wk[y][x][c][o] = Wp[(y*14+x)*3+c][o]
    Wk = Wp.reshape(PATCH, PATCH, 3, D)
    want = np.zeros((H // PATCH, W // PATCH, D))
    for oy in range(H // PATCH):
        for ox in range(W // PATCH):
            for y in range(PATCH):
                for x in range(PATCH):
                    want[oy, ox] += img[oy * PATCH + y, ox * PATCH + x] @ Wk[y, x]
    want += bp
    np.testing.assert_allclose(got, want.reshape(-1, D), rtol=1e-5, atol=1e-5)
    # library convolution (NCHW input, OIHW weight), float64
    t = F.conv2d(torch.from_numpy(img).permute(2, 0, 1)[None], torch.from_numpy(Wk).permute(3, 2, 0, 1),
                 torch.from_numpy(bp), stride=PATCH)
    np.testing.assert_allclose(got, t[0].permute(1, 2, 0).reshape(-1, D).numpy(), rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("side", [28, 42])
def test_pack_then_embed_is_the_patch_convolution(side):
    """The oracle's image packing followed by its embedding GEMM equals torch's
    14x14 stride-14 convolution of the images (float64): a wrong token order, a
    transposed patch or a channel-order slip in the packing would fail this."""
    D, B = 8, 2
    img = synth.uniform(6, 100, (B, side, side, 3)).astype(np.float64)
    Wp = synth.normal(6, 101, (588, D), std=0.05).astype(np.float64)
    bp = synth.normal(6, 102, (D,), std=0.01).astype(np.float64)
    pix = oracle.pack_patches(img)
    assert pix.shape == (B, (side // PATCH) ** 2, 588)
    got = oracle.patch_embed(pix, Wp, bp, np.zeros((pix.shape[1], D)))
    Wk = Wp.reshape(PATCH, PATCH, 3, D)
    t = F.conv2d(torch.from_numpy(img).permute(0, 3, 1, 2), torch.from_numpy(Wk).permute(3, 2, 0, 1),
                 torch.from_numpy(bp), stride=PATCH)
    np.testing.assert_allclose(got, t.permute(0, 2, 3, 1).reshape(B, -1, D).numpy(), rtol=1e-5, atol=1e-5)


def test_patch_embed_adds_position_per_token():
    pix = synth.uniform(6, 1, (2, 4, 588))
    Wp = synth.normal(6, 2, (588, 8), std=0.05)
    pos = synth.normal(6, 3, (4, 8))
    zero = oracle.patch_embed(pix, Wp, np.zeros(8), np.zeros((4, 8)))
    got = oracle.patch_embed(pix, Wp, np.zeros(8), pos)
    np.testing.assert_allclose(got - zero, np.broadcast_to(pos.astype(np.float32), got.shape), atol=1e-6)


def test_linear_matches_float64_matmul_and_gelu_residual():
    A = synth.normal(7, 1, (37, 300)).astype(np.float64)
    W = synth.normal(7, 2, (300, 70), std=0.05).astype(np.float64)
    b = synth.normal(7, 3, (70,), std=0.01).astype(np.float64)
    R = synth.normal(7, 4, (37, 70)).astype(np.float64)
    np.testing.assert_allclose(oracle.linear(A, W, b), A @ W + b, rtol=1e-5, atol=1e-5)
    got = oracle.linear(A, W, b, residual=R, act=1)
    want = F.gelu(torch.from_numpy(A @ W + b), approximate="tanh").numpy() + R
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5)
    # few rows take the column-split path
    np.testing.assert_allclose(oracle.linear(A[:2], W, b), A[:2] @ W + b, rtol=1e-5, atol=1e-5)


def test_gelu_tanh_form():
    """GELU is the tanh form (reading of the pages' "GELU"); pinned to torch's
    approximate='tanh' and to its limits."""
    x = np.linspace(-12, 12, 4001)
    want = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(oracle.gelu(x), want, rtol=1e-6, atol=1e-7)
    assert oracle.gelu([0.0])[0] == 0.0
    assert abs(oracle.gelu([30.0])[0] - 30.0) < 1e-6 and abs(oracle.gelu([-30.0])[0]) < 1e-6
    # differs from the erf form by a small, nonzero amount
    erf = F.gelu(torch.from_numpy(x)).numpy()
    assert 1e-5 < np.abs(oracle.gelu(x) - erf).max() < 1e-3


def test_layernorm_invariants():
    """LayerNorm: eps 1e-6, affine, centred biased variance ("SigLIP ViT benchmark",
    LayerNorm paragraph)."""
    x = (synth.normal(8, 1, (64, 1152)).astype(np.float64) * 3.0 + 1.5)
    ones, zeros = np.ones(1152), np.zeros(1152)
    y = oracle.layernorm(x, ones, zeros).astype(np.float64)
    assert np.abs(y.mean(axis=1)).max() < 1e-6
    var = x.var(axis=1)
    np.testing.assert_allclose(y.var(axis=1), var / (var + 1e-6), rtol=1e-6)
    y2 = oracle.layernorm(x, 2 * ones, 3 * zeros + 3).astype(np.float64)
    np.testing.assert_allclose(y2, 2 * y + 3, rtol=1e-6, atol=1e-6)
    t = F.layer_norm(torch.from_numpy(x), (1152,), eps=1e-6).numpy()
    np.testing.assert_allclose(y, t, rtol=1e-5, atol=1e-5)
    # eps matters for a nearly constant row: var 1e-6 halves the normalised variance
    row = np.array([[1.0 + 1e-3, 1.0 - 1e-3] * 576])
    yr = oracle.layernorm(row, ones, zeros).astype(np.float64)
    assert abs(yr.var() - 0.5) < 1e-3


def test_softmax_rows_sum_to_one_and_shift_invariant():
    x = synth.normal(9, 1, (16, 729)).astype(np.float64) * 4
    p = oracle.softmax_rows(x).astype(np.float64)
    assert np.abs(p.sum(axis=1) - 1).max() < 1e-6
    np.testing.assert_allclose(oracle.softmax_rows(x + 100.0), p, rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(p, torch.softmax(torch.from_numpy(x), dim=1).numpy(), rtol=1e-5, atol=1e-8)


def _naive_attention(q, k, v, heads, dh):
    """Separate triple-loop restatement for tiny shapes."""
    B, T, _ = q.shape
    o = np.zeros_like(q, dtype=np.float64)
    for b in range(B):
        for h in range(heads):
            sl = slice(h * dh, (h + 1) * dh)
            for i in range(T):
                s = [sum(q[b, i, sl][d] * k[b, j, sl][d] for d in range(dh)) / math.sqrt(dh) for j in range(T)]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                tot = sum(e)
                for d in range(dh):
                    o[b, i, h * dh + d] = sum(e[j] * v[b, j, h * dh + d] for j in range(T)) / tot
    return o


def test_attention_brute_force_4_tokens_2_heads():
    """vit-small shape (4 tokens, 2 heads of 72; "SigLIP ViT benchmark", --vit-small)."""
    B, T, H, dh = 2, 4, 2, 72
    q, k, v = (synth.normal(10, i, (B, T, H * dh)).astype(np.float64) for i in range(3))
    got = oracle.attention(q, k, v, H, dh)
    np.testing.assert_allclose(got, _naive_attention(q, k, v, H, dh), rtol=1e-5, atol=1e-6)


def test_attention_library_and_degenerate_cases():
    B, T, H, dh = 1, 37, 3, 72
    q, k, v = (synth.normal(11, i, (B, T, H * dh)).astype(np.float64) * 2 for i in range(3))
    got = oracle.attention(q, k, v, H, dh)
    tq, tk, tv = (torch.from_numpy(a).view(B, T, H, dh).transpose(1, 2) for a in (q, k, v))
    want = F.scaled_dot_product_attention(tq, tk, tv).transpose(1, 2).reshape(B, T, H * dh).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5)
    # one token: the output is V
    np.testing.assert_allclose(oracle.attention(q[:, :1], k[:, :1], v[:, :1], H, dh), v[:, :1], rtol=1e-6, atol=1e-6)
    # permuting keys with values leaves the output unchanged; permuting queries permutes it
    perm = np.random.default_rng(0).permutation(T)
    np.testing.assert_allclose(oracle.attention(q, k[:, perm], v[:, perm], H, dh), got, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(oracle.attention(q[:, perm], k, v, H, dh), got[:, perm], rtol=1e-5, atol=1e-6)


def _small_model(seed=0, tokens=4, layers=1):
    d = synth.Dims(tokens, 588, 144, 2, 288, layers)
    return d, synth.model(seed, d)


def test_map_single_key_returns_projected_value():
    """MAP with one token: softmax over one key is 1, so the pooled vector is that
    token's V projection, then the output projection and the LN/MLP residual
    ("SigLIP ViT benchmark": network paragraph and flowchart)."""
    d, p = _small_model(tokens=1)
    m = oracle.OracleModel(p, 1, 588, 144, 2, 288)
    xf = synth.normal(12, 1, (3, 1, 144)).astype(np.float64)
    got = m.map_pool(xf)
    f = {k: (np.asarray(v, dtype=np.float64) if not isinstance(v, list) else v) for k, v in p.items()}
    D = 144
    v = xf[:, 0] @ f["map_kv_w"][:, D:] + f["map_kv_b"][D:]
    A = v @ f["map_out_w"] + f["map_out_b"]
    ln = F.layer_norm(torch.from_numpy(A), (D,), torch.from_numpy(f["map_ln_g"]), torch.from_numpy(f["map_ln_b"]),
                      eps=1e-6).numpy()
    hdn = F.gelu(torch.from_numpy(ln @ f["map_fc1_w"] + f["map_fc1_b"]), approximate="tanh").numpy()
    want = A + hdn @ f["map_fc2_w"] + f["map_fc2_b"]
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5)


def test_map_identical_keys_ignore_the_probe():
    d, p = _small_model(tokens=4)
    xrow = synth.normal(13, 1, (1, 1, 144))
    xf = np.repeat(xrow, 4, axis=1)
    a = oracle.OracleModel(p, 4, 588, 144, 2, 288).map_pool(xf)
    p2 = dict(p)
    p2["probe"] = synth.normal(13, 2, (1, 144))
    b = oracle.OracleModel(p2, 4, 588, 144, 2, 288).map_pool(xf)
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)


def _torch_encode(p, pix, heads, layers):
    """float64 restatement of the network from torch library routines (F.linear,
    F.layer_norm, F.scaled_dot_product_attention, F.gelu tanh) on small shapes."""
    t = {k: ([torch.from_numpy(np.asarray(x, dtype=np.float64)) for x in v] if isinstance(v, list)
             else torch.from_numpy(np.asarray(v, dtype=np.float64))) for k, v in p.items()}
    x = torch.from_numpy(np.asarray(pix, dtype=np.float64))
    B, T, _ = x.shape
    D = t["pos"].shape[1]
    dh = D // heads

    def lin(a, w, b):
        return F.linear(a, w.T, b)

    def mha(q, k, v):
        sh = lambda a: a.reshape(a.shape[0], a.shape[1], heads, dh).transpose(1, 2)
        o = F.scaled_dot_product_attention(sh(q), sh(k), sh(v))
        return o.transpose(1, 2).reshape(q.shape[0], q.shape[1], D)

    x = lin(x, t["patch_w"], t["patch_b"]) + t["pos"]
    for l in range(layers):
        y = F.layer_norm(x, (D,), t["ln1_g"][l], t["ln1_b"][l], eps=1e-6)
        q, k, v = lin(y, t["qkv_w"][l], t["qkv_b"][l]).split(D, dim=-1)
        x = x + lin(mha(q, k, v), t["out_w"][l], t["out_b"][l])
        y = F.layer_norm(x, (D,), t["ln2_g"][l], t["ln2_b"][l], eps=1e-6)
        x = x + lin(F.gelu(lin(y, t["fc1_w"][l], t["fc1_b"][l]), approximate="tanh"), t["fc2_w"][l], t["fc2_b"][l])
    xf = F.layer_norm(x, (D,), t["enc_ln_g"], t["enc_ln_b"], eps=1e-6)
    q = lin(t["probe"], t["map_q_w"], t["map_q_b"]).expand(B, 1, D)
    k, v = lin(xf, t["map_kv_w"], t["map_kv_b"]).split(D, dim=-1)
    A = lin(mha(q, k, v), t["map_out_w"], t["map_out_b"])
    y = F.layer_norm(A, (D,), t["map_ln_g"], t["map_ln_b"], eps=1e-6)
    out = A + lin(F.gelu(lin(y, t["map_fc1_w"], t["map_fc1_b"]), approximate="tanh"), t["map_fc2_w"], t["map_fc2_b"])
    return out[:, 0].numpy()


@pytest.mark.parametrize("dims", ["vit_small", "four_token"])
def test_whole_network_against_torch_float64(dims):
    d = synth.vit_small(2) if dims == "vit_small" else synth.four_token(1)
    p = synth.model(0, d)
    pix = synth.pixels(1, 2, d.tokens, d.patch_dim)
    m = oracle.OracleModel(p, d.tokens, d.patch_dim, d.width, d.heads, d.mlp)
    got = m.encode(pix)
    want = _torch_encode(p, pix, d.heads, d.layers)
    np.testing.assert_allclose(got, want, rtol=2e-5, atol=2e-5)
    # layer count is honoured: fewer layers give a different embedding
    if d.layers > 1:
        assert np.abs(m.encode(pix, layers=1) - got).max() > 1e-3


def test_e4m3_matches_torch_float8_cast():
    """OCP E4M3 (e4m3fn), round to nearest even; torch's float8_e4m3fn cast is the
    library routine for in-range values. Saturation (satfinite) by definition."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = codes[np.isfinite(codes)]
    assert len(finite) == 254 and finite.max() == 448 and np.sort(np.abs(finite))[2] == 2.0**-9
    for c in finite:  # every code is a fixed point
        assert oracle.e4m3(c) == c
    x = np.concatenate([np.linspace(-460, 460, 20001), np.linspace(-0.05, 0.05, 20001)])
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3(v) for v in x.astype(np.float32)])
    assert np.array_equal(got, want)
    # ties go to even: 1 + 1/16 lies halfway between 1 and 1.125 -> 1; 1 + 3/16 -> 1.25
    assert oracle.e4m3(1.0625) == 1.0 and oracle.e4m3(1.1875) == 1.25
    assert oracle.e4m3(500.0) == 448.0 and oracle.e4m3(-1e9) == -448.0
    assert math.isnan(oracle.e4m3(float("nan")))


def test_fp8_mode_quantises_both_gemm_operands():
    """FP8 GEMMs at scale -4: operands are E4M3(16 x)/16 ("SigLIP ViT benchmark",
    FP8 example and the paragraph after it; reading of the scale convention)."""
    A = synth.normal(14, 1, (9, 64)).astype(np.float64)
    W = synth.normal(14, 2, (64, 24), std=0.1).astype(np.float64)
    q = lambda a: torch.from_numpy((16 * a).astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy() / 16
    np.testing.assert_allclose(oracle.linear(A, W, fp8=True), q(A) @ q(W), rtol=1e-5, atol=1e-6)
    assert np.abs(oracle.linear(A, W, fp8=True) - A @ W).max() > 1e-3


def test_fp8_attention_products_round_q_and_k_only():
    """FP8 attention products ("FP8 attention and resident image/embedding transfers":
    the QK product on E4M3 operands at scale 2^-4): the oracle's scores use
    E4M3(16 q)/16 and E4M3(16 k)/16, rounded by torch's float8 cast here, while V and
    the softmax stay exact; and the whole-network mode applies it to Q and K only."""
    B, H, T, dh = 2, 2, 9, 72
    q = synth.normal(15, 1, (B, T, H * dh)).astype(np.float64)
    k = synth.normal(15, 2, (B, T, H * dh)).astype(np.float64)
    v = synth.normal(15, 3, (B, T, H * dh)).astype(np.float64)
    r8 = lambda a: torch.from_numpy((16 * a).astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy() / 16
    want = oracle.attention(r8(q), r8(k), v, H, dh)
    got = oracle.attention(q, k, v, H, dh, qk_fp8=True)
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-6)
    assert np.abs(got - oracle.attention(q, k, v, H, dh)).max() > 1e-4  # the rounding does change the scores
    # V is not rounded: rounding it too gives a different result
    assert np.abs(got - oracle.attention(r8(q), r8(k), r8(v), H, dh)).max() > 1e-4
    # whole network: the mode only touches attention (same as unquantised with Q, K exact
    # when the FP8 attention bit is off); with it on, the output moves but stays close
    d = synth.vit_small(1)
    m = oracle.OracleModel.from_synth(0, d)
    pix = synth.pixels(1, 2, d.tokens, d.patch_dim)
    base, qk = m.encode(pix), m.encode(pix, fp8_attention=True)
    assert 0 < np.abs(base - qk).max() < 0.1
