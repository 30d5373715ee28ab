"""The resident parameters read back through the C ABI (sv_export_weights,
sv_export_weights_e4m3) equal the values the seeded generator draws: every
tensor bit for bit, in the generator's order and logical layout, which checks
the upload's transposes, the patch weight's K padding, the LayerNorm fold into
the QKV / MLP-up weights (scale 1) and the E4M3 copies of the dense weights."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,dims", [("so400m_1layer", synth.so400m(1)), ("vit_small", synth.vit_small(2))])
def test_export_equals_generator(sv, name, dims):
    d = dims
    sv.sv_init_weights_dims(5, d.tokens, d.patch_dim, d.width, d.heads, d.mlp, d.layers)
    infos = synth.tensor_infos(d)
    n = sv.sv_weights_count()
    assert n == sum(t.rows * t.cols for t in infos)
    got = np.full(n, np.nan, dtype=np.float32)
    sv.sv_export_weights(got, n)
    off = 0
    for tid, t in enumerate(infos):
        want = synth.tensor(5, d, tid).astype(np.float32).ravel()
        assert np.array_equal(got[off:off + want.size].view(np.uint32), want.view(np.uint32)), t.name
        off += want.size
    n8 = sv.sv_weights_count_e4m3()
    got8 = np.zeros(n8, dtype=np.uint8)
    sv.sv_export_weights_e4m3(got8, n8)
    off = 0
    for tid, t in enumerate(infos):
        tname = t.name.decode()
        if not (tname.endswith("_w") or tname == "probe"):
            continue
        w = synth.tensor(5, d, tid).astype(np.float32)
        want = torch.from_numpy(16.0 * w).to(torch.float8_e4m3fn).view(torch.uint8).numpy().ravel()
        assert np.array_equal(got8[off:off + want.size], want), tname
        off += want.size
    assert off == n8, name


def test_export_rejects_a_short_buffer(sv):
    sv.sv_init_weights_dims(0, 4, 588, 144, 2, 288, 1)
    n = sv.sv_weights_count()
    buf = np.zeros(n - 1, dtype=np.float32)
    with pytest.raises(sv.SvError) as e:
        sv.sv_export_weights(buf, n - 1)
    assert e.value.status == sv.SV_ERR_INVALID_ARG
