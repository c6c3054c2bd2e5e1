"""GPU parity for the other index formats: the two-bit vector LUT ("2x16": 16
two-component centroids, a four-bit index per output pair) and the four-bit
scalar LUT ("lut4": 16 entries, a four-bit index per weight), through the same
C ABI and kernels as the three-bit format (model card
"anemll/anemll-forge-qwen3.8-27B", release-comparison table rows "MLP gate / up
/ down" and "Token mixers"). Layout and lookups are compared bit for bit; float
outputs with the tolerance of tests/parity.py."""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vq3_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402
from tests.parity import assert_parity  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = ["2x16", "lut4"]


@pytest.fixture(scope="module")
def vq3():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3 as m
    return m


def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(DEV)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("d_in,d_out", [(256, 256), (128, 512), (5120, 17408), (17408, 5120)])
def test_dequant_bit_exact(vq3, fmt, d_in, d_out):
    m = S.matrix(S.rng(d_in + 11), d_in, d_out, 64, fmt)
    lin = vq3.Linear.from_matrix(m, DEV)
    w_raw = vq3.dequant_dense(lin, False).cpu().numpy()
    w_sc = vq3.dequant_dense(lin, True).cpu().numpy()
    for r0 in range(0, d_out, 2048):
        r1 = min(d_out, r0 + 2048)
        ref_raw = O.dense_weight(m.stream, m.codebook, m.scales, d_in, d_out, apply_scale=False, rows=(r0, r1),
                                 fmt=fmt)
        ref_sc = O.dense_weight(m.stream, m.codebook, m.scales, d_in, d_out, apply_scale=True, rows=(r0, r1),
                                fmt=fmt)
        assert np.array_equal(w_raw[r0:r1].view(np.uint16), ref_raw.astype(np.float16).view(np.uint16))
        assert np.array_equal(w_sc[r0:r1].view(np.uint16), ref_sc.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows", [1, 8, 9, 16, 17, 64, 100, 300])
def test_linear_ragged_rows(vq3, fmt, rows):
    # below 17 rows the decode kernel, from 17 rows on the tensor-core GEMM
    m = S.matrix(S.rng(13), 1024, 512, 1024, fmt)
    m.signs = S.sign_bits(S.rng(13, 2), 1024)
    x = S.activations(S.rng(13, 0), rows, 1024)
    got = vq3.linear_forward(f16(x), vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    assert_parity(got, O.linear_f64(x, m), f"{fmt} linear rows={rows}")


@pytest.mark.parametrize("fmt", FMTS)
def test_codebook_permutation_invariance_bit_exact(vq3, fmt):
    d_in, d_out = 512, 256
    _, vec, entries = O.FORMATS[fmt]
    m = S.matrix(S.rng(14), d_in, d_out, 512, fmt)
    perm = np.random.default_rng(3).permutation(entries)
    idx = O.index_matrix(m.stream, d_in, d_out, fmt=fmt)
    m2 = S.Matrix(d_in, d_out, 512, m.codebook[perm], O.pack_indices(np.argsort(perm)[idx], 4), m.scales, None, fmt)
    for rows in (8, 64):
        x = f16(S.activations(S.rng(14, 0), rows, d_in))
        a = vq3.linear_forward(x, vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
        b = vq3.linear_forward(x, vq3.Linear.from_matrix(m2, DEV)).cpu().numpy()
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.fixture(scope="module", params=FMTS)
def block(vq3, request):
    fmt = request.param
    # 2048 rows: the benchmark times these formats there (the first rows of a taller X
    # equal a shorter X, so one oracle run serves every row count below)
    wl = S.mlp_format(fmt, rows=2048)
    blk = wl.layers[0]
    return fmt, wl, blk, vq3.MLP.from_block(blk, DEV), O.mlp_f64(wl.x, blk, workers=min(16, os.cpu_count() or 1))


@pytest.mark.parametrize("rows", [1, 8, 16, 17, 64, 2048])
def test_mlp_5120x17408(vq3, block, rows):
    fmt, wl, blk, layer, ref = block
    got = vq3.mlp_forward(f16(wl.x[:rows]), layer).cpu().numpy()
    assert_parity(got, ref[:rows], f"{fmt} mlp 5120x17408 T={rows}")


def test_mlp_repeat_deterministic(vq3, block):
    fmt, wl, blk, layer, ref = block
    for rows in (8, 64):
        x = f16(wl.x[:rows])
        ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, layer))
        a = vq3.mlp_forward(x, layer, ws=ws).clone()
        b = vq3.mlp_forward(x, layer, ws=ws)
        assert torch.equal(a, b)
        assert vq3.workspace_status(ws) == 0
