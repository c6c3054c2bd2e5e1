"""GPU parity for the low-rank correction of a linear layer, W = diag(s) C[idx]
+ U V on the rotated input (model card "anemll/anemll-forge-qwen3.8-27B",
table row "Token mixers": rank-64 factors): the decode kernel (up to 16 rows)
and the tensor-core GEMM (from 17 rows) against the oracle."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vq3_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402
from tests.parity import assert_parity  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def vq3():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3 as m
    return m


def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(DEV)


@pytest.mark.parametrize("fmt", ["2x64", "2x16", "lut4"])
@pytest.mark.parametrize("rank", [8, 64])
@pytest.mark.parametrize("rows", [1, 8, 16, 17, 64, 300])
def test_linear_with_factors(vq3, fmt, rank, rows):
    m = S.matrix(S.rng(70), 1024, 512, 1024, fmt)
    m.signs = S.sign_bits(S.rng(70, 2), 1024)
    S.add_lowrank(S.rng(70, 3), m, rank, 0.02)
    x = S.activations(S.rng(70, 0), rows, 1024)
    got = vq3.linear_forward(f16(x), vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    ref = O.linear_f64(x, m)
    assert_parity(got, ref, f"{fmt} rank {rank} rows={rows}")
    # the correction is not negligible: without it the output would fail the same bar
    m0 = S.Matrix(m.d_in, m.d_out, m.block, m.codebook, m.stream, m.scales, m.signs, fmt)
    assert O.rel_max_err(O.linear_f64(x, m0), ref) > 1e-2


@pytest.mark.parametrize("rows", [8, 64])
def test_token_mixer_shape_with_factors(vq3, rows):
    # a 5120 -> 6144 projection with rank-64 factors (token-mixer shapes are not on the pages: synthetic)
    m = S.matrix(S.rng(71), 5120, 6144, 1024, "2x16")
    S.add_lowrank(S.rng(71, 3), m, 64, 0.02)
    x = S.activations(S.rng(71, 0), rows, 5120)
    got = vq3.linear_forward(f16(x), vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    assert_parity(got, O.linear_f64(x, m), f"5120->6144 rank 64 rows={rows}")


def test_zero_factors_bit_identical(vq3):
    m = S.matrix(S.rng(72), 512, 256, 512)
    x = f16(S.activations(S.rng(72, 0), 8, 512))
    a = vq3.linear_forward(x, vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    m.lr_u = np.zeros((256, 16), np.float16)
    m.lr_v = np.zeros((16, 512), np.float16)
    b = vq3.linear_forward(x, vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


# Below 17 rows the correction is formed inside the decode kernel: the CTAs that decode the
# first segment group project their rotated activations on V, and the output step adds U z.
# These shapes place the first group's cells differently: at 5120 -> 12288 (80 column groups,
# 12 segment groups, 152 CTAs, first-group cells weighted 1.25 in the CTA ranges) sixteen CTAs
# hold the first group and the last of them also starts the second; at 17408 -> 12288 with 12
# rows (two 8-row tiles, 16 stage slots per round) a CTA's 17-18 first-group cells take two
# rounds, and the first round's 16 take three batches of factor columns (7, 7, 2).
@pytest.mark.parametrize("fmt", ["2x16", "2x64", "lut4"])
@pytest.mark.parametrize("rows", [8, 16])
def test_fused_lowrank_token_mixer_5120x12288(vq3, fmt, rows):
    m = S.matrix(S.rng(73, 1), 5120, 12288, 1024, fmt)
    m.signs = S.sign_bits(S.rng(73, 2), 5120)
    S.add_lowrank(S.rng(73, 3), m, 64, 0.02)
    lin = vq3.Linear.from_matrix(m, DEV)
    assert vq3.linear_kernel_launches(rows, lin) == 1
    x = S.activations(S.rng(73, 0), rows, 5120)
    ws = vq3.workspace(vq3.linear_workspace_bytes(rows, lin))
    got = vq3.linear_forward(f16(x), lin, ws=ws).cpu().numpy()
    assert vq3.workspace_status(ws) == 0
    assert_parity(got, O.linear_f64(x, m, workers=8), f"5120->12288 {fmt} rank 64 rows={rows}")
    # the workspace is reused as it is left: a second call gives the same bits
    again = vq3.linear_forward(f16(x), lin, ws=ws).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), again.view(np.uint16))


@pytest.mark.parametrize("rank,rows", [(8, 3), (64, 12)])
def test_fused_lowrank_first_group_over_two_rounds(vq3, rank, rows):
    m = S.matrix(S.rng(74, 1), 17408, 12288, 1024, "2x16")
    S.add_lowrank(S.rng(74, 3), m, rank, 0.02)
    lin = vq3.Linear.from_matrix(m, DEV)
    x = S.activations(S.rng(74, 0), rows, 17408)
    got = vq3.linear_forward(f16(x), lin).cpu().numpy()
    ref = O.linear_f64(x, m, workers=8)
    assert_parity(got, ref, f"17408->12288 rank {rank} rows={rows}")
    m0 = S.Matrix(m.d_in, m.d_out, m.block, m.codebook, m.stream, m.scales, m.signs, "2x16")
    assert O.rel_max_err(O.linear_f64(x, m0, workers=8), ref) > 1e-2


def test_linear_kernel_launches(vq3):
    m = S.matrix(S.rng(75), 1024, 512, 1024)
    plain = vq3.Linear.from_matrix(m, DEV)
    S.add_lowrank(S.rng(75, 3), m, 16, 0.02)
    lr = vq3.Linear.from_matrix(m, DEV)
    assert [vq3.linear_kernel_launches(r, plain) for r in (0, 1, 16, 17, 300)] == [0, 1, 1, 2, 2]
    assert [vq3.linear_kernel_launches(r, lr) for r in (0, 1, 16, 17, 300)] == [0, 1, 1, 5, 5]


@pytest.mark.parametrize("rows", [64, 2048])
def test_prefill_lowrank_token_mixer_5120x12288(vq3, rows):
    # from 17 rows the correction runs as projection (split over the input), reduction and
    # expansion on the tensor cores, added in the GEMM epilogue; 64 rows: the narrow GEMM (x' in
    # its operand order), 2048: the wide one
    m = S.matrix(S.rng(76, 1), 5120, 12288, 1024, "2x16")
    S.add_lowrank(S.rng(76, 3), m, 64, 0.02)
    lin = vq3.Linear.from_matrix(m, DEV)
    x = S.activations(S.rng(76, 0), rows, 5120)
    got = vq3.linear_forward(f16(x), lin).cpu().numpy()
    if rows <= 64:
        assert_parity(got, O.linear_f64(x, m, workers=8), f"5120->12288 rank 64 rows={rows}")
    else:
        # sampled rows against the oracle (every 64th row and the last)
        idx = np.r_[0:rows:64, rows - 1]
        assert_parity(got[idx], O.linear_f64(x[idx], m, workers=8), f"5120->12288 rank 64 rows={rows} (sampled)")
