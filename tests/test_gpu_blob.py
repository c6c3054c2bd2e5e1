"""A matrix loaded from its packed-weight blob computes exactly what the same matrix packed
directly computes (the blob's GPU-layout section is used as it is)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("fmt,rank", [("2x64", 0), ("2x16", 64), ("lut4", 16)])
@pytest.mark.parametrize("rows", [8, 64])
def test_from_blob_bit_identical(fmt, rank, rows):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3
    m = S.matrix(S.rng(210), 1024, 512, 1024, fmt)
    m.signs = S.sign_bits(S.rng(211), 1024)
    if rank:
        S.add_lowrank(S.rng(212), m, rank, 0.02)
    x = torch.from_numpy(S.activations(S.rng(213), rows, 1024)).to(DEV)
    a = vq3.linear_forward(x, vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    b = vq3.linear_forward(x, vq3.Linear.from_blob(vq3.save_blob(m), DEV)).cpu().numpy()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
