"""GPU parity for one pre-norm residual layer, r' = fp16(r + delta), out =
MLP(fp16(RMSNorm(r'))): fused into the block's kernel up to 16 rows, a separate
RMSNorm kernel from 17 rows on (the stacked workload's residual add and RMSNorm,
eps 1e-6, unit weight, FP16 storage), against the oracle."""

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


@pytest.fixture(scope="module")
def blk(vq3):
    b = S.mlp_block(S.rng(21, 1), 5120, 17408, 1024)
    return b, vq3.MLP.from_block(b, DEV)


def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(DEV)


@pytest.mark.parametrize("rows", [1, 8, 16, 17, 64])
@pytest.mark.parametrize("with_delta", [True, False])
def test_residual_layer(vq3, blk, rows, with_delta):
    b, layer = blk
    r = S.activations(S.rng(22, 0), rows, 5120)
    d = (S.activations(S.rng(23, 0), rows, 5120) * 0.5).astype(np.float16) if with_delta else None
    r_out = torch.empty((rows, 5120), dtype=torch.float16, device=DEV)
    out = torch.empty_like(r_out)
    vq3.mlp_forward_residual(f16(r), f16(d) if d is not None else None, layer, r_out, out)
    r2 = O.residual_add(r, d) if d is not None else r
    assert np.array_equal(r_out.cpu().numpy().view(np.uint16), np.asarray(r2, np.float16).view(np.uint16))
    n = O.rmsnorm(r2, 1e-6)
    assert_parity(out.cpu().numpy(), O.mlp_f64(n, b), f"residual layer rows={rows} delta={with_delta}")


def test_residual_chain_matches_stack(vq3):
    # four layers through two residual buffers equal the oracle's pre-norm stack
    blocks = [S.mlp_block(S.rng(24 + i, 1), 1024, 2048, 1024) for i in range(4)]
    layers = [vq3.MLP.from_block(bb, DEV) for bb in blocks]
    x = S.activations(S.rng(24, 0), 8, 1024)
    ra, rb = f16(x), torch.empty((8, 1024), dtype=torch.float16, device=DEV)
    ya, yb = torch.empty_like(rb), torch.empty_like(rb)
    delta = None
    for i, layer in enumerate(layers):
        vq3.mlp_forward_residual(ra, delta, layer, rb, ya)
        ra, rb = rb, ra
        delta = ya
        ya, yb = yb, ya
    normed = torch.empty_like(ra)
    vq3.residual_rmsnorm(ra, delta, 1e-6, normed)  # the last residual add: the standalone step
    ref = O.stack(x, blocks, 1e-6)
    assert_parity(ra.cpu().numpy(), ref, "4-layer residual chain")
