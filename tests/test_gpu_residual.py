"""GPU parity for one pre-norm residual layer, r' = fp16(r + delta), out =
MLP(fp16(RMSNorm(r'))): fused into the block's kernel up to 16 rows, a separate
RMSNorm kernel from 17 rows on (the stacked workload's residual add and RMSNorm,
eps 1e-6, unit weight, FP16 storage), against the oracle; and for the sublayer
chained through sums of squares (out = MLP(RMSNorm(r)), r_next = fp16(r + out),
FP32 partial sums of r_next^2 per 16 columns)."""

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


def partial_squares(r):
    """FP32 sums of r^2 per 16 columns: each square rounded to FP32, added in column order."""
    q = np.asarray(r, np.float16).astype(np.float32)
    q = (q * q).astype(np.float32).reshape(q.shape[0], -1, 16)
    s = np.zeros(q.shape[:2], np.float32)
    for k in range(16):
        s = (s + q[..., k]).astype(np.float32)
    return s


@pytest.mark.parametrize("rows", [1, 8, 16, 17, 40])
@pytest.mark.parametrize("with_ss", [False, True])
def test_prenorm_step(vq3, blk, rows, with_ss):
    b, layer = blk
    r = S.activations(S.rng(25, 0), rows, 5120)
    ss = torch.from_numpy(partial_squares(r)).to(DEV) if with_ss else None
    out = torch.empty((rows, 5120), dtype=torch.float16, device=DEV)
    r_next = torch.empty_like(out)
    ss_next = torch.empty((rows, 5120 // 16), dtype=torch.float32, device=DEV)
    vq3.mlp_prenorm_step(f16(r), layer, out, r_next, ss=ss, ss_next=ss_next)
    got = out.cpu().numpy()
    assert_parity(got, O.mlp_f64(O.rmsnorm(r, 1e-6), b), f"prenorm step rows={rows} ss={with_ss}")
    rn = r_next.cpu().numpy()
    assert np.array_equal(rn.view(np.uint16), O.residual_add(r, got).view(np.uint16))
    assert np.array_equal(ss_next.cpu().numpy(), partial_squares(rn))


@pytest.mark.parametrize("rows", [8, 5, 20])
def test_prenorm_chain_matches_stack(vq3, rows):
    # four sublayers, each taking the previous one's residual and partial sums
    blocks = [S.mlp_block(S.rng(30 + i, 1), 1024, 2048, 1024) for i in range(4)]
    layers = [vq3.MLP.from_block(bb, DEV) for bb in blocks]
    x = S.activations(S.rng(30, 0), rows, 1024)
    r = [f16(x), torch.empty((rows, 1024), dtype=torch.float16, device=DEV)]
    ss = [None, torch.empty((rows, 64), dtype=torch.float32, device=DEV),
          torch.empty((rows, 64), dtype=torch.float32, device=DEV)]
    out = torch.empty((rows, 1024), dtype=torch.float16, device=DEV)
    for i, layer in enumerate(layers):
        ss_in = ss[0] if i == 0 else ss[1 + (i - 1) % 2]
        vq3.mlp_prenorm_step(r[i % 2], layer, out, r[(i + 1) % 2], ss=ss_in, ss_next=ss[1 + i % 2])
    ref = O.stack(x, blocks, 1e-6)
    assert_parity(r[len(layers) % 2].cpu().numpy(), ref, f"4-sublayer chain rows={rows}")


@pytest.mark.parametrize("fmt", ["2x16", "lut4"])
@pytest.mark.parametrize("rows", [8, 20])
def test_prenorm_step_formats(vq3, fmt, rows):
    bb = S.mlp_block(S.rng(40, 1), 1024, 2048, 1024, fmt)
    layer = vq3.MLP.from_block(bb, DEV)
    r = S.activations(S.rng(41, 0), rows, 1024)
    out = torch.empty((rows, 1024), dtype=torch.float16, device=DEV)
    r_next = torch.empty_like(out)
    ss_next = torch.empty((rows, 64), dtype=torch.float32, device=DEV)
    vq3.mlp_prenorm_step(f16(r), layer, out, r_next, ss=torch.from_numpy(partial_squares(r)).to(DEV),
                         ss_next=ss_next)
    got = out.cpu().numpy()
    assert_parity(got, O.mlp_f64(O.rmsnorm(r, 1e-6), bb), f"prenorm step {fmt} rows={rows}")
    rn = r_next.cpu().numpy()
    assert np.array_equal(rn.view(np.uint16), O.residual_add(r, got).view(np.uint16))
    assert np.array_equal(ss_next.cpu().numpy(), partial_squares(rn))


@pytest.mark.parametrize("rows", [8, 20])
def test_prenorm_step_repeats_bit_identical(vq3, blk, rows):
    _, layer = blk
    r = f16(S.activations(S.rng(42, 0), rows, 5120))
    ss = torch.from_numpy(partial_squares(r.cpu().numpy())).to(DEV)
    outs = []
    for _ in range(2):
        out = torch.empty((rows, 5120), dtype=torch.float16, device=DEV)
        r_next = torch.empty_like(out)
        ss_next = torch.empty((rows, 320), dtype=torch.float32, device=DEV)
        vq3.mlp_prenorm_step(r, layer, out, r_next, ss=ss, ss_next=ss_next)
        outs.append((out.cpu().numpy().view(np.uint16), r_next.cpu().numpy().view(np.uint16),
                     ss_next.cpu().numpy().view(np.uint32)))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
