"""The 64-layer stack at T = 8 rows on the GPU: 64 independent MLP blocks at the
5120/17408 shape (6.4 GB of packed weights), a residual add and a unit-weight
RMSNorm between layers (eps 1e-6, FP16 storage), as the oracle's `stack` defines.

Running the oracle through 64 full layers takes minutes, so sampled layers are
checked teacher-forced: for layer l the oracle recomputes the step from the
GPU's own residual r_l (RMSNorm, MLP, residual add) and the GPU's normed input,
MLP output and next residual are compared with it. The 4-layer free-running
stack in test_gpu_parity.py covers error growth across layers."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vq3_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402
from tests.parity import assert_parity  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LAYERS = 64
SAMPLED = (0, 21, 42, 63)


def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to("cuda")


def test_stack_64_layers_sampled_teacher_forced():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3

    seed, rows, eps = 3, 8, 1e-6
    # the same draws as synth.inputs.mlp_stack(seed=3, rows=8, layers=64), one layer at a time
    x = S.activations(S.rng(seed, 0), rows, S.HIDDEN)
    g = S.rng(seed, 1)
    layers, kept = [], {}
    for li in range(LAYERS):
        blk = S.mlp_block(g, S.HIDDEN, S.INTERMEDIATE, 1024)
        layers.append(vq3.MLP.from_block(blk, "cuda"))
        if li in SAMPLED:
            kept[li] = blk

    resid = f16(x)
    normed = torch.empty_like(resid)
    y = torch.empty_like(resid)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, layers[0]))
    seen, r_after = {}, {}
    for li, layer in enumerate(layers):
        vq3.residual_rmsnorm(resid, y if li > 0 else None, eps, normed)
        if li - 1 in SAMPLED:
            r_after[li - 1] = resid.cpu().numpy()  # r_l + y_l of the sampled layer before
        r_l = resid.cpu().numpy() if li in SAMPLED else None
        vq3.mlp_forward(normed, layer, out=y, ws=ws)
        if li in SAMPLED:
            seen[li] = (r_l, normed.cpu().numpy(), y.cpu().numpy())
    vq3.residual_rmsnorm(resid, y, eps, normed)
    r_end = resid.cpu().numpy()
    r_after[LAYERS - 1] = r_end
    assert vq3.workspace_status(ws) == 0
    assert np.isfinite(r_end.astype(np.float64)).all()

    for li in SAMPLED:
        r_l, n_gpu, y_gpu = seen[li]
        n_ref = O.rmsnorm(r_l, eps)
        # RMSNorm: within one FP16 ulp of the FP64 value
        tol = np.spacing(np.abs(n_ref)).astype(np.float64) + 2.0 ** -24
        assert np.all(np.abs(n_gpu.astype(np.float64) - n_ref.astype(np.float64)) <= tol), f"layer {li} RMSNorm"
        # MLP of layer l on the GPU's own normed input
        assert_parity(y_gpu, O.mlp_f64(n_gpu, kept[li]), f"stack layer {li} MLP")
        # residual add: the exact FP16 sum of the GPU's operands
        assert np.array_equal(r_after[li].view(np.uint16), O.residual_add(r_l, y_gpu).view(np.uint16)), li
