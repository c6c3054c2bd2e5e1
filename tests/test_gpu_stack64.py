"""The 64-layer stack at T = 8 rows on the GPU: 64 independent MLP blocks at the
5120/17408 shape (6.4 GB of packed weights), a residual add and a unit-weight
RMSNorm between layers (eps 1e-6, FP16 storage), as the oracle's `stack` defines.

Two checks:
  * free running, as the benchmark runs it: 64 vq3_mlp_prenorm_step calls chained
    through the FP32 partial sums of squares, from X to r_64, compared with the
    oracle's stack over the same 64 layers (each layer's error logged);
  * teacher forced, on sampled layers, through the separate RMSNorm kernel and
    vq3_mlp_forward: for layer l the oracle recomputes the step from the GPU's own
    residual r_l and the GPU's normed input, MLP output and next residual are
    compared with it."""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vq3_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402
from tests.parity import MIN_ROW_COSINE, REL_MAX_ERR, assert_parity  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LAYERS = 64
SAMPLED = (0, 21, 42, 63)


def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to("cuda")


def _layers(seed):
    """The same draws as synth.inputs.mlp_stack(seed, rows, layers=64), one layer at a time."""
    g = S.rng(seed, 1)
    for _ in range(LAYERS):
        yield S.mlp_block(g, S.HIDDEN, S.INTERMEDIATE, 1024)


def test_stack_64_layers_free_running_prenorm_chain():
    """The stack as the benchmark runs it: 64 chained vq3_mlp_prenorm_step calls from X.

    Every layer's step is gated at the full tolerance, teacher forced: the oracle's MLP of
    RMSNorm(r_l), with r_l the GPU's own residual, against the GPU's output of that layer
    (max|diff| / max|ref| <= 2e-3, row cosine >= 0.9999), and the GPU's next residual equal
    to the exact FP16 sum r_l + out_l. The free-running residuals are compared with the
    oracle's own 64-layer stack at every layer: row cosine >= 0.9999, and each layer's max
    error logged. (A one-ulp change of X alone moves the oracle's r_64 by more than 2e-3,
    see test_oracle_stack_sensitivity.py, so the free-running max error is logged, not gated.)
    Both oracle chains run in one pass over the layers: 8 free-running and 8 teacher-forced
    rows per MLP call."""
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3

    seed, rows, eps = 3, 8, 1e-6
    x = S.activations(S.rng(seed, 0), rows, S.HIDDEN)
    layers = [vq3.MLP.from_block(blk, "cuda") for blk in _layers(seed)]
    res = [f16(x), torch.empty((rows, S.HIDDEN), dtype=torch.float16, device="cuda")]
    ss = [torch.empty((rows, S.HIDDEN // 16), dtype=torch.float32, device="cuda") for _ in range(2)]
    out = torch.empty_like(res[0])
    ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, layers[0]))
    r_gpu, y_gpu = [x], []
    for li, layer in enumerate(layers):
        vq3.mlp_prenorm_step(res[li % 2], layer, out, res[(li + 1) % 2], ss=ss[li % 2] if li > 0 else None,
                             ss_next=ss[(li + 1) % 2], eps=eps, ws=ws)
        y_gpu.append(out.cpu().numpy())
        r_gpu.append(res[(li + 1) % 2].cpu().numpy())
    assert vq3.workspace_status(ws) == 0
    del layers

    workers = min(16, os.cpu_count() or 1)
    r_ref = x
    log, bad = [], []
    for li, blk in enumerate(_layers(seed)):
        n_free = O.rmsnorm(r_ref, eps)
        n_forced = O.rmsnorm(r_gpu[li], eps)
        y = O.mlp_f64(np.vstack([n_free, n_forced]), blk, workers)
        r_ref = O.residual_add(r_ref, y[:rows].astype(np.float16))
        e_step = O.rel_max_err(y_gpu[li], y[rows:])
        c_step = O.row_cosine(y_gpu[li], y[rows:]).min()
        exact_add = np.array_equal(r_gpu[li + 1].view(np.uint16), O.residual_add(r_gpu[li], y_gpu[li]).view(np.uint16))
        e_free = O.rel_max_err(r_gpu[li + 1], r_ref)
        c_free = O.row_cosine(r_gpu[li + 1], r_ref).min()
        log.append(f"layer {li + 1}: step rel_max_err={e_step:.2e} cos={c_step:.8f} add_exact={exact_add}; "
                   f"free-running r rel_max_err={e_free:.2e} cos={c_free:.8f}")
        if not (e_step <= REL_MAX_ERR and c_step >= MIN_ROW_COSINE and exact_add and c_free >= MIN_ROW_COSINE):
            bad.append(li + 1)
    print("\n".join(log))
    assert not bad, f"layers failing the gates: {bad}\n" + "\n".join(log)


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
