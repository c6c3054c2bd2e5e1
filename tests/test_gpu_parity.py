"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Layout and index unpacking are compared bit for bit; the
float outputs by max|gpu-ref|/max|ref| <= 2e-3 and per-row cosine >= 0.9999."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vq3_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402
from tests.parity import assert_parity  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vq3():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3 as m
    return m


DEV = "cuda"


def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(DEV)


def f16_ulp_close(got, ref):
    """Within one FP16 ulp of the exact value (the only rounding is the final one)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64) + 2.0 ** -24
    return np.all(np.abs(got - ref) <= tol)


# ------------------------------------------------------------------ rotation

@pytest.mark.parametrize("block", [2, 4, 8, 16, 32, 64, 128, 256, 512, 1024])
@pytest.mark.parametrize("signs", [False, True])
def test_fwht_matches_oracle(vq3, block, signs):
    rows, n = 3, 4 * max(block, 64)
    x = S.activations(S.rng(block, 0), rows, n)
    sw = S.sign_bits(S.rng(block, 2), n) if signs else None
    sg = torch.from_numpy(sw.view(np.int32)).to(DEV) if signs else None
    got = vq3.fwht_rotate(f16(x), block, sg).cpu().numpy()
    ref = O.rotate(x.astype(np.float64), block, sw)
    assert f16_ulp_close(got, ref)


def test_fwht_in_place_and_double_rotation(vq3):
    x = S.activations(S.rng(1, 0), 5, 17408)
    t = f16(x)
    vq3.fwht_rotate(t, 1024, None, out=t)
    once = t.cpu().numpy()
    assert f16_ulp_close(once, O.rotate(x.astype(np.float64), 1024))
    vq3.fwht_rotate(t, 1024, None, out=t)
    twice = t.cpu().numpy().astype(np.float64)
    assert np.allclose(twice, x.astype(np.float64), rtol=2e-3, atol=2e-3)


def test_fwht_closed_forms(vq3):
    b = 1024
    e = np.zeros((2, b), np.float16)
    e[0, 5] = 1
    e[1, :] = 0.5
    got = vq3.fwht_rotate(f16(e), b).cpu().numpy().astype(np.float64)
    assert np.array_equal(got[0], O.hadamard(b)[:, 5] / 32.0)
    expect = np.zeros(b)
    expect[0] = 0.5 * 32
    assert np.array_equal(got[1], expect)


# ------------------------------------------------------------------ layout (bit-exact)

@pytest.mark.parametrize("d_in,d_out", [(256, 256), (128, 512), (5120, 17408), (17408, 5120)])
def test_dequant_bit_exact(vq3, d_in, d_out):
    m = S.matrix(S.rng(d_in + 7), d_in, d_out, 64)
    lin = vq3.Linear.from_matrix(m, DEV)
    w_raw = vq3.dequant_dense(lin, False).cpu().numpy()
    w_sc = vq3.dequant_dense(lin, True).cpu().numpy()
    for r0 in range(0, d_out, 2048):
        r1 = min(d_out, r0 + 2048)
        ref_raw = O.dense_weight(m.stream, m.codebook, m.scales, d_in, d_out, apply_scale=False, rows=(r0, r1))
        ref_sc = O.dense_weight(m.stream, m.codebook, m.scales, d_in, d_out, apply_scale=True, rows=(r0, r1))
        assert np.array_equal(w_raw[r0:r1].view(np.uint16), ref_raw.astype(np.float16).view(np.uint16))
        assert np.array_equal(w_sc[r0:r1].view(np.uint16), ref_sc.astype(np.float16).view(np.uint16))


# ------------------------------------------------------------------ linear

def test_linear_256_config(vq3):
    wl = S.linear_256(seed=0, rows=8)
    m = wl.layers[0]
    lin = vq3.Linear.from_matrix(m, DEV)
    got = vq3.linear_forward(f16(wl.x), lin).cpu().numpy()
    assert_parity(got, O.linear_f64(wl.x, m), "linear 256x256 T=8")


@pytest.mark.parametrize("rows", [1, 3, 8, 9, 16, 17, 33, 64, 100, 300])
def test_linear_ragged_rows(vq3, rows):
    m = S.matrix(S.rng(3), 1024, 512, 1024)
    m.signs = S.sign_bits(S.rng(3, 2), 1024)
    x = S.activations(S.rng(3, 0), rows, 1024)
    lin = vq3.Linear.from_matrix(m, DEV)
    got = vq3.linear_forward(f16(x), lin).cpu().numpy()
    assert_parity(got, O.linear_f64(x, m), f"linear rows={rows}")


def test_linear_closed_form_all_equal(vq3):
    d_in, d_out, b, k = 256, 256, 64, 37
    m = S.matrix(S.rng(4), d_in, d_out, b)
    m.stream = O.pack_indices(np.full((d_out // 2) * d_in, k))
    x = S.activations(S.rng(4, 0), 8, d_in)
    got = vq3.linear_forward(f16(x), vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    C = m.codebook.astype(np.float64)
    xs = x.astype(np.float64)[:, ::b].sum(axis=1)
    expect = np.stack([m.scales.astype(np.float64)[o] * C[k][o % 2] * np.sqrt(b) * xs for o in range(d_out)], 1)
    assert_parity(got, expect, "closed form")


def test_codebook_permutation_invariance_bit_exact(vq3):
    d_in, d_out = 512, 256
    m = S.matrix(S.rng(6), d_in, d_out, 512)
    perm = np.random.default_rng(2).permutation(64)
    idx = O.index_matrix(m.stream, d_in, d_out)
    m2 = S.Matrix(d_in, d_out, 512, m.codebook[perm], O.pack_indices(np.argsort(perm)[idx]), m.scales)
    x = f16(S.activations(S.rng(6, 0), 8, d_in))
    a = vq3.linear_forward(x, vq3.Linear.from_matrix(m, DEV)).cpu().numpy()
    b = vq3.linear_forward(x, vq3.Linear.from_matrix(m2, DEV)).cpu().numpy()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


# ------------------------------------------------------------------ MLP block

@pytest.fixture(scope="module")
def cfg1(vq3):
    wl = S.mlp_27b(seed=1, rows=8)
    blk = wl.layers[0]
    return wl, blk, vq3.MLP.from_block(blk, DEV), O.mlp_f64(wl.x, blk)


def test_mlp_27b_T8(vq3, cfg1):
    wl, blk, layer, ref = cfg1
    got = vq3.mlp_forward(f16(wl.x), layer).cpu().numpy()
    assert_parity(got, ref, "mlp 5120x17408 T=8")


def test_mlp_repeat_deterministic_and_counters_reset(vq3, cfg1):
    wl, blk, layer, ref = cfg1
    ws = vq3.workspace(vq3.mlp_workspace_bytes(8, layer))
    x = f16(wl.x)
    a = vq3.mlp_forward(x, layer, ws=ws).cpu().numpy()
    b = vq3.mlp_forward(x, layer, ws=ws).cpu().numpy()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert_parity(b, ref, "second call")
    assert vq3.workspace_status(ws) == 0


def test_mlp_host_api_equals_device_api(vq3, cfg1):
    wl, blk, layer, ref = cfg1
    ws = vq3.workspace(vq3.mlp_host_workspace_bytes(8, layer))
    got = vq3.mlp_forward_host(wl.x, layer, ws)
    dev = vq3.mlp_forward(f16(wl.x), layer).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), dev.view(np.uint16))


def test_mlp_zero_input_gives_zero(vq3, cfg1):
    wl, blk, layer, ref = cfg1
    got = vq3.mlp_forward(torch.zeros((8, 5120), dtype=torch.float16, device=DEV), layer).cpu().numpy()
    assert not got.any()


def test_mlp_prefill_outliers_T64(vq3):
    wl = S.mlp_prefill_outliers(seed=2, rows=64)
    blk = wl.layers[0]
    assert np.abs(wl.x).max() > 50
    got = vq3.mlp_forward(f16(wl.x), vq3.MLP.from_block(blk, DEV)).cpu().numpy()
    assert_parity(got, O.mlp_f64(wl.x, blk), "mlp T=64 outliers")


@pytest.fixture(scope="module")
def sweep(vq3):
    wl = S.mlp_sweep(seed=4, rows=max(S.SWEEP_ROWS))
    blk = wl.layers[0]
    return wl, blk, vq3.MLP.from_block(blk, DEV), O.mlp_f64(wl.x, blk)


@pytest.mark.parametrize("rows", S.SWEEP_ROWS)
def test_mlp_row_sweep(vq3, sweep, rows):
    wl, blk, layer, ref = sweep
    # the first `rows` rows of the tallest X are the sweep input at that T
    got = vq3.mlp_forward(f16(wl.x[:rows]), layer).cpu().numpy()
    assert_parity(got, ref[:rows], f"sweep T={rows}")


@pytest.mark.parametrize("rows", [17, 40, 65, 129, 300, 1000])
def test_mlp_ragged_prefill_rows(vq3, sweep, rows):
    """Row counts on the tensor-core path that leave a partly filled row tile (64-, 128- and 256-row tiles)."""
    wl, blk, layer, ref = sweep
    got = vq3.mlp_forward(f16(wl.x[:rows]), layer).cpu().numpy()
    assert_parity(got, ref[:rows], f"ragged prefill T={rows}")


def test_mlp_prefill_repeat_bit_identical(vq3, sweep):
    """Split tiles are summed in a fixed order: two calls give the same bits."""
    wl, blk, layer, ref = sweep
    x = f16(wl.x[:512])
    ws = vq3.workspace(vq3.mlp_workspace_bytes(512, layer))
    a = vq3.mlp_forward(x, layer, ws=ws).clone()
    b = vq3.mlp_forward(x, layer, ws=ws)
    assert torch.equal(a, b)
    assert vq3.workspace_status(ws) == 0


def test_workspace_shared_across_row_counts(vq3, sweep):
    """One workspace, sized for the largest call, serves the many-row and the
    few-row path in any order (their counter words sit at the same place)."""
    wl, blk, layer, ref = sweep
    ws = vq3.workspace(max(vq3.mlp_workspace_bytes(r, layer) for r in (8, 32, 2048)))
    for rows in (2048, 8, 64, 16, 32, 2048, 1):
        got = vq3.mlp_forward(f16(wl.x[:rows]), layer, ws=ws).cpu().numpy()
        assert_parity(got, ref[:rows], f"shared workspace T={rows}")
    assert vq3.workspace_status(ws) == 0


def test_mlp_with_seeded_signs(vq3):
    wl = S.mlp_27b(seed=12, rows=8, hidden=1024, inter=2048, block=1024)
    blk = S.add_signs(S.rng(12, 2), wl.layers[0])
    got = vq3.mlp_forward(f16(wl.x), vq3.MLP.from_block(blk, DEV)).cpu().numpy()
    assert_parity(got, O.mlp_f64(wl.x, blk), "mlp signs")


def test_mlp_rows_zero_noop(vq3, cfg1):
    wl, blk, layer, ref = cfg1
    out = torch.full((1, 5120), 7.0, dtype=torch.float16, device=DEV)
    x = torch.zeros((1, 5120), dtype=torch.float16, device=DEV)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(1, layer))
    from ctypes import byref
    rc = vq3.lib.vq3_mlp_forward(x.data_ptr(), 0, byref(layer.struct), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert (out == 7.0).all()


# ------------------------------------------------------------------ residual + RMSNorm and the stack

def test_residual_rmsnorm(vq3):
    r = S.activations(S.rng(7, 0), 8, 5120)
    d = S.activations(S.rng(8, 0), 8, 5120)
    rt, dt = f16(r), f16(d)
    n = vq3.residual_rmsnorm(rt, dt, 1e-6).cpu().numpy()
    r_ref = O.residual_add(r, d)
    assert np.array_equal(rt.cpu().numpy().view(np.uint16), r_ref.view(np.uint16))
    assert f16_ulp_close(n, (r_ref.astype(np.float64) / np.sqrt((r_ref.astype(np.float64) ** 2).mean(1, keepdims=True) + 1e-6)))


def run_stack(vq3, x, layers, eps=1e-6):
    """Config-3 call sequence: for each layer, residual add of the previous output + RMSNorm, then the MLP."""
    resid = f16(x)
    normed = torch.empty_like(resid)
    y = torch.empty_like(resid)
    ws = vq3.workspace(vq3.mlp_workspace_bytes(x.shape[0], layers[0]))
    trace = [resid.cpu().numpy()]
    for i, layer in enumerate(layers):
        vq3.residual_rmsnorm(resid, y if i > 0 else None, eps, normed)
        vq3.mlp_forward(normed, layer, out=y, ws=ws)
        if i > 0:
            trace.append(resid.cpu().numpy())
    vq3.residual_rmsnorm(resid, y, eps, normed)
    trace.append(resid.cpu().numpy())
    return resid.cpu().numpy(), trace


def test_stack_4_layers_full_width(vq3):
    wl = S.mlp_stack(seed=3, rows=8, layers=4)
    layers = [vq3.MLP.from_block(b, DEV) for b in wl.layers]
    got, trace = run_stack(vq3, wl.x, layers)
    otrace = []
    ref = O.stack(wl.x, wl.layers, trace=otrace)
    for li, (g, r) in enumerate(zip(trace, otrace)):
        assert_parity(g, r, f"stack layer {li}")
    assert_parity(got, ref, "stack r_4")
