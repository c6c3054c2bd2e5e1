"""GPU parity for the gated delta-rule token mixer (blocks of 8 tokens, the
pages' closed-form block inverse; "anemll/anemll-forge-qwen3.8-27B", "Faster
exact graph (previous update)", bullet "Gated DeltaNet") against the
token-by-token FP64 recurrence of oracle/delta_rule.py."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import delta_rule as D  # noqa: E402
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


def run_gpu(vq3, w):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    state = t(w.state)
    out = vq3.delta_rule_forward(t(w.q), t(w.k), t(w.v), t(w.beta), t(w.alpha), state)
    return out.cpu().numpy(), state.cpu().numpy()


def run_oracle(w):
    T, H, _ = w.q.shape
    outs = np.empty((T, H, w.v.shape[2]))
    states = np.empty(w.state.shape)
    for h in range(H):
        o, s = D.recurrent(w.q[:, h].astype(np.float64), w.k[:, h].astype(np.float64), w.v[:, h].astype(np.float64),
                           w.beta[:, h], w.alpha[:, h], w.state[h])
        outs[:, h] = o
        states[h] = s
    return outs, states


@pytest.mark.parametrize("tokens", [1, 8, 13, 64, 136])
@pytest.mark.parametrize("d_k,d_v", [(128, 128), (64, 32), (32, 16), (24, 16)])
def test_delta_rule_matches_recurrence(vq3, tokens, d_k, d_v):
    # d_k a multiple of 16 up to 128: the tensor-core kernel (64 tokens staged at a time, so 136
    # tokens take three chunks); d_k = 24: the CUDA-core kernel
    w = S.delta_rule_inputs(seed=9, tokens=tokens, heads=16, d_k=d_k, d_v=d_v)
    out, state = run_gpu(vq3, w)
    ref_out, ref_state = run_oracle(w)
    assert_parity(out.reshape(-1, d_v), ref_out.reshape(-1, d_v), f"delta out T={tokens}")
    assert_parity(state.reshape(-1, d_v), ref_state.reshape(-1, d_v), f"delta state T={tokens}")


def test_delta_rule_blocks_chain(vq3):
    # two calls of 8 tokens through the state equal one call of 16
    w = S.delta_rule_inputs(seed=10, tokens=16, heads=4, d_k=128, d_v=64)
    out_all, st_all = run_gpu(vq3, w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    state = t(w.state)
    o1 = vq3.delta_rule_forward(t(w.q[:8]), t(w.k[:8]), t(w.v[:8]), t(w.beta[:8]), t(w.alpha[:8]), state)
    o2 = vq3.delta_rule_forward(t(w.q[8:]), t(w.k[8:]), t(w.v[8:]), t(w.beta[8:]), t(w.alpha[8:]), state)
    assert np.array_equal(np.concatenate([o1.cpu().numpy(), o2.cpu().numpy()]).view(np.uint16),
                          out_all.view(np.uint16))
    assert np.array_equal(state.cpu().numpy(), st_all)


def test_delta_rule_deterministic(vq3):
    w = S.delta_rule_inputs(seed=11, tokens=64, heads=8, d_k=128, d_v=128)
    a = run_gpu(vq3, w)
    b = run_gpu(vq3, w)
    assert np.array_equal(a[0].view(np.uint16), b[0].view(np.uint16)) and np.array_equal(a[1], b[1])
