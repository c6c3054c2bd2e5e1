"""Failure detection of the decode kernel's hand-offs, on the GPU, without a fault.

The kernel's steps hand over through counter words in the workspace, and every
wait on a counter is bounded in time: when it runs out the kernel sets the
workspace status word to 3, every later wait of the launch returns at once, and
the kernel ends. Here the failure is made on the host: the counter words are
preset to 0xFFFFFFFF, so the increments of a launch wrap around and each counter
ends one short of its target. Some wait then runs out (about a second), the call
returns with the status word at 3, the CUDA context stays usable, and after
vq3_workspace_init the same workspace gives the oracle's result again.
(The prefill GEMM's bounded waits are not exercised this way.)"""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vq3_oracle as O  # noqa: E402
from synth import inputs as S  # noqa: E402
from tests.parity import assert_parity  # noqa: E402

pytestmark = pytest.mark.gpu

STATUS_BYTES = 256  # the status word's slot at the start of every workspace


def test_decode_kernel_wait_runs_out_and_workspace_recovers():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3

    rows = 5
    wl = S.mlp_27b(seed=12, rows=rows, hidden=1024, inter=2048, block=1024)
    blk = wl.layers[0]
    layer = vq3.MLP.from_block(blk, "cuda")
    assert vq3.mlp_kernel_launches(rows, layer) == 1  # the decode kernel alone
    x = torch.from_numpy(wl.x).to("cuda")
    stream = torch.cuda.current_stream()
    ws = vq3.workspace(vq3.mlp_workspace_bytes(rows, layer))
    ref = O.mlp_f64(wl.x, blk)

    ws[STATUS_BYTES:].fill_(255)  # counter words (and the scratch after them) all ones
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    vq3.mlp_forward(x, layer, ws=ws)  # the launch itself succeeds
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert vq3.workspace_status(ws) == 3
    assert elapsed < 30.0, elapsed  # the waits gave up in bounded time

    # the context is still usable: other work runs and checks out
    y = torch.arange(16, device="cuda", dtype=torch.float32).sum().item()
    assert y == 120.0

    rc = vq3.lib.vq3_workspace_init(ws.data_ptr(), ws.numel(), stream.cuda_stream)
    assert rc == 0, vq3.lib.vq3_last_error().decode()
    for call in range(2):
        out = vq3.mlp_forward(x, layer, ws=ws)
        torch.cuda.synchronize()
        assert vq3.workspace_status(ws) == 0
        assert_parity(out.cpu().numpy(), ref, f"after recovery, call {call}")
    assert np.isfinite(out.cpu().numpy().astype(np.float64)).all()
