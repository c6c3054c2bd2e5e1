"""vq3_mlp_forward_noalloc against vq3_mlp_forward, through the C ABI.

The no-alloc entry point exists for callers that cannot call cudaMalloc (a
plugin inside a framework that owns all device memory, a server that reserved
its memory budget up front): it runs the same MLP block with its scratch in a
fixed array inside the library instead of a caller workspace. This file runs
last so that a failure here comes after every other test has run.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from synth import inputs as S  # noqa: E402
from tests.parity import assert_parity  # noqa: E402

pytestmark = pytest.mark.gpu


def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from bit_vector_lut_gb300 import vq3
    f = vq3.lib.vq3_mlp_forward_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(vq3.vq3_mlp_layer), ctypes.c_void_p,
                  ctypes.c_void_p]
    return vq3, f


def test_noalloc_matches_workspace_entry_point_twice():
    vq3, noalloc = _lib()
    dev = torch.device("cuda:0")
    wl = S.mlp_27b(seed=1, rows=8)
    layer = vq3.MLP.from_block(wl.layers[0], dev)
    x = torch.from_numpy(wl.x).to(dev)
    stream = torch.cuda.current_stream(dev)
    ref = vq3.mlp_forward(x, layer, stream=stream).cpu().numpy()
    for call in range(2):
        out = torch.full_like(x, float("nan"))
        rc = noalloc(x.data_ptr(), x.shape[0], ctypes.byref(layer.struct), out.data_ptr(), stream.cuda_stream)
        assert rc == 0, vq3.lib.vq3_last_error().decode()
        torch.cuda.synchronize(dev)
        assert_parity(out.cpu().numpy(), ref, f"no-alloc call {call}")
        # every wait of the call ended in time: the array's status word reads 0
        assert vq3.noalloc_status(stream) == 0


def test_noalloc_allocates_no_device_memory():
    # the point of the entry point: after a first call (which looks up the array's
    # address), a call changes neither the driver's free memory nor torch's pool
    vq3, noalloc = _lib()
    dev = torch.device("cuda:0")
    wl = S.mlp_27b(seed=1, rows=64)
    layer = vq3.MLP.from_block(wl.layers[0], dev)
    x = torch.from_numpy(wl.x).to(dev)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    rc = noalloc(x.data_ptr(), x.shape[0], ctypes.byref(layer.struct), out.data_ptr(), stream.cuda_stream)
    assert rc == 0, vq3.lib.vq3_last_error().decode()
    torch.cuda.synchronize(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    reserved0 = torch.cuda.memory_reserved(dev)
    rc = noalloc(x.data_ptr(), x.shape[0], ctypes.byref(layer.struct), out.data_ptr(), stream.cuda_stream)
    assert rc == 0, vq3.lib.vq3_last_error().decode()
    torch.cuda.synchronize(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert torch.cuda.memory_reserved(dev) == reserved0


def test_noalloc_runs_rows_beyond_one_pass():
    # 64 rows: more rows than the largest pass that fits the fixed array, so several passes
    vq3, noalloc = _lib()
    dev = torch.device("cuda:0")
    wl = S.mlp_prefill_outliers(seed=2, rows=64)
    layer = vq3.MLP.from_block(wl.layers[0], dev)
    x = torch.from_numpy(wl.x).to(dev)
    stream = torch.cuda.current_stream(dev)
    ref = vq3.mlp_forward(x, layer, stream=stream).cpu().numpy()
    out = torch.full_like(x, float("nan"))
    rc = noalloc(x.data_ptr(), x.shape[0], ctypes.byref(layer.struct), out.data_ptr(), stream.cuda_stream)
    assert rc == 0, vq3.lib.vq3_last_error().decode()
    torch.cuda.synchronize(dev)
    assert_parity(out.cpu().numpy(), ref, "no-alloc, 64 rows")


def test_noalloc_narrow_block_uses_32_row_passes():
    # a narrow block fits 32-row passes of the decode kernel: 40 rows = one pass of 32 and one of 8
    from oracle import vq3_oracle as O
    vq3, noalloc = _lib()
    dev = torch.device("cuda:0")
    wl = S.mlp_27b(seed=13, rows=40, hidden=1024, inter=2048, block=1024)
    blk = wl.layers[0]
    layer = vq3.MLP.from_block(blk, dev)
    x = torch.from_numpy(wl.x).to(dev)
    stream = torch.cuda.current_stream(dev)
    out = torch.full_like(x, float("nan"))
    rc = noalloc(x.data_ptr(), x.shape[0], ctypes.byref(layer.struct), out.data_ptr(), stream.cuda_stream)
    assert rc == 0, vq3.lib.vq3_last_error().decode()
    torch.cuda.synchronize(dev)
    assert_parity(out.cpu().numpy(), O.mlp_f64(wl.x, blk), "no-alloc narrow, 40 rows")


def test_noalloc_rejects_widths_beyond_the_fixed_scratch():
    # hidden 16384 / intermediate 262144 needs more than 32 MiB of scratch even in 8-row
    # passes; the call is refused on the host before anything is launched, so the
    # descriptor's device pointers are never read (aligned placeholders)
    vq3, noalloc = _lib()
    H, I = 16384, 262144
    fake = 1 << 20

    def lin(d_in, d_out):
        return vq3.vq3_linear(d_in, d_out, 1024, fake, fake, fake, None)

    layer = vq3.vq3_mlp_layer(lin(H, I), lin(H, I), lin(I, H))
    rows = 8
    cap = 32 * 1024 * 1024
    assert vq3.lib.vq3_mlp_workspace_bytes(rows, ctypes.byref(layer)) > cap
    rc = noalloc(fake, rows, ctypes.byref(layer), fake, None)
    assert rc == -5
    assert "VQ3_NOALLOC_SCRATCH_BYTES" in vq3.lib.vq3_last_error().decode()
