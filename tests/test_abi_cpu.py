"""Host-side checks of the C-ABI library (no GPU): it loads, exports every
symbol include/vq3.h declares, packs the canonical stream losslessly, and
rejects bad arguments with the documented status before touching the GPU."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import vq3_oracle as O
from synth import inputs as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
vq3 = pytest.importorskip("bit_vector_lut_gb300.vq3", reason="libvq3.so not built")


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "vq3.h")).read()
    return re.findall(r"VQ3_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)


def test_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 15
    lib = ctypes.CDLL(vq3.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_version_string():
    assert "sm_103a" in vq3.version()


@pytest.mark.parametrize("d_in,d_out", [(64, 256), (256, 256), (128, 512), (5120, 256)])
def test_pack_roundtrip(d_in, d_out):
    s = S.index_stream(S.rng(d_in + d_out), d_in, d_out)
    p = vq3.pack_layout(s, d_in, d_out)
    assert p.size == vq3.packed_bytes(d_in, d_out) == s.size
    assert np.array_equal(vq3.unpack_layout(p, d_in, d_out), s)


@pytest.mark.parametrize("pattern", ["zeros", "all63", "ramp", "alternate"])
def test_pack_edge_patterns(pattern):
    d_in, d_out = 128, 256
    n = (d_out // 2) * d_in
    idx = {"zeros": np.zeros(n, int), "all63": np.full(n, 63), "ramp": np.arange(n) % 64,
           "alternate": (np.arange(n) % 2) * 63}[pattern]
    s = O.pack_indices(idx)
    p = vq3.pack_layout(s, d_in, d_out)
    assert np.array_equal(vq3.unpack_layout(p, d_in, d_out), s)
    if pattern in ("zeros", "all63"):
        assert np.array_equal(np.unique(p), np.unique(s))


def test_pack_full_size_roundtrip():
    m = S.matrix(S.rng(1), 5120, 17408, 1024)
    p = vq3.pack_layout(m.stream, 5120, 17408)
    assert p.size == 33_423_360
    assert np.array_equal(vq3.unpack_layout(p, 5120, 17408), m.stream)


def test_layout_is_a_permutation_of_index_fields():
    # the GPU layout is a permutation of index positions: a single nonzero index
    # moves to exactly one 6-bit field of the packed buffer
    d_in, d_out = 64, 256
    for (p_, i_) in [(0, 0), (5, 9), (127, 63), (17, 40)]:
        idx = np.zeros((d_out // 2, d_in), int)
        idx[p_, i_] = 0b101101
        pk = vq3.pack_layout(O.pack_indices(idx), d_in, d_out)
        bits = np.unpackbits(pk, bitorder="little")
        assert bits.sum() == 4


def test_sizes_and_unsupported_shapes():
    assert vq3.packed_bytes(5120, 17408) == 33_423_360
    assert vq3.packed_bytes(100, 256) == 0
    assert vq3.packed_bytes(64, 96) == 0
    with pytest.raises(vq3.Vq3Error) as e:
        vq3.pack_layout(np.zeros(10, np.uint8), 100, 64)
    assert e.value.code == -3


def fake_linear(d_in=256, d_out=256, block=256, packed=0x10000, cb=0x20000, sc=0x30000, signs=None):
    return vq3.vq3_linear(d_in, d_out, block, packed, cb, sc, signs)


def test_error_paths_never_launch():
    L = fake_linear()
    lib = vq3.lib
    # rows == 0 is a valid no-op even with fake device pointers
    assert lib.vq3_linear_forward(0x40000, 0, ctypes.byref(L), 0x50000, 0x60000, 1 << 20, None) == 0
    # negative rows
    assert lib.vq3_linear_forward(0x40000, -1, ctypes.byref(L), 0x50000, 0x60000, 1 << 20, None) == -1
    # bad block size
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(fake_linear(block=3)), 0x50000, 0x60000, 1 << 20, None) == -1
    # d_in not a multiple of the block
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(fake_linear(d_in=320, block=256)), 0x50000, 0x60000,
                                  1 << 20, None) == -1
    # unsupported width
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(fake_linear(d_out=96)), 0x50000, 0x60000, 1 << 20,
                                  None) == -3
    # null pointers
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(fake_linear(packed=None)), 0x50000, 0x60000, 1 << 20,
                                  None) == -1
    assert lib.vq3_linear_forward(None, 8, ctypes.byref(L), 0x50000, 0x60000, 1 << 20, None) == -1
    # misaligned packed indices / activations
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(fake_linear(packed=0x10008)), 0x50000, 0x60000,
                                  1 << 20, None) == -2
    assert lib.vq3_linear_forward(0x40004, 8, ctypes.byref(L), 0x50000, 0x60000, 1 << 20, None) == -2
    # workspace too small
    need = lib.vq3_linear_workspace_bytes(8, ctypes.byref(L))
    assert need > 0
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(L), 0x50000, 0x60000, need - 1, None) == -5
    assert "workspace" in lib.vq3_last_error().decode()


def test_mlp_descriptor_checks():
    lib = vq3.lib
    g = fake_linear(256, 512, 256)
    u = fake_linear(256, 512, 256)
    d = fake_linear(512, 256, 256)
    ok = vq3.vq3_mlp_layer(g, u, d)
    assert lib.vq3_mlp_forward(0x40000, 0, ctypes.byref(ok), 0x50000, 0x60000, 1 << 24, None) == 0
    bad_down = vq3.vq3_mlp_layer(g, u, fake_linear(512, 512, 256))
    assert lib.vq3_mlp_forward(0x40000, 8, ctypes.byref(bad_down), 0x50000, 0x60000, 1 << 24, None) == -1
    bad_signs = vq3.vq3_mlp_layer(g, fake_linear(256, 512, 256, signs=0x70000), d)
    assert lib.vq3_mlp_forward(0x40000, 8, ctypes.byref(bad_signs), 0x50000, 0x60000, 1 << 24, None) == -1
    assert lib.vq3_mlp_workspace_bytes(8, ctypes.byref(ok)) > 0
    assert lib.vq3_mlp_host_workspace_bytes(8, ctypes.byref(ok)) > lib.vq3_mlp_workspace_bytes(8, ctypes.byref(ok))


def test_prenorm_step_argument_checks():
    lib = vq3.lib
    L = vq3.vq3_mlp_layer(fake_linear(256, 512, 256), fake_linear(256, 512, 256), fake_linear(512, 256, 256))
    f = lib.vq3_mlp_prenorm_step
    ws = 1 << 24
    # zero rows: nothing to do, no launch
    assert f(0x40000, None, 0, ctypes.byref(L), 1e-6, 0x50000, 0x60000, None, 0x70000, ws, None) == 0
    # bad eps, null r_next, r_next aliasing r, ss_next aliasing ss, out aliasing r
    assert f(0x40000, None, 8, ctypes.byref(L), -1.0, 0x50000, 0x60000, None, 0x70000, ws, None) == -1
    assert f(0x40000, None, 8, ctypes.byref(L), 1e-6, 0x50000, None, None, 0x70000, ws, None) == -1
    assert f(0x40000, None, 8, ctypes.byref(L), 1e-6, 0x50000, 0x40000, None, 0x70000, ws, None) == -1
    assert f(0x40000, 0x80000, 8, ctypes.byref(L), 1e-6, 0x50000, 0x60000, 0x80000, 0x70000, ws, None) == -1
    assert f(0x40000, None, 8, ctypes.byref(L), 1e-6, 0x40000, 0x60000, None, 0x70000, ws, None) == -1
    # misaligned partial sums
    assert f(0x40000, 0x80004, 8, ctypes.byref(L), 1e-6, 0x50000, 0x60000, 0x90000, 0x70000, ws, None) == -2
    assert "16-byte" in lib.vq3_last_error().decode()


def test_fwht_argument_checks():
    lib = vq3.lib
    assert lib.fwht_rotate(0x40000, 0, 1024, 1024, None, 0x50000, None) == 0
    assert lib.fwht_rotate(0x40000, 2, 1000, 1024, None, 0x50000, None) == -1
    assert lib.fwht_rotate(0x40000, 2, 2048, 2048, None, 0x50000, None) == -1
    assert lib.fwht_rotate(0x40002, 2, 1024, 1024, None, 0x50000, None) == -2
    assert lib.vq3_residual_rmsnorm(0x40000, None, 0, 64, 1e-6, 0x50000, None) == 0
    assert lib.vq3_residual_rmsnorm(0x40000, None, 2, 64, -1.0, 0x50000, None) == -1


# ---------------------------------------------------------------- other index formats

@pytest.mark.parametrize("fmt", ["2x16", "lut4"])
@pytest.mark.parametrize("d_in,d_out", [(64, 64), (256, 256), (128, 512), (5120, 256)])
def test_pack_roundtrip_formats(fmt, d_in, d_out):
    s = S.index_stream(S.rng(d_in + d_out + 7), d_in, d_out, fmt)
    p = vq3.pack_layout(s, d_in, d_out, fmt)
    assert p.size == vq3.packed_bytes(d_in, d_out, fmt) == s.size
    assert np.array_equal(vq3.unpack_layout(p, d_in, d_out, fmt), s)


@pytest.mark.parametrize("fmt", ["2x16", "lut4"])
def test_layout_formats_are_permutations_of_index_fields(fmt):
    # a single nonzero four-bit index (0b1011: three set bits) moves to exactly one field
    _, nb, vec = vq3.FORMATS[fmt]
    d_in, d_out = 128, 128
    for (g_, i_) in [(0, 0), (5, 9), (d_out // vec - 1, 127), (17, 40)]:
        idx = np.zeros((d_out // vec, d_in), int)
        idx[g_, i_] = 0b1011
        pk = vq3.pack_layout(O.pack_indices(idx, nb), d_in, d_out, fmt)
        assert np.unpackbits(pk, bitorder="little").sum() == 3
        assert np.array_equal(O.index_matrix(vq3.unpack_layout(pk, d_in, d_out, fmt), d_in, d_out, fmt=fmt), idx)


def test_format_checks():
    lib = vq3.lib
    assert vq3.packed_bytes(5120, 17408, "2x16") == 5120 * 17408 * 2 // 8
    assert vq3.packed_bytes(5120, 17408, "lut4") == 5120 * 17408 * 4 // 8
    assert lib.vq3_packed_bytes_fmt(7, 256, 256) == 0
    dst = np.zeros(1024, np.uint8)
    src = np.zeros(1024, np.uint8)
    rc = lib.vq3_pack_layout_fmt(7, src.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), 64, 64,
                                 dst.ctypes.data_as(ctypes.c_void_p))
    assert rc == -3
    bad = fake_linear()
    bad.format = 7
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(bad), 0x50000, 0x60000, 1 << 24, None) == -3
    g = fake_linear(256, 512, 256)
    u = fake_linear(256, 512, 256)
    d = fake_linear(512, 256, 256)
    d.format = 1
    mixed = vq3.vq3_mlp_layer(g, u, d)
    assert lib.vq3_mlp_forward(0x40000, 8, ctypes.byref(mixed), 0x50000, 0x60000, 1 << 24, None) == -1


def test_lowrank_descriptor_checks():
    lib = vq3.lib
    L = fake_linear()
    L.lr_rank, L.lr_u, L.lr_v = 12, 0x80000, 0x90000
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(L), 0x50000, 0x60000, 1 << 24, None) == -3
    L.lr_rank, L.lr_u, L.lr_v = 64, None, None
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(L), 0x50000, 0x60000, 1 << 24, None) == -1
    L.lr_rank, L.lr_u, L.lr_v = 64, 0x80008, 0x90000
    assert lib.vq3_linear_forward(0x40000, 8, ctypes.byref(L), 0x50000, 0x60000, 1 << 24, None) == -2
    L.lr_u = 0x80000
    assert lib.vq3_linear_workspace_bytes(8, ctypes.byref(L)) > lib.vq3_linear_workspace_bytes(8, ctypes.byref(fake_linear()))
    g = fake_linear(256, 512, 256)
    g.lr_rank, g.lr_u, g.lr_v = 64, 0x80000, 0x90000
    mlp = vq3.vq3_mlp_layer(g, fake_linear(256, 512, 256), fake_linear(512, 256, 256))
    assert lib.vq3_mlp_forward(0x40000, 8, ctypes.byref(mlp), 0x50000, 0x60000, 1 << 24, None) == -3


def test_delta_rule_argument_checks():
    f = vq3.lib.vq3_delta_rule_forward
    p = 0x10000
    assert f(p, p, p, p, p, 8, 4, 100, 64, p, p, None) == -3   # d_k not a multiple of 8
    assert f(p, p, p, p, p, 8, 4, 128, 24, p, p, None) == -3   # d_v not a multiple of 16
    assert f(p, p, p, p, p, 8, 0, 128, 64, p, p, None) == -1   # no heads
    assert f(p, p, p, p, p, 8, 4, 128, 64, None, p, None) == -1
    assert f(None, None, None, None, None, 0, 4, 128, 64, p, None, None) == 0  # zero tokens: nothing to do


def test_bounds_check_unsupported_in_normal_build():
    # the normal build records nothing: the call says so without touching the GPU
    if "bounds-check" in vq3.version():
        pytest.skip("VQ3_LIB selects the bounds-check build")
    with pytest.raises(vq3.Vq3Error, match="VQ3_BOUNDS_CHECK"):
        vq3.bounds_check()


@pytest.mark.parametrize("src", ["rotate.cu", "lowrank.cu", "delta.cu"])
def test_bounds_check_variant_compiles(tmp_path, src):
    # the instrumented form of the smaller kernel files compiles (the whole library is built in
    # that form, and run, by the GPU test)
    from bit_vector_lut_gb300 import build as B
    r = subprocess.run(
        [B.nvcc(), *B.ARCH, *B.NVCC_FLAGS, "-DVQ3_BOUNDS_CHECK", "-c", os.path.join(B.CSRC, src), "-o",
         str(tmp_path / "x.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]


def declarations():
    """{name: (return type, [argument types])} of every VQ3_API function in include/vq3.h."""
    txt = open(os.path.join(ROOT, "include", "vq3.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    out = {}
    for m in re.finditer(r"VQ3_API\s+([\w\s\*]+?)\b(\w+)\s*\(([^)]*)\)\s*;", txt):
        ret, name, args = m.group(1).strip(), m.group(2), " ".join(m.group(3).split())
        types = []
        if args and args != "void":
            for a in args.split(","):
                a = a.strip()
                types.append(a[: len(a) - len(re.search(r"\w+$", a).group(0))].strip() if "*" in a or " " in a else a)
        out[name] = (ret, types)
    return out


def _kind(ctype_name: str) -> str:
    t = ctype_name.replace("const ", "").strip()
    if "*" in t:
        return "ptr"
    return {"int": "int", "size_t": "size", "float": "float", "unsigned": "uint"}[t]


def _ctypes_kind(t) -> str:
    if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int: "int", ctypes.c_size_t: "size", ctypes.c_float: "float", ctypes.c_uint: "uint"}[t]


def test_binding_signatures_match_the_header():
    # every declared call has a binding whose argument and return kinds match the header's
    # (a size_t passed as a 32-bit int, or a dropped argument, would corrupt the call)
    decl = declarations()
    assert len(decl) >= 30
    for name, (ret, args) in decl.items():
        f = getattr(vq3.lib, name)
        assert f.argtypes is not None, f"{name}: no ctypes signature"
        assert [_kind(a) for a in args] == [_ctypes_kind(t) for t in f.argtypes], name
        assert _kind(ret) == _ctypes_kind(f.restype), name
