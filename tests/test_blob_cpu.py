"""Packed-weight blob of one matrix (vq3_blob_write / vq3_blob_read, host only): round trips in
every index format, the header's content hash against the published FNV-1a definition, and every
check of the reader (magic, version, truncation, corrupt contents, a GPU-layout section that is
not the layout of the canonical stream)."""

import struct

import numpy as np
import pytest

pytest.importorskip("torch")

from synth import inputs as S  # noqa: E402

HASH_AT = 8 + 4 + 4 + 5 * 4 + 4 + 8 * 8 + 8 * 8  # header: magic, version, header bytes, 5 ints, flags, offsets, sizes


@pytest.fixture(scope="module")
def vq3():
    from bit_vector_lut_gb300 import vq3 as m
    return m


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit, written from its published definition."""
    h = 0xCBF29CE484222325
    for b in data:
        h = ((h ^ b) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def test_fnv1a64_published_vectors():
    # the reference values published with the FNV definition
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def small(fmt, signs=True, rank=0, seed=0):
    m = S.matrix(S.rng(200 + seed), 256, 128, 256, fmt)
    if signs:
        m.signs = S.sign_bits(S.rng(201 + seed), 256)
    if rank:
        S.add_lowrank(S.rng(202 + seed), m, rank, 0.02)
    return m


@pytest.mark.parametrize("fmt", ["2x64", "2x16", "lut4"])
@pytest.mark.parametrize("signs,rank", [(False, 0), (True, 0), (True, 16)])
def test_round_trip(vq3, fmt, signs, rank):
    m = small(fmt, signs, rank)
    data = vq3.save_blob(m)
    assert len(data) == vq3.blob_bytes(m.d_in, m.d_out, fmt, rank, signs)
    assert data[:8] == b"VQ3BLOB1"
    b = vq3.load_blob(data)
    assert (b["d_in"], b["d_out"], b["block"], b["fmt"]) == (m.d_in, m.d_out, m.block, fmt)
    assert np.array_equal(b["stream"], np.asarray(m.stream, np.uint8))
    assert np.array_equal(b["packed"], vq3.pack_layout(m.stream, m.d_in, m.d_out, fmt))
    assert np.array_equal(b["scales"].view(np.uint16), np.asarray(m.scales, np.float16).view(np.uint16))
    assert np.array_equal(b["codebook"].view(np.uint16),
                          np.asarray(m.codebook, np.float16).reshape(-1).view(np.uint16))
    if signs:
        assert np.array_equal(b["signs"], np.asarray(m.signs, np.uint32))
    else:
        assert b["signs"] is None
    if rank:
        assert np.array_equal(b["lr_u"].view(np.uint16), np.asarray(m.lr_u, np.float16).view(np.uint16))
        assert np.array_equal(b["lr_v"].view(np.uint16), np.asarray(m.lr_v, np.float16).view(np.uint16))
    else:
        assert b["lr_u"] is None and b["lr_v"] is None
    # the header's hash is FNV-1a 64 of everything after the 256-byte header
    (h,) = struct.unpack_from("<Q", data, HASH_AT)
    assert h == fnv1a64(data[256:])
    # deterministic: the same matrix gives the same bytes
    assert vq3.save_blob(m) == data


def test_header_fields(vq3):
    m = small("2x16", True, 8)
    data = vq3.save_blob(m)
    magic, version, hdr, d_in, d_out, block, fmt, rank, flags = struct.unpack_from("<8sII5iI", data, 0)
    assert (magic, version, hdr) == (b"VQ3BLOB1", 1, 256)
    assert (d_in, d_out, block, fmt, rank, flags) == (256, 128, 256, 1, 8, 1)
    offsets = struct.unpack_from("<8Q", data, 40)
    assert all(o % 256 == 0 for o in offsets) and offsets[0] == 256


def rehash(data: bytearray) -> bytearray:
    struct.pack_into("<Q", data, HASH_AT, fnv1a64(bytes(data[256:])))
    return data


def test_reader_checks(vq3):
    m = small("2x64", True, 16)
    data = bytearray(vq3.save_blob(m))
    with pytest.raises(vq3.Vq3Error, match="magic"):
        vq3.load_blob(b"NOTABLOB" + bytes(data[8:]))
    bad = bytearray(data)
    struct.pack_into("<I", bad, 8, 2)
    with pytest.raises(vq3.Vq3Error, match="version"):
        vq3.load_blob(bytes(bad))
    with pytest.raises(vq3.Vq3Error):
        vq3.load_blob(bytes(data[:-1]))
    with pytest.raises(vq3.Vq3Error):
        vq3.load_blob(bytes(data[:100]))
    bad = bytearray(data)
    bad[300] ^= 1  # a payload byte: the hash no longer matches
    with pytest.raises(vq3.Vq3Error, match="hash"):
        vq3.load_blob(bytes(bad))
    # a GPU-layout byte changed and the hash recomputed: the layout check catches it
    packed_at = struct.unpack_from("<8Q", data, 40)[1]
    bad = bytearray(data)
    bad[packed_at + 5] ^= 0x10
    with pytest.raises(vq3.Vq3Error, match="layout"):
        vq3.load_blob(bytes(rehash(bad)))
    # a descriptor the section table does not match (d_out changed, hash recomputed)
    bad = bytearray(data)
    struct.pack_into("<i", bad, 20, 192)
    with pytest.raises(vq3.Vq3Error):
        vq3.load_blob(bytes(rehash(bad)))
    # the untouched blob still reads
    assert vq3.load_blob(bytes(data))["d_out"] == 128


def test_writer_rejects(vq3):
    m = small("2x64", False, 0)
    m.d_out = 100  # not a multiple of 64
    with pytest.raises(vq3.Vq3Error):
        vq3.save_blob(m)
    m = small("2x64", False, 0)
    m.block = 3
    with pytest.raises(vq3.Vq3Error):
        vq3.save_blob(m)
    assert vq3.blob_bytes(256, 128, "2x64", 12, False) == 0  # rank not a multiple of 8
