"""Python binding of libvq3.so (argument marshalling only).

Every step of the VQ3 MLP path runs in the library's CUDA kernels; this module
only turns torch tensors into raw pointers and streams, and raises on a
non-zero status. PyTorch supplies device memory and streams. Importing this
module fails loudly when the library has not been built: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_size_t, c_uint8, c_void_p

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# VQ3_LIB may name another build of the same library (the bounds-check build, libvq3_bc.so)
LIB_PATH = os.environ.get("VQ3_LIB") or os.path.join(_PKG, "libvq3.so")

VQ3_OK = 0
ERRORS = {-1: "VQ3_EINVAL", -2: "VQ3_EALIGN", -3: "VQ3_EUNSUPPORTED", -4: "VQ3_ECUDA", -5: "VQ3_ENOSPACE"}


class Vq3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class vq3_linear(ctypes.Structure):
    _fields_ = [("d_in", c_int), ("d_out", c_int), ("block", c_int), ("packed", c_void_p),
                ("codebook", c_void_p), ("scales", c_void_p), ("signs", c_void_p), ("format", c_int),
                ("lr_rank", c_int), ("lr_u", c_void_p), ("lr_v", c_void_p)]


# index formats (VQ3_FORMAT_* in vq3.h): name -> (code, index bits, output channels per index)
FORMATS = {"2x64": (0, 6, 2), "2x16": (1, 4, 2), "lut4": (2, 4, 1)}


class vq3_mlp_layer(ctypes.Structure):
    _fields_ = [("gate", vq3_linear), ("up", vq3_linear), ("down", vq3_linear)]


class vq3_blob_view(ctypes.Structure):
    _fields_ = [("d_in", c_int), ("d_out", c_int), ("block", c_int), ("format", c_int), ("lr_rank", c_int),
                ("has_signs", c_int), ("canonical", c_void_p), ("packed", c_void_p), ("scales", c_void_p),
                ("codebook", c_void_p), ("codebook_bytes", c_size_t), ("signs", c_void_p), ("lr_u", c_void_p),
                ("lr_v", c_void_p)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "vq3_packed_bytes": (c_size_t, [c_int, c_int]),
        "vq3_pack_layout": (c_int, [POINTER(c_uint8), c_int, c_int, c_void_p]),
        "vq3_unpack_layout": (c_int, [c_void_p, c_int, c_int, POINTER(c_uint8)]),
        "vq3_packed_bytes_fmt": (c_size_t, [c_int, c_int, c_int]),
        "vq3_pack_layout_fmt": (c_int, [c_int, POINTER(c_uint8), c_int, c_int, c_void_p]),
        "vq3_unpack_layout_fmt": (c_int, [c_int, c_void_p, c_int, c_int, POINTER(c_uint8)]),
        "vq3_blob_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
        "vq3_blob_write": (c_int, [c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                   c_void_p, c_void_p, c_void_p, c_size_t]),
        "vq3_blob_read": (c_int, [c_void_p, c_size_t, POINTER(vq3_blob_view)]),
        "fwht_rotate": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
        "vq3_linear_workspace_bytes": (c_size_t, [c_int, POINTER(vq3_linear)]),
        "vq3_mlp_workspace_bytes": (c_size_t, [c_int, POINTER(vq3_mlp_layer)]),
        "vq3_workspace_init": (c_int, [c_void_p, c_size_t, c_void_p]),
        "vq3_workspace_status": (c_int, [c_void_p, POINTER(c_int), c_void_p]),
        "vq3_linear_forward": (c_int, [c_void_p, c_int, POINTER(vq3_linear), c_void_p, c_void_p, c_size_t, c_void_p]),
        "vq3_mlp_forward": (c_int, [c_void_p, c_int, POINTER(vq3_mlp_layer), c_void_p, c_void_p, c_size_t, c_void_p]),
        "vq3_mlp_kernel_launches": (c_int, [c_int, POINTER(vq3_mlp_layer)]),
        "vq3_linear_kernel_launches": (c_int, [c_int, POINTER(vq3_linear)]),
        "vq3_mlp_host_workspace_bytes": (c_size_t, [c_int, POINTER(vq3_mlp_layer)]),
        "vq3_mlp_forward_host": (c_int, [c_void_p, c_int, POINTER(vq3_mlp_layer), c_void_p, c_void_p, c_size_t,
                                         c_void_p]),
        "vq3_residual_rmsnorm": (c_int, [c_void_p, c_void_p, c_int, c_int, c_float, c_void_p, c_void_p]),
        "vq3_dequant_dense": (c_int, [POINTER(vq3_linear), c_int, c_void_p, c_void_p]),
        "vq3_delta_rule_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                           c_int, c_void_p, c_void_p, c_void_p]),
        "vq3_mlp_forward_residual": (c_int, [c_void_p, c_void_p, c_int, POINTER(vq3_mlp_layer), c_float, c_void_p,
                                             c_void_p, c_void_p, c_size_t, c_void_p]),
        "vq3_mlp_prenorm_step": (c_int, [c_void_p, c_void_p, c_int, POINTER(vq3_mlp_layer), c_float, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
        "vq3_mlp_forward_noalloc": (c_int, [c_void_p, c_int, POINTER(vq3_mlp_layer), c_void_p, c_void_p]),
        "vq3_noalloc_status": (c_int, [POINTER(c_int), c_void_p]),
        "vq3_last_error": (ctypes.c_char_p, []),
        "vq3_version": (ctypes.c_char_p, []),
        "vq3_bounds_check": (c_int, [POINTER(ctypes.c_uint), c_int, c_int]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def _check(rc: int) -> None:
    if rc != VQ3_OK:
        raise Vq3Error(rc, lib.vq3_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def version() -> str:
    return lib.vq3_version().decode()


BOUNDS_FILES = ("decode", "lowrank", "delta", "rotate", "prefill", "prefill_wide")


def bounds_check(reset: bool = True) -> dict[str, tuple[int, int]]:
    """Bounds-check build only: {kernel file: (accesses skipped, site of the first)}.
    Raises Vq3Error (VQ3_EUNSUPPORTED) in the normal build."""
    buf = (ctypes.c_uint * (2 * len(BOUNDS_FILES)))()
    _check(lib.vq3_bounds_check(buf, len(buf), 1 if reset else 0))
    return {name: (int(buf[2 * f]), int(buf[2 * f + 1])) for f, name in enumerate(BOUNDS_FILES)}


# ---------------------------------------------------------------- layout (host)

def packed_bytes(d_in: int, d_out: int, fmt: str = "2x64") -> int:
    return int(lib.vq3_packed_bytes_fmt(FORMATS[fmt][0], d_in, d_out))


def pack_layout(canonical: np.ndarray, d_in: int, d_out: int, fmt: str = "2x64") -> np.ndarray:
    """Canonical little-endian index stream -> GPU layout (host bytes)."""
    src = np.ascontiguousarray(canonical, dtype=np.uint8)
    dst = np.empty(max(packed_bytes(d_in, d_out, fmt), 1), dtype=np.uint8)
    _check(lib.vq3_pack_layout_fmt(FORMATS[fmt][0], src.ctypes.data_as(POINTER(c_uint8)), d_in, d_out,
                                   dst.ctypes.data_as(c_void_p)))
    return dst


def unpack_layout(packed: np.ndarray, d_in: int, d_out: int, fmt: str = "2x64") -> np.ndarray:
    code, nb, vec = FORMATS[fmt]
    src = np.ascontiguousarray(packed, dtype=np.uint8)
    n = (nb * (d_out // vec) * d_in + 7) // 8
    dst = np.empty(n, dtype=np.uint8)
    _check(lib.vq3_unpack_layout_fmt(code, src.ctypes.data_as(c_void_p), d_in, d_out,
                                     dst.ctypes.data_as(POINTER(c_uint8))))
    return dst


# ---------------------------------------------------------------- weights on the device

_FORMAT_NAMES = {v[0]: k for k, v in FORMATS.items()}


def blob_bytes(d_in: int, d_out: int, fmt: str = "2x64", lr_rank: int = 0, has_signs: bool = False) -> int:
    """Size of the packed-weight blob of one matrix (0 if the descriptor is unsupported)."""
    return int(lib.vq3_blob_bytes(d_in, d_out, FORMATS[fmt][0], lr_rank, int(bool(has_signs))))


def _np_ptr(a):
    return None if a is None else a.ctypes.data_as(c_void_p)


def save_blob(m) -> bytes:
    """The packed-weight blob of one matrix (any object with d_in, d_out, block, stream, codebook,
    scales, signs and optionally fmt, lr_u, lr_v), built by vq3_blob_write."""
    fmt = getattr(m, "fmt", "2x64") or "2x64"
    stream = np.ascontiguousarray(m.stream, dtype=np.uint8)
    scales = np.ascontiguousarray(m.scales, dtype=np.float16)
    codebook = np.ascontiguousarray(m.codebook, dtype=np.float16).reshape(-1)
    signs = None if m.signs is None else np.ascontiguousarray(m.signs, dtype=np.uint32)
    lr_u, lr_v = getattr(m, "lr_u", None), getattr(m, "lr_v", None)
    rank = 0
    if lr_u is not None:
        lr_u = np.ascontiguousarray(lr_u, dtype=np.float16)
        lr_v = np.ascontiguousarray(lr_v, dtype=np.float16)
        rank = int(lr_u.shape[1])
    n = blob_bytes(m.d_in, m.d_out, fmt, rank, signs is not None)
    if n == 0:
        raise Vq3Error(-3, f"blob: unsupported matrix {m.d_in} x {m.d_out} ({fmt}, rank {rank})")
    out = np.empty(n, dtype=np.uint8)
    _check(lib.vq3_blob_write(m.d_in, m.d_out, m.block, FORMATS[fmt][0], _np_ptr(stream), _np_ptr(scales),
                              _np_ptr(codebook), _np_ptr(signs), rank, _np_ptr(lr_u), _np_ptr(lr_v),
                              _np_ptr(out), n))
    return out.tobytes()


def load_blob(data: bytes) -> dict:
    """Checks a packed-weight blob (vq3_blob_read) and returns copies of its parts as numpy arrays."""
    buf = np.frombuffer(data, dtype=np.uint8)
    view = vq3_blob_view()
    _check(lib.vq3_blob_read(_np_ptr(buf), buf.size, ctypes.byref(view)))
    base = buf.ctypes.data

    def part(ptr, count, dtype):
        off = ptr - base
        return buf[off:off + count * np.dtype(dtype).itemsize].view(dtype).copy()

    fmt = _FORMAT_NAMES[view.format]
    nbytes = packed_bytes(view.d_in, view.d_out, fmt)
    out = {"d_in": view.d_in, "d_out": view.d_out, "block": view.block, "fmt": fmt,
           "stream": part(view.canonical, nbytes, np.uint8), "packed": part(view.packed, nbytes, np.uint8),
           "scales": part(view.scales, view.d_out, np.float16),
           "codebook": part(view.codebook, view.codebook_bytes // 2, np.float16),
           "signs": part(view.signs, view.d_in // 32, np.uint32) if view.has_signs else None,
           "lr_u": None, "lr_v": None}
    if view.lr_rank:
        out["lr_u"] = part(view.lr_u, view.d_out * view.lr_rank, np.float16).reshape(view.d_out, view.lr_rank)
        out["lr_v"] = part(view.lr_v, view.lr_rank * view.d_in, np.float16).reshape(view.lr_rank, view.d_in)
    return out


class Linear:
    """One VQ3 matrix resident on the GPU (packed indices, codebook, scales, signs)."""

    def __init__(self, d_in, d_out, block, packed: torch.Tensor, codebook: torch.Tensor, scales: torch.Tensor,
                 signs: torch.Tensor | None = None, fmt: str = "2x64", lr_u: torch.Tensor | None = None,
                 lr_v: torch.Tensor | None = None):
        self.d_in, self.d_out, self.block, self.fmt = int(d_in), int(d_out), int(block), fmt
        self.packed, self.codebook, self.scales, self.signs = packed, codebook, scales, signs
        self.lr_u, self.lr_v = lr_u, lr_v
        rank = 0 if lr_u is None else int(lr_u.shape[1])
        self.struct = vq3_linear(self.d_in, self.d_out, self.block, _ptr(packed), _ptr(codebook), _ptr(scales),
                                 _ptr(signs), FORMATS[fmt][0], rank, _ptr(lr_u), _ptr(lr_v))

    @classmethod
    def from_canonical(cls, d_in, d_out, block, stream, codebook, scales, signs=None, device="cuda",
                       fmt: str = "2x64", lr_u=None, lr_v=None):
        packed = torch.from_numpy(pack_layout(stream, d_in, d_out, fmt)).to(device)
        cb = torch.from_numpy(np.ascontiguousarray(codebook, dtype=np.float16).reshape(-1)).to(device)
        sc = torch.from_numpy(np.ascontiguousarray(scales, dtype=np.float16)).to(device)
        sg = None
        if signs is not None:
            sg = torch.from_numpy(np.ascontiguousarray(signs, dtype=np.uint32).view(np.int32)).to(device)
        lu = lv = None
        if lr_u is not None:
            lu = torch.from_numpy(np.ascontiguousarray(lr_u, dtype=np.float16)).to(device)
            lv = torch.from_numpy(np.ascontiguousarray(lr_v, dtype=np.float16)).to(device)
        return cls(d_in, d_out, block, packed, cb, sc, sg, fmt, lu, lv)

    @classmethod
    def from_blob(cls, data: bytes, device="cuda"):
        """From a packed-weight blob (save_blob): its GPU-layout section is copied as it is."""
        b = load_blob(data)
        packed = torch.from_numpy(b["packed"]).to(device)
        cb = torch.from_numpy(b["codebook"]).to(device)
        sc = torch.from_numpy(b["scales"]).to(device)
        sg = None if b["signs"] is None else torch.from_numpy(b["signs"].view(np.int32)).to(device)
        lu = lv = None
        if b["lr_u"] is not None:
            lu = torch.from_numpy(b["lr_u"]).to(device)
            lv = torch.from_numpy(b["lr_v"]).to(device)
        return cls(b["d_in"], b["d_out"], b["block"], packed, cb, sc, sg, b["fmt"], lu, lv)

    @classmethod
    def from_matrix(cls, m, device="cuda"):
        """From any object with d_in, d_out, block, stream, codebook, scales, signs (and fmt) fields."""
        return cls.from_canonical(m.d_in, m.d_out, m.block, m.stream, m.codebook, m.scales, m.signs, device,
                                  getattr(m, "fmt", "2x64") or "2x64", getattr(m, "lr_u", None),
                                  getattr(m, "lr_v", None))


class MLP:
    """One SwiGLU block: gate and up share the input rotation; down has its own."""

    def __init__(self, gate: Linear, up: Linear, down: Linear):
        self.gate, self.up, self.down = gate, up, down
        self.struct = vq3_mlp_layer(gate.struct, up.struct, down.struct)

    @classmethod
    def from_block(cls, blk, device="cuda"):
        gate = Linear.from_matrix(blk.gate, device)
        if blk.up.signs is not None and blk.gate.signs is not None and np.array_equal(blk.up.signs, blk.gate.signs):
            up = Linear.from_canonical(blk.up.d_in, blk.up.d_out, blk.up.block, blk.up.stream, blk.up.codebook,
                                       blk.up.scales, None, device, getattr(blk.up, "fmt", "2x64") or "2x64")
            up.signs = gate.signs
            up.struct.signs = gate.struct.signs
        else:
            up = Linear.from_matrix(blk.up, device)
        down = Linear.from_matrix(blk.down, device)
        return cls(gate, up, down)

    @property
    def hidden(self) -> int:
        return self.gate.d_in


# ---------------------------------------------------------------- workspaces

def linear_workspace_bytes(rows: int, lin: Linear) -> int:
    return int(lib.vq3_linear_workspace_bytes(rows, ctypes.byref(lin.struct)))


def mlp_workspace_bytes(rows: int, layer: MLP) -> int:
    return int(lib.vq3_mlp_workspace_bytes(rows, ctypes.byref(layer.struct)))


def mlp_host_workspace_bytes(rows: int, layer: MLP) -> int:
    return int(lib.vq3_mlp_host_workspace_bytes(rows, ctypes.byref(layer.struct)))


def workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A device buffer of nbytes, zero-filled by the library (counters start at zero)."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _check(lib.vq3_workspace_init(ws.data_ptr(), ws.numel(), _stream(stream)))
    return ws


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """0 unless a kernel's bounded wait ran out while using this workspace."""
    v = c_int(0)
    _check(lib.vq3_workspace_status(ws.data_ptr(), ctypes.byref(v), _stream(stream)))
    return int(v.value)


# ---------------------------------------------------------------- operations

def fwht_rotate(x: torch.Tensor, block: int, signs: torch.Tensor | None = None, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    rows, n = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check(lib.fwht_rotate(x.data_ptr(), rows, n, block, _ptr(signs), out.data_ptr(), _stream(stream)))
    return out


def linear_forward(x: torch.Tensor, lin: Linear, out=None, ws=None, stream=None) -> torch.Tensor:
    rows = x.shape[0]
    if out is None:
        out = torch.empty((rows, lin.d_out), dtype=torch.float16, device=x.device)
    if ws is None:
        ws = workspace(linear_workspace_bytes(rows, lin), x.device, stream)
    _check(lib.vq3_linear_forward(x.data_ptr(), rows, ctypes.byref(lin.struct), out.data_ptr(), ws.data_ptr(),
                                  ws.numel(), _stream(stream)))
    return out


def mlp_forward(x: torch.Tensor, layer: MLP, out=None, ws=None, stream=None) -> torch.Tensor:
    rows = x.shape[0]
    if out is None:
        out = torch.empty((rows, layer.down.d_out), dtype=torch.float16, device=x.device)
    if ws is None:
        ws = workspace(mlp_workspace_bytes(rows, layer), x.device, stream)
    _check(lib.vq3_mlp_forward(x.data_ptr(), rows, ctypes.byref(layer.struct), out.data_ptr(), ws.data_ptr(),
                               ws.numel(), _stream(stream)))
    return out


def mlp_forward_noalloc(x: torch.Tensor, layer: MLP, out=None, stream=None) -> torch.Tensor:
    """The MLP block with its scratch in the library's fixed device array (no workspace)."""
    rows = x.shape[0]
    if out is None:
        out = torch.empty((rows, layer.down.d_out), dtype=torch.float16, device=x.device)
    _check(lib.vq3_mlp_forward_noalloc(x.data_ptr(), rows, ctypes.byref(layer.struct), out.data_ptr(),
                                       _stream(stream)))
    return out


def noalloc_status(stream=None) -> int:
    """Status word of the fixed array: 0, or 3 when a wait in the last no-alloc call gave up."""
    v = c_int(0)
    _check(lib.vq3_noalloc_status(ctypes.byref(v), _stream(stream)))
    return int(v.value)


def mlp_kernel_launches(rows: int, layer: MLP) -> int:
    return int(lib.vq3_mlp_kernel_launches(rows, ctypes.byref(layer.struct)))


def linear_kernel_launches(rows: int, lin: Linear) -> int:
    return int(lib.vq3_linear_kernel_launches(rows, ctypes.byref(lin.struct)))


def mlp_forward_host(x: np.ndarray, layer: MLP, ws: torch.Tensor, out: np.ndarray | None = None,
                     stream=None) -> np.ndarray:
    """Host buffers in and out (the library copies through the workspace and waits)."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    rows = x.shape[0]
    if out is None:
        out = np.empty((rows, layer.down.d_out), dtype=np.float16)
    _check(lib.vq3_mlp_forward_host(x.ctypes.data_as(c_void_p), rows, ctypes.byref(layer.struct),
                                    out.ctypes.data_as(c_void_p), ws.data_ptr(), ws.numel(), _stream(stream)))
    return out


def residual_rmsnorm(resid: torch.Tensor, delta: torch.Tensor | None, eps: float = 1e-6, normed=None,
                     stream=None) -> torch.Tensor:
    rows, n = resid.shape
    if normed is None:
        normed = torch.empty_like(resid)
    _check(lib.vq3_residual_rmsnorm(resid.data_ptr(), _ptr(delta), rows, n, eps, normed.data_ptr(), _stream(stream)))
    return normed


def dequant_dense(lin: Linear, apply_scale: bool, stream=None) -> torch.Tensor:
    w = torch.empty((lin.d_out, lin.d_in), dtype=torch.float16, device=lin.packed.device)
    _check(lib.vq3_dequant_dense(ctypes.byref(lin.struct), 1 if apply_scale else 0, w.data_ptr(), _stream(stream)))
    return w


# ---------------------------------------------------------------- gated delta rule

def delta_rule_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor, alpha: torch.Tensor,
                       state: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """Gated delta-rule token mixer over blocks of 8 tokens; `state` [H, d_k, d_v] FP32 is updated in place."""
    tokens, heads, d_k = q.shape
    d_v = v.shape[2]
    if out is None:
        out = torch.empty((tokens, heads, d_v), dtype=torch.float16, device=q.device)
    _check(lib.vq3_delta_rule_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(), alpha.data_ptr(),
                                      tokens, heads, d_k, d_v, state.data_ptr(), out.data_ptr(), _stream(stream)))
    return out


def mlp_forward_residual(r_in: torch.Tensor, delta: torch.Tensor | None, layer: MLP, r_out: torch.Tensor,
                         out: torch.Tensor, eps: float = 1e-6, ws=None, stream=None) -> torch.Tensor:
    """One pre-norm residual layer: r_out = fp16(r_in + delta); out = MLP(RMSNorm(r_out))."""
    rows = r_in.shape[0]
    if ws is None:
        ws = workspace(mlp_workspace_bytes(rows, layer), r_in.device, stream)
    _check(lib.vq3_mlp_forward_residual(r_in.data_ptr(), _ptr(delta), rows, ctypes.byref(layer.struct), eps,
                                        r_out.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return out


def mlp_prenorm_step(r: torch.Tensor, layer: MLP, out: torch.Tensor, r_next: torch.Tensor,
                     ss: torch.Tensor | None = None, ss_next: torch.Tensor | None = None, eps: float = 1e-6,
                     ws=None, stream=None) -> torch.Tensor:
    """One pre-norm MLP sublayer: out = MLP(RMSNorm(r)), r_next = fp16(r + out); ss / ss_next are the
    rows' FP32 sums of squares per 16 columns ([rows][d / 16]) of r and r_next."""
    rows = r.shape[0]
    if ws is None:
        ws = workspace(mlp_workspace_bytes(rows, layer), r.device, stream)
    _check(lib.vq3_mlp_prenorm_step(r.data_ptr(), _ptr(ss), rows, ctypes.byref(layer.struct), eps, out.data_ptr(),
                                    r_next.data_ptr(), _ptr(ss_next), ws.data_ptr(), ws.numel(), _stream(stream)))
    return r_next
