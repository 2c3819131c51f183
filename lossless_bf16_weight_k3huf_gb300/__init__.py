"""k3huf on GB300: lossless decode of bf16 weights whose high-byte plane is
Huffman coded (canonical, longest-first, 12-bit limit) and whose low-byte
plane is stored raw.

This module is a thin ctypes binding of the C ABI in ``include/k3huf.h``
(``_build/libk3huf.so``, built by ``_build.build()``): it only marshals
arguments.  Every step of the decode runs in the library's CUDA kernels;
there is no CPU fallback -- calls raise when the library is missing.
Device buffers and streams are plain pointers; torch tensors and streams
are accepted and converted with ``data_ptr()`` / ``cuda_stream``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

OK, E_ARG, E_EMPTY, E_OVERSUB, E_BADLEN, E_FORMAT, E_CUDA, E_NOMEM, E_IO = 0, -1, -2, -3, -4, -5, -6, -7, -8
ST_BADCODE, ST_OVERRUN, ST_INDEX, ST_HEADER, ST_TIMEOUT = 1, 2, 4, 8, 16
MAXLEN = 12
STRIPE_VALUES = 1 << 25

EXPORTS = [
    "k3huf_build", "k3huf_layer_info", "k3huf_tensor_info", "k3huf_decode_layer", "k3huf_decode_layer_ws",
    "k3huf_decode_layer_ex", "k3huf_decode_tensor",
    "k3huf_decode_stripe",
    "k3huf_set_decoder_variant", "k3huf_encode_layer", "k3huf_ring_create", "k3huf_ring_run",
    "k3huf_ring_destroy", "k3huf_last_cuda_error", "k3huf_strerror", "k3huf_feed_open", "k3huf_feed_direct",
    "k3huf_feed_read", "k3huf_feed_close", "k3huf_ring_create_staged", "k3huf_ring_run_file",
    "k3huf_encode_scratch_bytes", "k3huf_encode_bound", "k3huf_encode_layer_gpu", "k3huf_gemv_layer",
    "k3huf_gemv_layer_ex", "k3huf_gemv_layer_batch",
]
FILE_ALIGN = 4096


class K3HufError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = _lib().k3huf_strerror(code).decode() if _lib_handle is not None else str(code)
        if code == E_CUDA and _lib_handle is not None:
            msg += f" (cudaError {_lib_handle.k3huf_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{code}]" if what else f"{msg} [{code}]")


class LayerInfo(ctypes.Structure):
    _fields_ = [("chunk_syms", ctypes.c_uint32), ("n_tables", ctypes.c_uint32), ("n_tensors", ctypes.c_uint32),
                ("n_stripes", ctypes.c_uint32), ("raw_bytes", ctypes.c_uint64), ("blob_bytes", ctypes.c_uint64),
                ("out_bytes", ctypes.c_uint64), ("hdr_bytes", ctypes.c_uint32), ("stripe_values", ctypes.c_uint32),
                ("sub_syms", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class TensorInfo(ctypes.Structure):
    _fields_ = [("table", ctypes.c_uint32), ("first_stripe", ctypes.c_uint32), ("n_stripes", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32), ("n_values", ctypes.c_uint64), ("out_offset", ctypes.c_uint64)]


class RingStats(ctypes.Structure):
    _fields_ = [("total_ms", ctypes.c_float), ("decode_ms", ctypes.c_float), ("copy_ms", ctypes.c_float),
                ("h2d_bytes", ctypes.c_uint64), ("out_bytes", ctypes.c_uint64)]


class FeedStats(ctypes.Structure):
    _fields_ = [("total_ms", ctypes.c_float), ("read_ms", ctypes.c_float), ("copy_ms", ctypes.c_float),
                ("decode_ms", ctypes.c_float), ("read_bytes", ctypes.c_uint64), ("out_bytes", ctypes.c_uint64)]


_lib_handle = None
_lock = threading.Lock()
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t


def library_path() -> str:
    return _build.LIB


def _lib():
    """Load the library; raises if it was not built (no fallback)."""
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"k3huf CUDA library not built ({_build.LIB}); run "
                                   "lossless_bf16_weight_k3huf_gb300._build.build()")
            L = ctypes.CDLL(_build.LIB)
            L.k3huf_build.argtypes = [_vp, _vp]
            L.k3huf_layer_info.argtypes = [_vp, _sz, ctypes.POINTER(LayerInfo)]
            L.k3huf_tensor_info.argtypes = [_vp, _sz, ctypes.c_uint32, ctypes.POINTER(TensorInfo)]
            L.k3huf_decode_layer.argtypes = [_vp, _sz, _vp, _sz, _vp, _sz, _vp, _vp]
            L.k3huf_decode_layer_ws.argtypes = [_vp, _sz, _vp, _sz, _vp, _sz, _vp, _vp, _sz, _vp]
            L.k3huf_decode_layer_ex.argtypes = [_vp, _sz, _vp, _sz, _vp, _sz, _vp, _vp, _sz, ctypes.c_uint32, _vp]
            L.k3huf_decode_tensor.argtypes = [_vp, _sz, _vp, _sz, ctypes.c_uint32, _vp, _sz, _vp, _vp, _sz,
                                              ctypes.c_uint32, _vp]
            L.k3huf_decode_stripe.argtypes = [_vp, ctypes.c_uint32, ctypes.c_uint32, _vp, _sz, ctypes.c_uint32, _vp,
                                              _vp, _vp]
            L.k3huf_set_decoder_variant.argtypes = [ctypes.c_int]
            L.k3huf_encode_layer.argtypes = [ctypes.c_uint32, ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_uint64),
                                             ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int, ctypes.c_int, _vp, _sz,
                                             ctypes.POINTER(_sz)]
            L.k3huf_ring_create.argtypes = [_sz, ctypes.c_int, ctypes.POINTER(_vp)]
            L.k3huf_ring_run.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(_vp), ctypes.POINTER(_sz),
                                         ctypes.POINTER(_vp), ctypes.POINTER(_sz), _vp, ctypes.POINTER(RingStats)]
            L.k3huf_ring_destroy.argtypes = [_vp]
            L.k3huf_encode_scratch_bytes.argtypes = [ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint64), ctypes.c_uint32,
                                                     ctypes.c_uint32, ctypes.c_int, ctypes.POINTER(_sz)]
            L.k3huf_encode_bound.argtypes = [ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint64), ctypes.c_uint32,
                                             ctypes.c_uint32, ctypes.c_int, ctypes.POINTER(_sz)]
            L.k3huf_encode_layer_gpu.argtypes = [ctypes.c_uint32, ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_uint64),
                                                 ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int, _vp, _sz, _vp, _sz,
                                                 ctypes.POINTER(_sz), _vp]
            L.k3huf_gemv_layer.argtypes = [_vp, _sz, _vp, _sz, ctypes.c_uint32, ctypes.c_uint64, _vp, _vp, _vp, _vp]
            L.k3huf_gemv_layer_ex.argtypes = [_vp, _sz, _vp, _sz, ctypes.c_uint32, ctypes.c_uint64, _vp, _vp, _vp,
                                              ctypes.c_uint32, _vp]
            L.k3huf_gemv_layer_batch.argtypes = [_vp, _sz, _vp, _sz, ctypes.c_uint32, ctypes.c_uint64, _vp,
                                                 ctypes.c_uint32, _vp, _vp, ctypes.c_uint32, _vp]
            L.k3huf_feed_open.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(_vp)]
            L.k3huf_feed_direct.argtypes = [_vp]
            L.k3huf_feed_read.argtypes = [_vp, ctypes.c_uint64, _sz, _vp, _sz]
            L.k3huf_feed_close.argtypes = [_vp]
            L.k3huf_ring_create_staged.argtypes = [_sz, ctypes.c_int, ctypes.POINTER(_vp)]
            L.k3huf_ring_run_file.argtypes = [_vp, _vp, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                                              ctypes.POINTER(_sz), ctypes.POINTER(_vp), ctypes.POINTER(_sz), _vp,
                                              ctypes.POINTER(FeedStats)]
            L.k3huf_strerror.restype = ctypes.c_char_p
            L.k3huf_strerror.argtypes = [ctypes.c_int]
            _lib_handle = L
    return _lib_handle


def _check(rc: int, what: str):
    if rc != OK:
        raise K3HufError(rc, what)


def _host(a) -> np.ndarray:
    if isinstance(a, (bytes, bytearray, memoryview)):
        return np.frombuffer(a, dtype=np.uint8)
    if hasattr(a, "numpy") and not isinstance(a, np.ndarray):      # torch CPU tensor
        a = a.numpy()
    return np.ascontiguousarray(a).view(np.uint8).reshape(-1)


def _dptr(x) -> int:
    """Device pointer of a CUDA tensor (or an int address)."""
    if isinstance(x, int):
        return x
    if getattr(x, "is_cuda", False):
        return int(x.data_ptr())
    raise TypeError("expected a CUDA tensor or a device address")


def _nbytes(x) -> int:
    if isinstance(x, int):
        raise TypeError("size needed for a raw address")
    return int(x.numel() * x.element_size())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


# ---------------------------------------------------------------------------

def build_table(codelen) -> np.ndarray:
    """The 4096-entry (symbol << 4) | length table of a code-length vector."""
    cl = np.zeros(256, dtype=np.uint8)
    cl[: len(codelen)] = np.asarray(codelen, dtype=np.uint8)
    out = np.zeros(4096, dtype=np.uint16)
    _check(_lib().k3huf_build(cl.ctypes.data, out.ctypes.data), "k3huf_build")
    return out


def check_table(codelen) -> int:
    """Return code of the Kraft check of a code-length vector."""
    cl = np.zeros(256, dtype=np.uint8)
    cl[: len(codelen)] = np.asarray(codelen, dtype=np.uint8)
    return int(_lib().k3huf_build(cl.ctypes.data, None))


def layer_info(hdr) -> dict:
    h = _host(hdr)
    info = LayerInfo()
    _check(_lib().k3huf_layer_info(h.ctypes.data, h.size, ctypes.byref(info)), "k3huf_layer_info")
    return {f: getattr(info, f) for f, _ in LayerInfo._fields_}


def tensor_info(hdr, t: int) -> dict:
    h = _host(hdr)
    ti = TensorInfo()
    _check(_lib().k3huf_tensor_info(h.ctypes.data, h.size, t, ctypes.byref(ti)), "k3huf_tensor_info")
    return {f: getattr(ti, f) for f, _ in TensorInfo._fields_}


def encode_layer(tensors, chunk_syms: int = 4096, shared_table: bool = False, threads: int = 0,
                 out: np.ndarray | None = None, sub_syms: int = 256) -> np.ndarray:
    """Container bytes of a layer of bf16 tensors (numpy uint16 / torch bf16
    CPU); chunk_syms values per indexed chunk, sub_syms per sub-stream."""
    arrs = []
    for t in tensors:
        if hasattr(t, "view") and hasattr(t, "dtype") and str(getattr(t, "dtype", "")) == "torch.bfloat16":
            import torch
            t = t.contiguous().view(torch.int16).numpy().view(np.uint16)
        arrs.append(np.ascontiguousarray(t).reshape(-1).view(np.uint16))
    n = len(arrs)
    ptrs = (_vp * n)(*[a.ctypes.data for a in arrs])
    nv = (ctypes.c_uint64 * n)(*[a.size for a in arrs])
    size = _sz(0)
    L = _lib()
    _check(L.k3huf_encode_layer(n, ptrs, nv, chunk_syms, sub_syms, int(shared_table), threads, None, 0,
                                ctypes.byref(size)), "k3huf_encode_layer")
    if out is None:
        out = np.empty(size.value, dtype=np.uint8)
    elif out.size < size.value:
        raise ValueError("output buffer too small")
    _check(L.k3huf_encode_layer(n, ptrs, nv, chunk_syms, sub_syms, int(shared_table), threads, out.ctypes.data,
                                out.size, ctypes.byref(size)), "k3huf_encode_layer")
    return out[: size.value]


def encode_scratch_bytes(n_values, chunk_syms: int = 4096, sub_syms: int = 256, shared_table: bool = False) -> int:
    """Device scratch bytes that encode_layer_gpu needs for tensors of these sizes."""
    n = len(n_values)
    nv = (ctypes.c_uint64 * n)(*[int(v) for v in n_values])
    out = _sz(0)
    _check(_lib().k3huf_encode_scratch_bytes(n, nv, chunk_syms, sub_syms, int(shared_table), ctypes.byref(out)),
           "k3huf_encode_scratch_bytes")
    return int(out.value)


def encode_bound(sizes, chunk_syms: int = 4096, sub_syms: int = 256, shared_table: bool = False) -> int:
    """Bytes that hold the container of tensors of these sizes whatever their
    values (k3huf_encode_bound)."""
    n = len(sizes)
    nv = (ctypes.c_uint64 * n)(*[int(x) for x in sizes])
    out = _sz(0)
    _check(_lib().k3huf_encode_bound(n, nv, chunk_syms, sub_syms, int(shared_table), ctypes.byref(out)),
           "k3huf_encode_bound")
    return int(out.value)


def encode_layer_gpu(tensors, chunk_syms: int = 4096, sub_syms: int = 256, shared_table: bool = False,
                     stream=None, scratch=None, out=None):
    """Container of a layer of bf16 CUDA tensors (16-byte aligned), built on
    the GPU; returns a CUDA uint8 tensor.  ``scratch`` (a CUDA tensor) is
    allocated here when not given.  ``out``: a CUDA uint8 tensor of at least
    encode_bound(...) bytes, 256-byte aligned; the container is encoded in
    one call into its first bytes and that prefix is returned (without
    ``out``, a first call sizes the container and a second fills a tensor
    of exactly that size)."""
    import torch
    n = len(tensors)
    sizes = [int(t.numel()) for t in tensors]
    dev = tensors[0].device
    if scratch is None:
        scratch = torch.empty(encode_scratch_bytes(sizes, chunk_syms, sub_syms, shared_table), dtype=torch.uint8,
                              device=dev)
    ptrs = (_vp * n)(*[int(t.data_ptr()) for t in tensors])
    nv = (ctypes.c_uint64 * n)(*sizes)
    size = _sz(0)
    L = _lib()
    s = _stream(stream)
    if out is not None:
        _check(L.k3huf_encode_layer_gpu(n, ptrs, nv, chunk_syms, sub_syms, int(shared_table), _dptr(scratch),
                                        _nbytes(scratch), _dptr(out), _nbytes(out), ctypes.byref(size), s),
               "k3huf_encode_layer_gpu")
        return out[: size.value]
    _check(L.k3huf_encode_layer_gpu(n, ptrs, nv, chunk_syms, sub_syms, int(shared_table), _dptr(scratch),
                                    _nbytes(scratch), None, 0, ctypes.byref(size), s), "k3huf_encode_layer_gpu")
    blob = torch.empty(size.value, dtype=torch.uint8, device=dev)
    _check(L.k3huf_encode_layer_gpu(n, ptrs, nv, chunk_syms, sub_syms, int(shared_table), _dptr(scratch),
                                    _nbytes(scratch), _dptr(blob), _nbytes(blob), ctypes.byref(size), s),
           "k3huf_encode_layer_gpu")
    return blob


WORK_BYTES = 68
DECODE_EARLY_START = 1


def decode_layer(hdr, d_layer, d_out, d_status, stream=None, layer_bytes: int | None = None,
                 out_bytes: int | None = None, work=None, early_start: bool = False) -> None:
    """Launch the decode of a layer; asynchronous on ``stream``.  ``work``: a
    zeroed device buffer of at least WORK_BYTES that no other launch uses
    meanwhile (k3huf_decode_layer_ws: the end of the launch is spread over
    all CTAs), or None.  ``early_start`` (k3huf_decode_layer_ex): the launch
    may begin while the kernel before it in the stream finishes; that kernel
    must not write ``d_layer``."""
    h = _host(hdr)
    lb = _nbytes(d_layer) if layer_bytes is None else layer_bytes
    ob = _nbytes(d_out) if out_bytes is None else out_bytes
    if early_start:
        _check(_lib().k3huf_decode_layer_ex(h.ctypes.data, h.size, _dptr(d_layer), lb, _dptr(d_out), ob,
                                            _dptr(d_status), None if work is None else _dptr(work),
                                            0 if work is None else _nbytes(work), DECODE_EARLY_START,
                                            _stream(stream)), "k3huf_decode_layer_ex")
    elif work is None:
        _check(_lib().k3huf_decode_layer(h.ctypes.data, h.size, _dptr(d_layer), lb, _dptr(d_out), ob,
                                         _dptr(d_status), _stream(stream)), "k3huf_decode_layer")
    else:
        _check(_lib().k3huf_decode_layer_ws(h.ctypes.data, h.size, _dptr(d_layer), lb, _dptr(d_out), ob,
                                            _dptr(d_status), _dptr(work), _nbytes(work), _stream(stream)),
               "k3huf_decode_layer_ws")


def decode_tensor(hdr, d_layer, tensor: int, d_out, d_status, stream=None, layer_bytes: int | None = None,
                  out_bytes: int | None = None, work=None, early_start: bool = False) -> None:
    """Launch the decode of one tensor of a layer (k3huf_decode_tensor):
    ``d_out`` receives its bf16 bytes from offset 0.  ``work`` and
    ``early_start`` as for decode_layer."""
    h = _host(hdr)
    lb = _nbytes(d_layer) if layer_bytes is None else layer_bytes
    ob = _nbytes(d_out) if out_bytes is None else out_bytes
    _check(_lib().k3huf_decode_tensor(h.ctypes.data, h.size, _dptr(d_layer), lb, int(tensor), _dptr(d_out), ob,
                                      _dptr(d_status), None if work is None else _dptr(work),
                                      0 if work is None else _nbytes(work),
                                      DECODE_EARLY_START if early_start else 0, _stream(stream)),
           "k3huf_decode_tensor")


GEMV_ZERO_Y = 2


def gemv_layer(hdr, d_layer, tensor: int, cols: int, d_x, d_y, d_status, stream=None,
               layer_bytes: int | None = None, zero_y: bool = False, early_start: bool = False) -> None:
    """y += W x with tensor ``tensor`` of the layer as a row-major matrix of
    ``cols`` columns, decoded on chip (never written out); asynchronous.
    ``zero_y``: y = W x (the call zeroes y first); ``early_start``: the
    call's kernels may begin while the kernel before them finishes, which
    must not write ``d_layer`` (k3huf_gemv_layer_ex)."""
    h = _host(hdr)
    lb = _nbytes(d_layer) if layer_bytes is None else layer_bytes
    flags = (GEMV_ZERO_Y if zero_y else 0) | (DECODE_EARLY_START if early_start else 0)
    if flags:
        _check(_lib().k3huf_gemv_layer_ex(h.ctypes.data, h.size, _dptr(d_layer), lb, tensor, cols, _dptr(d_x),
                                          _dptr(d_y), _dptr(d_status), flags, _stream(stream)), "k3huf_gemv_layer_ex")
        return
    _check(_lib().k3huf_gemv_layer(h.ctypes.data, h.size, _dptr(d_layer), lb, tensor, cols, _dptr(d_x), _dptr(d_y),
                                   _dptr(d_status), _stream(stream)), "k3huf_gemv_layer")


def gemv_layer_batch(hdr, d_layer, tensor: int, cols: int, d_x, d_y, d_status, stream=None,
                     layer_bytes: int | None = None, zero_y: bool = False, early_start: bool = False) -> None:
    """Y += W X for several vectors with one decode of W (k3huf_gemv_layer_batch):
    ``d_x`` a CUDA bf16 tensor of n_vec x cols (n_vec 1, 2, 4 or 8), ``d_y`` a
    CUDA float32 tensor of n_vec x rows; ``zero_y``: Y = W X."""
    h = _host(hdr)
    lb = _nbytes(d_layer) if layer_bytes is None else layer_bytes
    n_vec = _nbytes(d_x) // (2 * cols)
    flags = (GEMV_ZERO_Y if zero_y else 0) | (DECODE_EARLY_START if early_start else 0)
    _check(_lib().k3huf_gemv_layer_batch(h.ctypes.data, h.size, _dptr(d_layer), lb, tensor, cols, _dptr(d_x), n_vec,
                                         _dptr(d_y), _dptr(d_status), flags, _stream(stream)),
           "k3huf_gemv_layer_batch")


def decode_stripe(codelen, chunk_syms: int, sub_syms: int, d_stripe, stripe_bytes: int, n_values: int, d_out,
                  d_status, stream=None) -> None:
    cl = np.zeros(256, dtype=np.uint8)
    cl[: len(codelen)] = np.asarray(codelen, dtype=np.uint8)
    _check(_lib().k3huf_decode_stripe(cl.ctypes.data, chunk_syms, sub_syms, _dptr(d_stripe), stripe_bytes, n_values,
                                      _dptr(d_out), _dptr(d_status), _stream(stream)), "k3huf_decode_stripe")


def set_decoder_variant(variant: int) -> None:
    """Codes per lockstep table lookup: 0 = default (2), 1 or 2."""
    _check(_lib().k3huf_set_decoder_variant(variant), "k3huf_set_decoder_variant")


class Feed:
    """A container file opened for the storage feed (O_DIRECT where the
    filesystem allows it), read with parallel preads."""

    def __init__(self, path: str, threads: int = 8):
        self._h = _vp()
        _check(_lib().k3huf_feed_open(os.fsencode(path), threads, ctypes.byref(self._h)), "k3huf_feed_open")

    @property
    def direct(self) -> bool:
        return _lib().k3huf_feed_direct(self._h) == 1

    def read(self, offset: int, nbytes: int, buf, buf_bytes: int | None = None) -> None:
        """Read into host memory at ``buf`` (an address or a numpy/torch CPU
        buffer); offset and the buffer 4096-byte aligned."""
        if isinstance(buf, int):
            addr, cap = buf, buf_bytes
        elif hasattr(buf, "data_ptr"):
            addr, cap = int(buf.data_ptr()), _nbytes(buf)
        else:
            addr, cap = buf.ctypes.data, buf.nbytes
        _check(_lib().k3huf_feed_read(self._h, offset, nbytes, addr, cap), "k3huf_feed_read")

    def close(self):
        if self._h:
            _lib().k3huf_feed_close(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def aligned_host(nbytes: int, align: int = FILE_ALIGN) -> np.ndarray:
    """A uint8 host array of nbytes whose first byte is align-aligned."""
    raw = np.empty(nbytes + align, dtype=np.uint8)
    off = (-raw.ctypes.data) % align
    return raw[off: off + nbytes]


def write_layers(path: str, blobs) -> list:
    """Write containers back to back into a file, each at a 4096-aligned
    offset; returns the offsets."""
    offs, pos = [], 0
    with open(path, "wb") as f:
        for b in blobs:
            b = _host(b)
            offs.append(pos)
            f.write(b.tobytes())
            pos += b.size
            pad = (-pos) % FILE_ALIGN
            f.write(b"\0" * pad)
            pos += pad
        f.flush()
        os.fsync(f.fileno())
    return offs


class Ring:
    """Pinned-host -> HBM double-buffered feed of layers into the decoder.
    ``staged=True`` also allocates pinned host slots, for ``run_file``."""

    def __init__(self, slot_bytes: int, n_slots: int = 2, staged: bool = False):
        self._h = _vp()
        create = _lib().k3huf_ring_create_staged if staged else _lib().k3huf_ring_create
        _check(create(slot_bytes, n_slots, ctypes.byref(self._h)), "k3huf_ring_create")

    def run_file(self, feed: "Feed", offsets, sizes, d_outs, d_status) -> dict:
        """Decode the containers stored in the feed's file at ``offsets``
        (``sizes`` bytes each) into ``d_outs`` (CUDA tensors)."""
        n = len(offsets)
        op = (ctypes.c_uint64 * n)(*[int(o) for o in offsets])
        sp = (_sz * n)(*[int(x) for x in sizes])
        dp = (_vp * n)(*[_dptr(d) for d in d_outs])
        db = (_sz * n)(*[_nbytes(d) for d in d_outs])
        st = FeedStats()
        _check(_lib().k3huf_ring_run_file(self._h, feed._h, n, op, sp, dp, db, _dptr(d_status), ctypes.byref(st)),
               "k3huf_ring_run_file")
        return {f: getattr(st, f) for f, _ in FeedStats._fields_}

    def run(self, h_layers, d_outs, d_status) -> dict:
        """h_layers: pinned host uint8 tensors (containers); d_outs: CUDA tensors."""
        n = len(h_layers)
        hp = (_vp * n)(*[int(h.data_ptr()) for h in h_layers])
        hb = (_sz * n)(*[_nbytes(h) for h in h_layers])
        dp = (_vp * n)(*[_dptr(d) for d in d_outs])
        db = (_sz * n)(*[_nbytes(d) for d in d_outs])
        st = RingStats()
        _check(_lib().k3huf_ring_run(self._h, n, hp, hb, dp, db, _dptr(d_status), ctypes.byref(st)),
               "k3huf_ring_run")
        return {f: getattr(st, f) for f, _ in RingStats._fields_}

    def close(self):
        if self._h:
            _lib().k3huf_ring_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def last_cuda_error() -> int:
    return int(_lib().k3huf_last_cuda_error())


def strerror(code: int) -> str:
    return _lib().k3huf_strerror(code).decode()
