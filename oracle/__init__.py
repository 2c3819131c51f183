"""CPU oracle of the k3_huf bf16 codec -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never does, and
this package imports nothing from it.

The arithmetic lives in ``k3huf_oracle.c`` (plain C, compiled here with gcc
on first use); this module only marshals arguments.  Method source: the
article "Kimi K3 纯 CPU 推理中的无损 Trunk 压缩：一次被解码速度判死刑的
Huffman 压缩实验", sections 核心思想, 已实现的部分 and 规范码分配与 Kraft 校验.
Every function here is pinned by ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3huf_oracle.c")
_SRC_PS = os.path.join(_HERE, "k3huf_pagestyle.c")     # the article-style decoder (CPU timing only)
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libk3huf_oracle.so")
_lock = threading.Lock()
_lib = None

E_OK, E_ARG, E_EMPTY, E_OVERSUB, E_BADLEN, E_FORMAT = 0, -1, -2, -3, -4, -5
MAXLEN = 12

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_intp = ctypes.POINTER(ctypes.c_int)
_u32p = ctypes.POINTER(ctypes.c_uint32)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no target-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_PS)):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-Wall", "-o", tmp, _SRC, _SRC_PS])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.orc_histogram.argtypes = [_u8p, ctypes.c_uint64, _u64p]
            L.orc_huffman_lengths.argtypes = [_u64p, _intp]
            L.orc_kraft.argtypes = [_intp, ctypes.c_int]
            L.orc_kraft.restype = ctypes.c_uint64
            L.orc_limit_lengths.argtypes = [_u64p, _intp, ctypes.c_int]
            L.orc_code_lengths.argtypes = [_u64p, ctypes.c_int, _intp]
            L.orc_check_codelen.argtypes = [_u8p, ctypes.c_int]
            L.orc_canonical.argtypes = [_intp, ctypes.c_int, _u32p, _u32p, _u32p]
            L.orc_decode_window.argtypes = [_u8p, ctypes.c_int, ctypes.c_uint32, _intp]
            L.orc_encode_layer.argtypes = [ctypes.c_int, ctypes.POINTER(_u8p), _u64p, ctypes.c_uint32,
                                           ctypes.c_uint32, ctypes.c_int, ctypes.c_int, _u8p, ctypes.c_uint64,
                                           _u64p]
            L.orc_layer_info.argtypes = [_u8p, ctypes.c_uint64, _u64p]
            L.orc_decode_stripe_range.argtypes = [_u8p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                                  ctypes.c_uint32, _u8p]
            L.orc_decode_layer.argtypes = [_u8p, ctypes.c_uint64, _u8p]
            L.orc_ps_build.argtypes = [_u8p, ctypes.POINTER(ctypes.c_uint16)]
            L.orc_ps_decode_stripe.argtypes = [_u8p, ctypes.c_uint64, ctypes.c_uint32, _u8p, _u8p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray, t=_u8p):
    return a.ctypes.data_as(t)


def _counts(cnt) -> np.ndarray:
    c = np.zeros(256, dtype=np.uint64)
    cnt = np.asarray(cnt, dtype=np.uint64)
    c[: len(cnt)] = cnt
    return c


def histogram(values: np.ndarray) -> np.ndarray:
    """cnt[256] of the high bytes of little-endian bf16 values (uint16)."""
    v = np.ascontiguousarray(values, dtype=np.uint16)
    cnt = np.zeros(256, dtype=np.uint64)
    lib().orc_histogram(_ptr(v.view(np.uint8)), v.size, _ptr(cnt, _u64p))
    return cnt


def huffman_lengths(cnt) -> np.ndarray:
    """Unconstrained Huffman code lengths (leaf depths) of a 256-symbol histogram."""
    c = _counts(cnt)
    ln = np.zeros(256, dtype=np.intc)
    lib().orc_huffman_lengths(_ptr(c, _u64p), _ptr(ln, _intp))
    return ln


def kraft(lengths, maxlen: int = MAXLEN) -> int:
    ln = np.zeros(256, dtype=np.intc)
    ln[: len(lengths)] = lengths
    return int(lib().orc_kraft(_ptr(ln, _intp), maxlen))


def limit_lengths(cnt, lengths, maxlen: int = MAXLEN) -> np.ndarray:
    c = _counts(cnt)
    ln = np.zeros(256, dtype=np.intc)
    ln[: len(lengths)] = lengths
    lib().orc_limit_lengths(_ptr(c, _u64p), _ptr(ln, _intp), maxlen)
    return ln


def code_lengths(cnt, maxlen: int = MAXLEN) -> np.ndarray:
    """The encoder's lengths: Huffman depths, then the BZip2-style limit."""
    c = _counts(cnt)
    ln = np.zeros(256, dtype=np.intc)
    lib().orc_code_lengths(_ptr(c, _u64p), maxlen, _ptr(ln, _intp))
    return ln


def check_codelen(codelen, maxlen: int = MAXLEN) -> int:
    cl = np.zeros(256, dtype=np.uint8)
    cl[: len(codelen)] = codelen
    return int(lib().orc_check_codelen(_ptr(cl), maxlen))


def canonical(lengths, maxlen: int = MAXLEN):
    """(codes[256], first[33], count[33]) of the longest-first canonical code."""
    ln = np.zeros(256, dtype=np.intc)
    ln[: len(lengths)] = lengths
    count = np.zeros(33, dtype=np.uint32)
    first = np.zeros(33, dtype=np.uint32)
    code = np.zeros(256, dtype=np.uint32)
    lib().orc_canonical(_ptr(ln, _intp), maxlen, _ptr(count, _u32p), _ptr(first, _u32p), _ptr(code, _u32p))
    return code, first, count


def decode_window(codelen, window: int, maxlen: int = MAXLEN):
    """(symbol, length) of the code at the top of a maxlen-bit window, or
    (-1, 0) when no code matches; a table error code (< -1) for a bad table."""
    cl = np.zeros(256, dtype=np.uint8)
    cl[: len(codelen)] = codelen
    used = ctypes.c_int(0)
    s = lib().orc_decode_window(_ptr(cl), maxlen, window, ctypes.byref(used))
    return int(s), int(used.value)


def encode_layer(tensors, chunk_syms: int = 4096, shared_table: bool = False, maxlen: int = MAXLEN,
                 sub_syms: int = 256) -> np.ndarray:
    """Container bytes (uint8) of a layer made of the given bf16 tensors
    (uint16 arrays); sub_syms = values per sub-stream (0: no sub index)."""
    ts = [np.ascontiguousarray(t, dtype=np.uint16).reshape(-1) for t in tensors]
    n = len(ts)
    ptrs = (_u8p * n)(*[_ptr(t.view(np.uint8)) for t in ts])
    nv = np.array([t.size for t in ts], dtype=np.uint64)
    size = ctypes.c_uint64(0)
    rc = lib().orc_encode_layer(n, ptrs, _ptr(nv, _u64p), chunk_syms, sub_syms, int(shared_table), maxlen,
                                None, 0, ctypes.byref(size))
    if rc:
        raise ValueError(f"oracle encode failed: {rc}")
    out = np.zeros(size.value, dtype=np.uint8)
    rc = lib().orc_encode_layer(n, ptrs, _ptr(nv, _u64p), chunk_syms, sub_syms, int(shared_table), maxlen,
                                _ptr(out), out.size, ctypes.byref(size))
    if rc:
        raise ValueError(f"oracle encode failed: {rc}")
    return out


def container_bytes(tensors, chunk_syms: int = 4096, shared_table: bool = False, maxlen: int = MAXLEN,
                    sub_syms: int = 256) -> int:
    """Size in bytes of the container encode_layer would write for these
    tensors: the encoder's sizing pass alone (histograms, code lengths and
    the layout's arithmetic), without packing any bits."""
    ts = [np.ascontiguousarray(t, dtype=np.uint16).reshape(-1) for t in tensors]
    n = len(ts)
    ptrs = (_u8p * n)(*[_ptr(t.view(np.uint8)) for t in ts])
    nv = np.array([t.size for t in ts], dtype=np.uint64)
    size = ctypes.c_uint64(0)
    rc = lib().orc_encode_layer(n, ptrs, _ptr(nv, _u64p), chunk_syms, sub_syms, int(shared_table), maxlen,
                                None, 0, ctypes.byref(size))
    if rc:
        raise ValueError(f"oracle encode failed: {rc}")
    return int(size.value)


def layer_info(blob: np.ndarray) -> dict:
    info = np.zeros(10, dtype=np.uint64)
    rc = lib().orc_layer_info(_ptr(blob), blob.size, _ptr(info, _u64p))
    if rc:
        raise ValueError(f"not a k3huf layer: {rc}")
    keys = ["chunk_syms", "n_tables", "n_tensors", "n_stripes", "raw_bytes", "blob_bytes",
            "hdr_bytes", "out_bytes", "maxlen", "sub_syms"]
    return {k: int(v) for k, v in zip(keys, info)}


def decode_layer(blob: np.ndarray):
    """(rc, output bytes) of the bit-serial decode of a whole layer."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    info = layer_info(blob)
    out = np.zeros(info["out_bytes"], dtype=np.uint8)
    rc = lib().orc_decode_layer(_ptr(blob), blob.size, _ptr(out))
    return int(rc), out


def decode_chunks(blob: np.ndarray, stripe: int, first_chunk: int, n_chunks: int, out: np.ndarray) -> int:
    """Bit-serial decode of chunks [first_chunk, first_chunk+n_chunks) of a
    stripe into ``out`` (a layer-output-sized uint8 buffer); returns rc."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    return int(lib().orc_decode_stripe_range(_ptr(blob), blob.size, stripe, first_chunk, n_chunks, _ptr(out)))


# --- the article-style decoder (k3huf_pagestyle.c): CPU timing beside the oracle ---

def pagestyle_table(codelen) -> np.ndarray:
    """The article-style decoder's 4096-entry table, (symbol << 4) | length
    per 12-bit window, 0 where no code starts."""
    cl = np.ascontiguousarray(codelen, dtype=np.uint8)
    lut = np.zeros(4096, np.uint16)
    rc = lib().orc_ps_build(_ptr(cl), lut.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    if rc:
        raise ValueError(f"orc_ps_build: {rc}")
    return lut


def pagestyle_decode_stripe(blob: np.ndarray, stripe: int, out: np.ndarray, hi: np.ndarray | None = None) -> int:
    """Decode one stripe with the article-style decoder into ``out`` (the
    layer's output buffer); ``hi``: scratch of at least the stripe's value
    count.  Returns 0 or E_FORMAT / E_ARG."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    if hi is None:
        hi = np.empty(1 << 25, np.uint8)
    return int(lib().orc_ps_decode_stripe(_ptr(blob), blob.size, stripe, _ptr(hi), _ptr(out)))


def pagestyle_decode_layer(blob: np.ndarray):
    """(rc, output) of the article-style decoder over every stripe."""
    info = layer_info(blob)
    out = np.zeros(info["out_bytes"], np.uint8)
    hi = np.empty(1 << 25, np.uint8)
    for s in range(info["n_stripes"]):
        rc = pagestyle_decode_stripe(blob, s, out, hi)
        if rc:
            return rc, out
    return 0, out
