"""The GPU encoder entry point that allocates nothing
(k3huf_encode_layer_gpu_noalloc).  It serves callers that may not allocate
device memory themselves -- a plugin or custom operator whose host framework
owns the GPU's memory and hands it only its inputs and outputs -- by
working in a fixed scratch array inside the library.  Called through the C
ABI, its containers must equal those of the scratch-taking encoder byte for
byte, on two calls in a row (the second call finds the first call's
leftovers in the shared array)."""
import ctypes

import numpy as np
import pytest

import workloads

torch = pytest.importorskip("torch")
k3 = pytest.importorskip("lossless_bf16_weight_k3huf_gb300")


@pytest.fixture(scope="module")
def noalloc():
    k3._build.build()
    f = ctypes.CDLL(k3.library_path()).k3huf_encode_layer_gpu_noalloc
    f.argtypes = [ctypes.c_uint32, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_uint64), ctypes.c_uint32,
                  ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t),
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def encode_noalloc(f, tensors):
    n = len(tensors)
    ptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in tensors])
    nv = (ctypes.c_uint64 * n)(*[t.numel() for t in tensors])
    size = ctypes.c_size_t(0)
    stream = torch.cuda.current_stream().cuda_stream
    assert f(n, ptrs, nv, 4096, 256, 0, None, 0, ctypes.byref(size), stream) == k3.OK
    blob = torch.empty(size.value, dtype=torch.uint8, device="cuda")      # the caller's own output buffer
    assert f(n, ptrs, nv, 4096, 256, 0, blob.data_ptr(), blob.numel(), ctypes.byref(size), stream) == k3.OK
    torch.cuda.synchronize()
    return blob


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
def test_noalloc_encoder_matches_scratch_encoder_on_two_calls(noalloc):
    layers = [[workloads.heavy_tail(n=1 << 20)],
              [workloads.normal_tensor((700, 333), 0.02, 11), workloads.normal_tensor((4097,), 0.5, 12)]]
    for ts in layers:
        d = [torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.int16)).cuda() for x in ts]
        got = encode_noalloc(noalloc, d)
        ref = k3.encode_layer_gpu(d)
        torch.cuda.synchronize()
        assert got.numel() == ref.numel()
        assert torch.equal(got, ref)


def test_noalloc_encoder_refuses_layers_beyond_its_scratch(noalloc):
    """A layer whose scratch exceeds the fixed 32 MiB is refused before any
    CUDA call.  The tensor pointer is a placeholder that must never reach the
    device, so the size is checked first: the call is made only when the
    scratch the layer needs is known to be larger than the fixed array."""
    n = 1 << 35
    assert k3.encode_scratch_bytes([n]) > 32 << 20
    nv = (ctypes.c_uint64 * 1)(n)
    ptrs = (ctypes.c_void_p * 1)(1 << 20)
    size = ctypes.c_size_t(0)
    assert noalloc(1, ptrs, nv, 4096, 256, 0, None, 0, ctypes.byref(size), None) == k3.E_ARG


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
def test_noalloc_encoder_refuses_host_pointers(noalloc):
    """The fixed array used is the current device's copy, so every pointer
    must be device memory of the current device: a host pointer given as
    the tensor, or as the output, is refused before any work is issued."""
    x = np.ascontiguousarray(workloads.normal_tensor((4096,), 0.02, 13)).view(np.int16)
    d = torch.from_numpy(x).cuda()
    size = ctypes.c_size_t(0)
    nv = (ctypes.c_uint64 * 1)(x.size)
    stream = torch.cuda.current_stream().cuda_stream
    host = np.zeros(1 << 16, dtype=np.uint8)
    host_addr = host.ctypes.data + (-host.ctypes.data) % 256
    ptrs = (ctypes.c_void_p * 1)(host.ctypes.data + (-host.ctypes.data) % 16)
    assert noalloc(1, ptrs, nv, 4096, 256, 0, None, 0, ctypes.byref(size), stream) == k3.E_ARG
    ptrs = (ctypes.c_void_p * 1)(d.data_ptr())
    assert noalloc(1, ptrs, nv, 4096, 256, 0, None, 0, ctypes.byref(size), stream) == k3.OK
    assert 0 < size.value <= host.size - 256
    assert noalloc(1, ptrs, nv, 4096, 256, 0, host_addr, size.value, ctypes.byref(size), stream) == k3.E_ARG
    torch.cuda.synchronize()
