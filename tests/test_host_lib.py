"""Host side of the C ABI, on CPU: the library loads and exports every
declared entry point, the table build matches the oracle's definition of a
table window, the pack-time encoder writes the oracle's container byte for
byte, and header validation rejects malformed containers.  No CUDA call is
made here (every call below fails or succeeds before touching a device)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads

k3 = pytest.importorskip("lossless_bf16_weight_k3huf_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    k3._build.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "k3huf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(k3huf_\w+)\s*\(", src)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 12
    lib = ctypes.CDLL(k3.library_path())
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(k3.EXPORTS) | set(names)


def test_strerror_and_codes():
    for c in range(0, -9, -1):
        assert k3.strerror(c) != "unknown error"
    assert k3.strerror(-99) == "unknown error"


# --- table build vs the oracle's window decode --------------------------------

def _random_lengths(rng, complete):
    depths = [0]
    k = int(rng.integers(1, 257))
    while len(depths) < k:
        cand = [i for i, d in enumerate(depths) if d < 12]
        if not cand:
            break
        i = cand[int(rng.integers(len(cand)))]
        d = depths.pop(i)
        depths += [d + 1, d + 1]
    if depths == [0]:
        depths = [1]
    if not complete and len(depths) > 1:
        keep = rng.random(len(depths)) > 0.3
        keep[0] = True
        depths = [d for d, x in zip(depths, keep) if x]
    cl = np.zeros(256, dtype=np.uint8)
    cl[rng.choice(256, len(depths), replace=False)] = depths
    return cl


@pytest.mark.parametrize("seed", range(16))
def test_build_table_matches_oracle_windows(seed):
    rng = np.random.default_rng(seed)
    cl = _random_lengths(rng, complete=bool(seed % 2))
    lut = k3.build_table(cl)
    for w in range(4096):
        s, used = oracle.decode_window(cl, w)
        assert int(lut[w]) == ((s << 4) | used if s >= 0 else 0), (w, lut[w], s, used)


@pytest.mark.parametrize("seed", range(200))
def test_table_check_matches_oracle(seed):
    rng = np.random.default_rng(10_000 + seed)
    cl = np.zeros(256, dtype=np.uint8)
    k = int(rng.integers(0, 20))
    cl[rng.choice(256, k, replace=False)] = rng.integers(1, 15, k)
    assert k3.check_table(cl) == oracle.check_codelen(cl)


# --- encoder: byte-identical containers -----------------------------------------

CASES = {
    "tiny": lambda: [workloads.tiny()],
    "n1": lambda: [workloads.normal_tensor((1,), 0.02, 1)],
    "n4095": lambda: [workloads.normal_tensor((4095,), 0.02, 2)],
    "n4097": lambda: [workloads.normal_tensor((4097,), 0.02, 3)],
    "n100003": lambda: [workloads.normal_tensor((100_003,), 0.02, 4)],
    "single": lambda: [workloads.single_symbol(30_001)],
    "two": lambda: [workloads.two_symbol(30_001)],
    "uniform": lambda: [workloads.uniform_bytes(300_000)],
    "heavy": lambda: [workloads.heavy_tail(n=1 << 21)],
    "multi": lambda: [workloads.normal_tensor((64, 96), 0.1, 3, 0), workloads.normal_tensor((5,), 0.3, 3, 1),
                      workloads.normal_tensor((96, 640), 0.04, 3, 2)],
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_encoder_matches_oracle_container(name):
    ts = CASES[name]()
    a = k3.encode_layer(ts, threads=4)
    b = oracle.encode_layer(ts)
    assert a.size == b.size
    assert np.array_equal(a, b)


@pytest.mark.parametrize("chunk_syms,sub_syms", [(1, 512), (7, 512), (1000, 512), (65536, 512), (1 << 21, 512),
                                                (4096, 0), (4096, 256), (4096, 8), (1000, 200), (5000, 1000)])
def test_encoder_chunk_sizes_match_oracle(chunk_syms, sub_syms):
    x = workloads.normal_tensor((300_001,), 0.05, 9)
    assert np.array_equal(k3.encode_layer([x], chunk_syms=chunk_syms, sub_syms=sub_syms, threads=3),
                          oracle.encode_layer([x], chunk_syms=chunk_syms, sub_syms=sub_syms))


def test_encoder_shared_table_matches_oracle():
    ts = CASES["multi"]()
    assert np.array_equal(k3.encode_layer(ts, shared_table=True), oracle.encode_layer(ts, shared_table=True))


def test_encoder_multi_stripe_matches_oracle():
    n = workloads.STRIPE_VALUES if hasattr(workloads, "STRIPE_VALUES") else (1 << 25)
    n += 12_345
    x = np.tile(workloads.tiny(), n // (1 << 21) + 1)[:n]
    a = k3.encode_layer([x])
    b = oracle.encode_layer([x])
    assert np.array_equal(a, b)


def test_encoder_thread_count_independent():
    x = workloads.projection(rows=256, cols=16384)
    ref = k3.encode_layer([x], threads=1)
    for t in (2, 5, 8):
        assert np.array_equal(k3.encode_layer([x], threads=t), ref)


def test_encoder_rejects_empty():
    with pytest.raises(k3.K3HufError):
        k3.encode_layer([np.zeros(0, np.uint16)])


# --- header validation -----------------------------------------------------------

def _blob():
    return k3.encode_layer(CASES["multi"]())


def test_layer_info_fields():
    b = _blob()
    info = k3.layer_info(b)
    ref = oracle.layer_info(b)
    for key in ("chunk_syms", "n_tables", "n_tensors", "n_stripes", "raw_bytes", "blob_bytes", "hdr_bytes", "out_bytes"):
        assert info[key] == ref[key]
    t2 = k3.tensor_info(b, 2)
    assert t2["n_values"] == 96 * 640 and t2["out_offset"] == 12544 and t2["first_stripe"] == 2


@pytest.mark.parametrize("offset,value,code", [
    (0, 0x00, k3.E_FORMAT),          # magic
    (4, 0x02, k3.E_FORMAT),          # version
    (6, 0x0B, k3.E_FORMAT),          # maxlen
    (40, 0x01, k3.E_FORMAT),         # stripe_values
    (64, 0x0D, k3.E_BADLEN),         # a 13-bit length in table 0
])
def test_layer_info_rejects(offset, value, code):
    b = _blob().copy()
    b[offset] = value
    with pytest.raises(k3.K3HufError) as e:
        k3.layer_info(b)
    assert e.value.code == code


def test_layer_info_rejects_oversubscribed_and_empty_tables():
    b = _blob().copy()
    b[64:64 + 256] = 1
    with pytest.raises(k3.K3HufError) as e:
        k3.layer_info(b)
    assert e.value.code == k3.E_OVERSUB
    b[64:64 + 256] = 0
    with pytest.raises(k3.K3HufError) as e:
        k3.layer_info(b)
    assert e.value.code == k3.E_EMPTY


def test_layer_info_rejects_directory_faults():
    good = _blob()
    info = k3.layer_info(good)
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    for off, delta in [(sdir + 0, 16), (sdir + 8, 1 << 40), (sdir + 16, 2), (sdir + 24, 1), (sdir + 32 + 28, 1)]:
        b = good.copy()
        v = int.from_bytes(b[off:off + 8].tobytes(), "little") + delta
        b[off:off + 8] = np.frombuffer((v % (1 << 64)).to_bytes(8, "little"), np.uint8)
        with pytest.raises(k3.K3HufError) as e:
            k3.layer_info(b)
        assert e.value.code in (k3.E_FORMAT, k3.E_ARG), off
    with pytest.raises(k3.K3HufError):
        k3.layer_info(good[:100])                     # shorter than hdr_bytes


def test_decode_argument_checks_need_no_device():
    """Null / misaligned device pointers and bad headers are refused on the
    host before any CUDA call."""
    b = _blob()
    L = k3._lib()
    st = L.k3huf_decode_layer(b.ctypes.data, b.size, None, b.size, 4096, 1 << 20, 4096, None)
    assert st == k3.E_ARG
    st = L.k3huf_decode_layer(b.ctypes.data, b.size, 4096 + 8, b.size, 4096, 1 << 20, 4096, None)
    assert st == k3.E_ARG
    bad = b.copy()
    bad[0] = 0
    st = L.k3huf_decode_layer(bad.ctypes.data, bad.size, 4096, bad.size, 4096, 1 << 20, 4096, None)
    assert st == k3.E_FORMAT
    st = L.k3huf_decode_layer(b.ctypes.data, b.size, 4096, b.size - 1, 4096, 1 << 20, 4096, None)
    assert st == k3.E_ARG                              # device blob shorter than the container
    cl = np.zeros(256, np.uint8)
    st = L.k3huf_decode_stripe(cl.ctypes.data, 4096, 512, 4096, 1 << 20, 100, 4096, 4096, None)
    assert st == k3.E_EMPTY
    # the work-area variant: its own checks first, then the same as above
    ws = L.k3huf_decode_layer_ws
    assert ws(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, None, 68, None) == k3.E_ARG    # no work area
    assert ws(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, 8192, 64, None) == k3.E_ARG   # too short
    assert ws(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, 8194, 68, None) == k3.E_ARG   # unaligned
    assert ws(b.ctypes.data, b.size, 4096 + 8, b.size, 4096, 1 << 20, 4096, 8192, 68, None) == k3.E_ARG
    assert ws(bad.ctypes.data, bad.size, 4096, bad.size, 4096, 1 << 20, 4096, 8192, 68, None) == k3.E_FORMAT
    assert k3.WORK_BYTES == 68
    # the variant with options: flags and (optional) work area checked first
    ex = L.k3huf_decode_layer_ex
    assert ex(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, None, 0, 2, None) == k3.E_ARG    # unknown flag
    assert ex(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, None, 0, 1 << 31, None) == k3.E_ARG
    assert ex(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, 8192, 64, 1, None) == k3.E_ARG   # too short
    assert ex(b.ctypes.data, b.size, 4096, b.size, 4096, 1 << 20, 4096, 8194, 68, 1, None) == k3.E_ARG   # unaligned
    assert ex(b.ctypes.data, b.size, 4096 + 8, b.size, 4096, 1 << 20, 4096, None, 0, 1, None) == k3.E_ARG
    assert ex(bad.ctypes.data, bad.size, 4096, bad.size, 4096, 1 << 20, 4096, None, 0, 1, None) == k3.E_FORMAT
    assert ex(b.ctypes.data, b.size, 4096, b.size - 1, 4096, 1 << 20, 4096, 8192, 68, 0, None) == k3.E_ARG
    assert k3.DECODE_EARLY_START == 1
    # one tensor of the layer: flags, work area, tensor index and its output
    # size are checked before any CUDA call (each case fails before a launch)
    dt = L.k3huf_decode_tensor
    n0 = k3.tensor_info(b, 0)["n_values"]
    assert dt(b.ctypes.data, b.size, 4096, b.size, 0, 4096, 2 * n0, 4096, None, 0, 2, None) == k3.E_ARG      # flag
    assert dt(b.ctypes.data, b.size, 4096, b.size, 0, 4096, 2 * n0, 4096, 8194, 68, 0, None) == k3.E_ARG     # work
    assert dt(b.ctypes.data, b.size, 4096, b.size, 99, 4096, 2 * n0, 4096, None, 0, 0, None) == k3.E_ARG     # tensor
    assert dt(b.ctypes.data, b.size, 4096, b.size, 0, 4096, 2 * n0 - 2, 4096, None, 0, 0, None) == k3.E_ARG  # short
    assert dt(b.ctypes.data, b.size, 4096, b.size, 0, 4104, 2 * n0, 4096, None, 0, 0, None) == k3.E_ARG     # unaligned
    assert dt(bad.ctypes.data, bad.size, 4096, bad.size, 0, 4096, 2 * n0, 4096, None, 0, 0, None) == k3.E_FORMAT
    # the GEMV with options: an unknown flag is refused first
    gx = L.k3huf_gemv_layer_ex
    assert gx(b.ctypes.data, b.size, 4096, b.size, 0, 8192, 4096, 4096, 4096, 4, None) == k3.E_ARG
    assert gx(b.ctypes.data, b.size, 4096, b.size, 0, 8192, 4096, 4096, 4096, 1 << 31, None) == k3.E_ARG
    assert gx(b.ctypes.data, b.size, 4096, b.size, 0, 0, 4096, 4096, 4096, 3, None) == k3.E_ARG   # cols 0
    assert gx(b.ctypes.data, b.size, 4096, b.size, 0, 8192, 4096, 4098, 4096, 3, None) == k3.E_ARG   # y unaligned
    assert k3.GEMV_ZERO_Y == 2
    assert L.k3huf_set_decoder_variant(3) == k3.E_ARG
    assert L.k3huf_set_decoder_variant(-1) == k3.E_ARG


# --- GPU encoder: host-side size query and argument checks (no CUDA call) --------

def test_encode_scratch_bytes():
    small = k3.encode_scratch_bytes([4096])
    big = k3.encode_scratch_bytes([1 << 26])
    assert 0 < small < big
    # per chunk: two u32 words (its bits and its first bit); 2^26 values in 4096-value chunks
    assert big >= 2 * 4 * (1 << 26) // 4096
    assert k3.encode_scratch_bytes([1 << 26], chunk_syms=1024) > big
    assert k3.encode_scratch_bytes([1 << 26], sub_syms=512) == big
    with pytest.raises(k3.K3HufError) as e:
        k3.encode_scratch_bytes([0])
    assert e.value.code == k3.E_ARG


def test_encode_bound_holds_every_container():
    """The bound (every code 12 bits) is at least the CPU encoder's
    container for these values, exceeds it by no more than the bits a
    12-bit code adds per value (plus alignment), and grows with the sizes."""
    cases = [
        [workloads.tiny()],
        [workloads.uniform_bytes(50_000)],
        [workloads.dyadic_long_codes(1 << 16)],
        [workloads.single_symbol(10_000)],
        [workloads.normal_tensor((n,), 0.02, 5) for n in (1, 4095, 4097, 33)],
    ]
    for tensors in cases:
        sizes = [np.asarray(t).size for t in tensors]
        for kw in ({}, {"chunk_syms": 1024, "sub_syms": 128}, {"shared_table": True}):
            blob = k3.encode_layer(tensors, **kw)
            bound = k3.encode_bound(sizes, **kw)
            assert blob.size <= bound <= blob.size + sum(12 * n // 8 + 16 + 256 for n in sizes) + 256
    assert k3.encode_bound([1 << 26]) > k3.encode_bound([1 << 25])
    with pytest.raises(k3.K3HufError) as e:
        k3.encode_bound([0])
    assert e.value.code == k3.E_ARG


def test_encode_gpu_argument_checks_need_no_device():
    """Misaligned pointers and short scratch are refused before any CUDA call."""
    L = k3._lib()
    n = 1000
    nv = (ctypes.c_uint64 * 1)(n)
    need = k3.encode_scratch_bytes([n])
    size = ctypes.c_size_t(0)

    def call(tensor, scratch, scratch_bytes, blob=None):
        ptrs = (ctypes.c_void_p * 1)(tensor)
        return L.k3huf_encode_layer_gpu(1, ptrs, nv, 4096, 256, 0, scratch, scratch_bytes, blob, 0,
                                        ctypes.byref(size), None)
    assert call(1 << 20, (1 << 21) + 8, need) == k3.E_ARG          # scratch not 256-byte aligned
    assert call((1 << 20) + 2, 1 << 21, need) == k3.E_ARG          # tensor not 16-byte aligned
    assert call(1 << 20, 1 << 21, need - 1) == k3.E_ARG            # scratch too small
    assert call(1 << 20, 1 << 21, need, (1 << 22) + 16) == k3.E_ARG  # blob not 256-byte aligned
    assert call(None, 1 << 21, need) == k3.E_ARG
