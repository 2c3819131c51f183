"""GPU encoder parity: the container built on the GPU from device tensors
equals the oracle's container byte for byte (integer work: the bar is
bit-exact), over the same cases as the CPU encoder's tests, and decodes back
to the input on the GPU."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
k3 = pytest.importorskip("lossless_bf16_weight_k3huf_gb300")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


@pytest.fixture(scope="module", autouse=True)
def built():
    k3._build.build()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.int16)).cuda()


def gpu_blob(ts, **kw):
    blob = k3.encode_layer_gpu([dev(x) for x in ts], **kw)
    torch.cuda.synchronize()
    return blob.cpu().numpy()


CASES = {
    "tiny": lambda: [workloads.tiny()],
    "n1": lambda: [workloads.normal_tensor((1,), 0.02, 1)],
    "n7": lambda: [workloads.normal_tensor((7,), 0.02, 5)],
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
def test_gpu_encoder_matches_oracle(name):
    ts = CASES[name]()
    assert np.array_equal(gpu_blob(ts), oracle.encode_layer(ts))


@pytest.mark.parametrize("chunk_syms,sub_syms", [(1, 256), (7, 256), (1000, 200), (4096, 0), (4096, 512),
                                                (4096, 8), (65536, 256), (1 << 21, 256), (5000, 1000), (64, 16),
                                                (256, 256), (1024, 256), (2048, 256), (4096, 256)])
def test_gpu_encoder_chunk_sizes(chunk_syms, sub_syms):
    x = workloads.normal_tensor((300_001,), 0.05, 9)
    assert np.array_equal(gpu_blob([x], chunk_syms=chunk_syms, sub_syms=sub_syms),
                          oracle.encode_layer([x], chunk_syms=chunk_syms, sub_syms=sub_syms))


def test_gpu_encoder_shared_table():
    ts = CASES["multi"]()
    assert np.array_equal(gpu_blob(ts, shared_table=True), oracle.encode_layer(ts, shared_table=True))


def test_gpu_encoder_multi_stripe_and_many_tensors():
    n = (1 << 25) + 12_345
    x = np.tile(workloads.tiny(), n // (1 << 21) + 1)[:n]
    assert np.array_equal(gpu_blob([x]), oracle.encode_layer([x]))
    ts = [workloads.normal_tensor((4096 + 17 * i,), 0.02, 500 + i) for i in range(70)]
    assert np.array_equal(gpu_blob(ts), oracle.encode_layer(ts))


def test_gpu_encode_then_gpu_decode():
    x = workloads.projection(rows=512, cols=16384)
    d = dev(x)
    blob = k3.encode_layer_gpu([d])
    info = k3.layer_info(blob.cpu().numpy())
    out = torch.empty(info["out_bytes"], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3.decode_layer(blob[: info["hdr_bytes"]].cpu().numpy(), blob, out, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(out[: 2 * x.size].view(torch.int16), d)


def test_gpu_encoder_scratch_reuse_needs_no_clearing():
    """The scratch is reused uninitialised between calls."""
    a, b = workloads.normal_tensor((50_000,), 0.02, 1), workloads.heavy_tail(n=1 << 18)
    need = max(k3.encode_scratch_bytes([a.size]), k3.encode_scratch_bytes([b.size]))
    scratch = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    for x in (a, b, a):
        got = k3.encode_layer_gpu([dev(x)], scratch=scratch)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), oracle.encode_layer([x]))


@pytest.mark.parametrize("name", ["uniform", "heavy", "multi", "n4097", "single"])
def test_gpu_encoder_one_call_into_bound_buffer(name):
    """One call into a buffer of k3huf_encode_bound bytes filled with a
    sentinel: the container is its prefix, equal to the oracle's, and the
    bytes after it are not written."""
    ts = CASES[name]() + ([workloads.dyadic_long_codes(1 << 16)] if name == "uniform" else [])
    bound = k3.encode_bound([np.asarray(t).size for t in ts])
    buf = torch.full((bound + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    got = k3.encode_layer_gpu([dev(x) for x in ts], out=buf[:bound])
    torch.cuda.synchronize()
    ref = oracle.encode_layer(ts)
    assert got.numel() == ref.size <= bound
    assert np.array_equal(got.cpu().numpy(), ref)
    assert bool((buf[ref.size:] == 0xA5).all())


def test_gpu_encoder_random_layers():
    """40 seeded random layers (alphabet size and skew, 1-4 tensors of
    1-600,000 values, the default layout or another, shared or per-tensor
    tables), each encoded into a buffer filled with garbage: the GPU
    container equals the oracle's byte for byte.  The
    default layout goes through the one-pass packer, whose look-back spans
    up to 147 chunks per stripe here, with ragged last chunks and lanes."""
    rng = np.random.default_rng(4242)
    for case in range(40):
        tensors = []
        for _ in range(int(rng.integers(1, 5))):
            n = int(rng.integers(1, 600_001))
            n_sym = int(rng.integers(1, 257))
            syms = rng.choice(256, size=n_sym, replace=False)
            w = float(rng.uniform(0.05, 1.0)) ** np.arange(n_sym, dtype=np.float64)
            hi = rng.choice(syms, size=n, p=w / w.sum()).astype(np.uint16)
            tensors.append((hi << 8) | rng.integers(0, 256, size=n, dtype=np.uint16))
        kw = {"shared_table": bool(rng.integers(0, 2))}
        if case % 4 == 3:
            kw["chunk_syms"] = int(rng.choice([1024, 2048, 8192]))
        # into a buffer of garbage: every byte of the container is written
        # (no pass zeroes it first on the default layout)
        bound = k3.encode_bound([t.size for t in tensors], **kw)
        buf = torch.full((bound,), 0xA5, dtype=torch.uint8, device="cuda")
        got = k3.encode_layer_gpu([dev(x) for x in tensors], out=buf, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), oracle.encode_layer(tensors, **kw)), case


@pytest.mark.parametrize("chunk_syms", [4096, 1024])
def test_gpu_encoder_short_buffer_writes_nothing(chunk_syms):
    """A buffer one byte shorter than the container: K3HUF_E_ARG, the size
    still reported, and not one byte of the buffer written (with the default
    layout the GPU finds the shortfall, with another the host)."""
    import ctypes
    ts = CASES["multi"]()
    ref = oracle.encode_layer(ts, chunk_syms=chunk_syms)
    d = [dev(x) for x in ts]
    scratch = torch.full((k3.encode_scratch_bytes([t.size for t in ts], chunk_syms=chunk_syms),), 0xA5,
                         dtype=torch.uint8, device="cuda")
    buf = torch.full((ref.size + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    L = k3._lib()
    ptrs = (ctypes.c_void_p * len(d))(*[t.data_ptr() for t in d])
    nv = (ctypes.c_uint64 * len(d))(*[t.numel() for t in d])
    size = ctypes.c_size_t(0)
    rc = L.k3huf_encode_layer_gpu(len(d), ptrs, nv, chunk_syms, 256, 0, scratch.data_ptr(), scratch.numel(),
                                  buf.data_ptr(), ref.size - 1, ctypes.byref(size), None)
    torch.cuda.synchronize()
    assert rc == k3.E_ARG
    assert size.value == ref.size
    assert bool((buf == 0xA5).all())
    # the same scratch, uncleared, then serves a call with room
    rc = L.k3huf_encode_layer_gpu(len(d), ptrs, nv, chunk_syms, 256, 0, scratch.data_ptr(), scratch.numel(),
                                  buf.data_ptr(), buf.numel(), ctypes.byref(size), None)
    torch.cuda.synchronize()
    assert rc == 0 and size.value == ref.size
    assert np.array_equal(buf[: ref.size].cpu().numpy(), ref)


def _with_counts(counts, seed):
    """bf16 values whose high bytes have exactly these counts (symbol s
    `counts[s]` times), shuffled, with random low bytes."""
    rng = np.random.default_rng(seed)
    hi = np.repeat(np.arange(256, dtype=np.uint16), np.asarray(counts, dtype=np.int64))
    rng.shuffle(hi)
    return (hi << 8) | rng.integers(0, 256, size=hi.size, dtype=np.uint16)


def _fib(n):
    a, b, out = 1, 1, []
    for _ in range(n):
        out.append(a)
        a, b = b, a + b
    return out


PLANNER_COUNTS = {
    # Fibonacci counts: a Huffman tree 26 levels deep, cut to 12 bits
    "fibonacci": lambda: [0] * 230 + _fib(26),
    # every symbol equally often: 255 merges, every weight tied
    "all_equal": lambda: [37] * 256,
    # pairs of equal counts doubling: leaves tie with the nodes made from
    # the pairs before them
    "doubling_pairs": lambda: sum(([1 << k, 1 << k] for k in range(12)), []) + [0] * 232,
    # many symbols seen once beside a few heavy ones: the cap lengthens a
    # long run of equal-count codes (ties to the larger symbol)
    "heavy_and_singletons": lambda: [200_000, 150_000, 90_000, 40_000] + [1] * 252,
}


@pytest.mark.parametrize("name", sorted(PLANNER_COUNTS))
@pytest.mark.parametrize("chunk_syms", [4096, 1024])
def test_gpu_encoder_tie_and_limiter_alphabets(name, chunk_syms):
    """Histograms built to exercise the code-length choices: ties between
    leaves, between internal nodes and across the two, a deep tree cut to
    12 bits, and a long run of equal counts for the cap to lengthen.  The
    default layout decides lengths, codes and layout on the GPU, chunk
    size 1024 on the host; both containers equal the oracle's byte for
    byte, alone and as tables of a two-tensor layer."""
    counts = PLANNER_COUNTS[name]()
    x = _with_counts(counts, 7)
    y = _with_counts(list(reversed(counts)), 8)
    for ts in ([x], [x, y]):
        assert np.array_equal(gpu_blob(ts, chunk_syms=chunk_syms), oracle.encode_layer(ts, chunk_syms=chunk_syms))


def test_gpu_encoder_concurrent_host_threads():
    """Two host threads encode at once, each on its own stream with its own
    scratch and output (the call stages its upload and its outcome in a
    pinned buffer of the calling thread): every container equals the
    oracle's."""
    import threading
    layers = [[workloads.normal_tensor((200_003,), 0.02, 40 + i)] for i in range(2)]
    refs = [oracle.encode_layer(ts) for ts in layers]
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            d = [dev(x) for x in layers[i]]
            scratch = torch.empty(k3.encode_scratch_bytes([x.size for x in layers[i]]), dtype=torch.uint8,
                                  device="cuda")
            out = torch.empty(k3.encode_bound([x.size for x in layers[i]]), dtype=torch.uint8, device="cuda")
            torch.cuda.synchronize()
            for _ in range(20):
                got = k3.encode_layer_gpu(d, stream=stream, scratch=scratch, out=out)
                stream.synchronize()
                if not np.array_equal(got.cpu().numpy(), refs[i]):
                    errors.append(i)
                    return
        except Exception as e:          # reported below, with the thread's index
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


@pytest.mark.parametrize("shared_table", [False, True])
def test_gpu_encoder_more_stripes_than_planner_threads(shared_table):
    """300 small tensors make 300 stripes, more than the planner's 256
    threads place in one round, so the stripes' offsets are summed over two
    rounds (and 300 tables are planned by 300 CTAs, or one table over all
    stripes): the container equals the oracle's byte for byte."""
    ts = [workloads.normal_tensor((97 + 31 * i,), 0.01 + 0.001 * (i % 7), 900 + i) for i in range(300)]
    assert np.array_equal(gpu_blob(ts, shared_table=shared_table), oracle.encode_layer(ts, shared_table=shared_table))
