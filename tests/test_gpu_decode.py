"""GPU parity: the CUDA decode (through the C ABI) against the CPU oracle.

Decoding is exact, so the bar is bit-exact bytes: the GPU output equals the
oracle's bit-serial decode of the same container, element by element, and
both equal the original tensor.  Small cases compare whole outputs; the
full-size workloads (launched exactly as the benchmark launches them)
compare every byte with the original tensor and sampled chunks with the
oracle's decode of those chunks."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
k3 = pytest.importorskip("lossless_bf16_weight_k3huf_gb300")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

SENTINEL = 0xA5
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def built():
    k3._build.build()
    yield
    k3.set_decoder_variant(0)


def gpu_decode(blob, variant=0, stream=None, status_init=0):
    """Decode on the GPU; returns (output bytes, status, guard intact)."""
    info = k3.layer_info(blob)
    d_blob = torch.from_numpy(np.ascontiguousarray(blob)).cuda()
    n = info["out_bytes"]
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
    d_out = buf[GUARD:GUARD + n]
    st = torch.full((1,), status_init, dtype=torch.int32, device="cuda")
    k3.set_decoder_variant(variant)
    k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, d_out, st, stream=stream)
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    guard_ok = bool((h[:GUARD] == SENTINEL).all() and (h[GUARD + n:] == SENTINEL).all())
    return h[GUARD:GUARD + n], int(st.item()), guard_ok


def tensor_regions(blob):
    info = k3.layer_info(blob)
    return [k3.tensor_info(blob, t) for t in range(info["n_tensors"])]


def check_parity(tensors, variant=0, **enc):
    blob = oracle.encode_layer(tensors, **enc)
    out, st, guard_ok = gpu_decode(blob, variant)
    assert st == 0 and guard_ok
    rc, ref = oracle.decode_layer(blob)
    assert rc == 0
    covered = np.zeros(out.size, dtype=bool)
    for t, x in zip(tensor_regions(blob), tensors):
        a, b = t["out_offset"], t["out_offset"] + 2 * t["n_values"]
        got = out[a:b]
        assert np.array_equal(got, ref[a:b]), f"first mismatch at byte {int(np.argmax(got != ref[a:b]))}"
        assert np.array_equal(got.view(np.uint16), np.asarray(x, np.uint16).reshape(-1))
        covered[a:b] = True
    assert (out[~covered] == SENTINEL).all()           # alignment gaps untouched
    return blob


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_tiny(variant):
    check_parity([workloads.tiny()], variant)


@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 9, 15, 16, 17, 63, 64, 65, 4095, 4096, 4097, 8191, 12289,
                               128 * 4096 - 1, 128 * 4096 + 1, 100_003])
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_ragged_sizes(n, variant):
    check_parity([workloads.normal_tensor((n,), 0.02, seed=n)], variant)


@pytest.mark.parametrize("chunk_syms,sub_syms", [(1, 0), (7, 0), (8, 0), (64, 0), (256, 0), (1000, 0), (4096, 0),
                                                (65536, 0), (4096, 512), (4096, 256), (4096, 1024), (4096, 8),
                                                (1000, 200), (1000, 8), (4096, 64), (2048, 512), (64, 16)])
def test_chunk_sizes(chunk_syms, sub_syms):
    check_parity([workloads.normal_tensor((70_001,), 0.05, seed=9)], chunk_syms=chunk_syms, sub_syms=sub_syms)


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_degenerate_planes(variant):
    check_parity([workloads.single_symbol(50_001)], variant)
    check_parity([workloads.two_symbol(50_001)], variant)
    check_parity([workloads.uniform_bytes(300_000)], variant)


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_long_code_pairs(variant):
    """One value in 32 carries a 12-bit code, so pairs that miss the lockstep
    window (and pairs of two 12-bit codes, 24 bits) come often, at every
    position of the four-lookup group."""
    x = workloads.dyadic_long_codes((1 << 20) + 4099)
    blob = check_parity([x], variant)
    lens = oracle.code_lengths(oracle.histogram(x))
    assert lens.max() == 12 and (lens == 12).sum() >= 100
    check_parity([x[: 300_001]], variant, sub_syms=64)


def test_work_pool_parity_and_reset():
    """With a work area the last sixteenth of every CTA's items is pooled
    (one pool per run of CTAs ending in one code table, drained by any CTA):
    the output is the same bytes, and the area is zero again after every
    launch, for one table and for several."""
    one = [workloads.normal_tensor((1 << 25,), 0.02, seed=21)]           # 4096 items: ~27 per CTA, one pooled
    several = [workloads.normal_tensor((1 << 24,), 0.02, seed=22), workloads.normal_tensor((1 << 24,), 0.7, seed=24),
               workloads.uniform_bytes(1 << 20, seed=23)]                # pools over three tables
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    for tensors in (one, several):
        blob = oracle.encode_layer(tensors)
        info = k3.layer_info(blob)
        d_blob = torch.from_numpy(blob).cuda()
        ref = torch.from_numpy(oracle.decode_layer(blob)[1]).cuda()
        for _ in range(3):
            d_out = torch.zeros(info["out_bytes"], dtype=torch.uint8, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, d_out, st, work=work)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert torch.equal(d_out, ref)
            assert int(work.abs().sum().item()) == 0


def test_early_start_chain():
    """Decodes launched with early start on one stream, each starting while
    the kernel before it runs: three layers (pooled with a work area, one
    table, and one that spans two launches), twice over.  Either every
    output is filled and every status zeroed first and the six decodes run
    back to back (a decode behind a decode), or each decode comes right
    after the fill of its output and the zeroing of its status (a write
    ahead of the previous kernel's end would be lost).  Every output equals
    the oracle's, every status is zero and the work area is zero again."""
    layers = [
        [workloads.normal_tensor((1 << 24,), 0.02, seed=41), workloads.normal_tensor((1 << 23,), 0.7, seed=42)],
        [workloads.normal_tensor((3 << 20,), 0.05, seed=43)],
        [workloads.normal_tensor((4096 + 17 * i,), 0.02, 600 + i) for i in range(70)],
    ]
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    cases = []
    for tensors in layers:
        blob = oracle.encode_layer(tensors)
        info = k3.layer_info(blob)
        # the decode writes the tensors' bytes only: the alignment gaps
        # between them keep the fill byte
        ref = np.full(info["out_bytes"], SENTINEL, np.uint8)
        dec = oracle.decode_layer(blob)[1]
        for t in tensor_regions(blob):
            a, b = t["out_offset"], t["out_offset"] + 2 * t["n_values"]
            ref[a:b] = dec[a:b]
        cases.append((blob[: info["hdr_bytes"]], torch.from_numpy(blob).cuda(), torch.from_numpy(ref).cuda(),
                      info["out_bytes"]))
    assert k3.layer_info(cases[2][0])["n_stripes"] > 64
    for fill_first in (True, False, True, False):
        outs = [torch.empty(n, dtype=torch.uint8, device="cuda") for _, _, _, n in cases * 2]
        sts = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in outs]
        if fill_first:
            for out, st in zip(outs, sts):
                out.fill_(SENTINEL)
                st.fill_(0)
        for li, ((hdr, d_blob, ref, n), out, st) in enumerate(zip(cases * 2, outs, sts)):
            if not fill_first:
                out.fill_(SENTINEL)
                st.fill_(0)
            k3.decode_layer(hdr, d_blob, out, st, work=work if li % 3 == 0 else None, early_start=True)
        torch.cuda.synchronize()
        for (hdr, d_blob, ref, n), out, st in zip(cases * 2, outs, sts):
            assert int(st.item()) == 0
            assert torch.equal(out, ref)
        assert int(work.abs().sum().item()) == 0


def test_early_start_waits_for_a_reader_of_its_output():
    """A kernel reads a decode's output right before an early-start decode
    of another layer overwrites that buffer: the reader sees the first
    layer's bytes (the decode writes only after the reader has completed)."""
    a = oracle.encode_layer([workloads.normal_tensor((1 << 23,), 0.02, 51)])
    b = oracle.encode_layer([workloads.normal_tensor((1 << 23,), 0.7, 52)])
    ia, ib = k3.layer_info(a), k3.layer_info(b)
    assert ia["out_bytes"] == ib["out_bytes"]
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ref_a = torch.from_numpy(oracle.decode_layer(a)[1]).cuda()
    ref_b = torch.from_numpy(oracle.decode_layer(b)[1]).cuda()
    out = torch.empty(ia["out_bytes"], dtype=torch.uint8, device="cuda")
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    for _ in range(3):
        st = torch.zeros(2, dtype=torch.int32, device="cuda")
        k3.decode_layer(a[: ia["hdr_bytes"]], da, out, st[0:1], work=work, early_start=True)
        seen = out.clone()                                # the reader of layer a's output
        k3.decode_layer(b[: ib["hdr_bytes"]], db, out, st[1:2], work=work, early_start=True)
        torch.cuda.synchronize()
        assert int(st.abs().sum().item()) == 0
        assert torch.equal(seen, ref_a) and torch.equal(out, ref_b)


def test_early_start_device_table_fault():
    """Early start with a device table that does not build: the status bit
    is written after the preceding kernel (the status fill) completes, so
    it is not lost."""
    blob = oracle.encode_layer([workloads.normal_tensor((1 << 22,), 0.02, 44)])
    info = k3.layer_info(blob)
    bad = blob.copy()
    bad[64:64 + 256] = 1
    d_good, d_bad = torch.from_numpy(blob).cuda(), torch.from_numpy(bad).cuda()
    for _ in range(3):
        out = torch.empty(info["out_bytes"], dtype=torch.uint8, device="cuda")
        st0 = torch.empty(1, dtype=torch.int32, device="cuda")
        st1 = torch.empty(1, dtype=torch.int32, device="cuda")
        st0.fill_(0)
        k3.decode_layer(blob[: info["hdr_bytes"]], d_good, out, st0, early_start=True)
        st1.fill_(0)
        k3.decode_layer(blob[: info["hdr_bytes"]], d_bad, out, st1, early_start=True)
        torch.cuda.synchronize()
        assert int(st0.item()) == 0
        assert int(st1.item()) & k3.ST_HEADER


def test_limiter_fired_alphabet():
    x = workloads.heavy_tail(n=1 << 22)
    blob = check_parity([x])
    assert k3.layer_info(blob)["n_tables"] == 1
    assert oracle.huffman_lengths(oracle.histogram(x)).max() > 12


def test_multi_tensor_and_shared_table():
    ts = [workloads.normal_tensor((64, 96), 0.1, 3, 0), workloads.normal_tensor((5,), 0.3, 3, 1),
          workloads.normal_tensor((96, 640), 0.04, 3, 2), workloads.normal_tensor((33,), 0.01, 3, 3)]
    check_parity(ts)
    check_parity(ts, shared_table=True)


def test_multi_stripe_tensor():
    n = (1 << 25) + 5003
    x = np.tile(workloads.tiny(), n // (1 << 21) + 1)[:n]
    blob = check_parity([x])
    assert k3.layer_info(blob)["n_stripes"] == 2


def test_many_stripes_span_launches():
    """More stripes than one launch carries (64): 70 small tensors."""
    ts = [workloads.normal_tensor((4096 + 17 * i,), 0.02, 500 + i) for i in range(70)]
    check_parity(ts)


def test_decode_tensor_alone():
    """k3huf_decode_tensor: every tensor of a layer (one of them two stripes
    long; per-tensor and shared tables) decoded alone into a buffer of its own
    size with guard bytes after it, plainly and with a work area and early
    start back to back: its bytes equal the input and the guard bytes stay.
    A tensor index out of range and a short output are refused."""
    tensors = [workloads.normal_tensor((300, 4097), 0.02, 7),
               workloads.normal_tensor(((1 << 25) + 12_345,), 0.05, 8),
               workloads.uniform_bytes(100_003, seed=9),
               workloads.normal_tensor((5,), 0.3, 10)]
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    for shared in (False, True):
        blob = k3.encode_layer(tensors, shared_table=shared)
        info = k3.layer_info(blob)
        hdr = blob[: info["hdr_bytes"]]
        d_blob = torch.from_numpy(blob).cuda()
        for t, x in enumerate(tensors):
            nb = 2 * x.size
            outs = [torch.full((nb + 256,), SENTINEL, dtype=torch.uint8, device="cuda") for _ in range(2)]
            st = torch.zeros(2, dtype=torch.int32, device="cuda")
            k3.decode_tensor(hdr, d_blob, t, outs[0], st[0:1], out_bytes=nb)
            k3.decode_tensor(hdr, d_blob, t, outs[1], st[1:2], out_bytes=nb, work=work, early_start=True)
            torch.cuda.synchronize()
            assert int(st.abs().sum().item()) == 0, (shared, t)
            want = torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.uint8)).cuda()
            for o in outs:
                assert torch.equal(o[:nb], want), (shared, t)
                assert bool((o[nb:] == SENTINEL).all()), (shared, t)
        assert int(work.abs().sum().item()) == 0
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty(2 * tensors[0].size, dtype=torch.uint8, device="cuda")
        with pytest.raises(k3.K3HufError) as e:
            k3.decode_tensor(hdr, d_blob, len(tensors), out, st)
        assert e.value.code == k3.E_ARG
        with pytest.raises(k3.K3HufError) as e:
            k3.decode_tensor(hdr, d_blob, 0, out, st, out_bytes=2 * tensors[0].size - 16)
        assert e.value.code == k3.E_ARG


def test_decode_stripe_entry():
    n = (1 << 25) + 70_000
    x = np.tile(workloads.tiny(), n // (1 << 21) + 1)[:n]
    blob = k3.encode_layer([x])
    info = k3.layer_info(blob)
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    d_blob = torch.from_numpy(blob).cuda()
    for s in range(2):
        e = sdir + 32 * s
        off = int.from_bytes(blob[e:e + 8].tobytes(), "little")
        sb = int.from_bytes(blob[e + 8:e + 16].tobytes(), "little")
        nv = int.from_bytes(blob[e + 24:e + 28].tobytes(), "little")
        out = torch.zeros(2 * nv, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k3.decode_stripe(blob[64:64 + 256], info["chunk_syms"], info["sub_syms"], d_blob[off:], sb, nv, out, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert np.array_equal(out.cpu().numpy().view(np.uint16), x[s * (1 << 25): s * (1 << 25) + nv])


def test_status_is_or_ed():
    _, st, _ = gpu_decode(oracle.encode_layer([workloads.tiny()]), status_init=0x40)
    assert st == 0x40


def test_on_a_side_stream():
    blob = oracle.encode_layer([workloads.tiny()])
    s = torch.cuda.Stream()
    out, st, ok = gpu_decode(blob, stream=s)
    assert st == 0 and ok
    assert np.array_equal(out.view(np.uint16)[: 1 << 21], workloads.tiny())


# --- corrupt streams: a status bit, never a fault ----------------------------------

def _stripe0(blob):
    info = k3.layer_info(blob)
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    return int.from_bytes(blob[sdir:sdir + 8].tobytes(), "little")


def _decode_device_copy(host_hdr_blob, device_blob):
    info = k3.layer_info(host_hdr_blob)
    d_blob = torch.from_numpy(np.ascontiguousarray(device_blob)).cuda()
    buf = torch.full((info["out_bytes"] + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3.decode_layer(host_hdr_blob[: info["hdr_bytes"]], d_blob, buf[GUARD:GUARD + info["out_bytes"]], st)
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert (h[:GUARD] == SENTINEL).all() and (h[GUARD + info["out_bytes"]:] == SENTINEL).all()
    return int(st.item())


def test_fault_chunk_index():
    blob = oracle.encode_layer([workloads.normal_tensor((20_000,), 0.02, 6)])
    bad = blob.copy()
    o = _stripe0(blob)
    bad[o + 32 + 4] ^= 1                                # chunk 1 starts one bit off
    assert oracle.decode_layer(bad)[0] != 0
    st = _decode_device_copy(blob, bad)
    assert st & k3.ST_INDEX


def test_fault_undecodable_window():
    x = np.array([0x0000, 0x0100, 0x0000, 0x0000] * 3, dtype=np.uint16)
    blob = oracle.encode_layer([x])
    o = _stripe0(blob)
    bits_off = int.from_bytes(blob[o + 24:o + 28].tobytes(), "little")
    # incomplete table {0:1, 1:2}: sym1 = 00, sym0 = 1; 12 symbols = 0,1,0,0 x3
    blob[64 + 1] = 2
    blob[o + 16:o + 24] = np.frombuffer((15).to_bytes(8, "little"), np.uint8)
    blob[o + bits_off:o + bits_off + 2] = [0b10011100, 0b11100110]
    so = o + 32 + 4 * 1                                # sub-stream starts past the end: all at bit 15
    k = int.from_bytes(blob[8:12].tobytes(), "little") // int.from_bytes(blob[56:60].tobytes(), "little") - 1
    blob[so:so + 2 * k] = np.frombuffer(np.full(k, 15, "<u2").tobytes(), np.uint8)
    assert oracle.decode_layer(blob)[0] == 0
    out, st, _ = gpu_decode(blob)
    assert st == 0 and np.array_equal(out[:24].view(np.uint16), x)
    bad = blob.copy()
    bad[o + bits_off] = 0b01011100                     # starts with 01: no code
    assert oracle.decode_layer(bad)[0] != 0
    st = _decode_device_copy(blob, bad)
    assert st & (k3.ST_BADCODE | k3.ST_INDEX)


def test_fault_device_header_mismatch():
    blob = oracle.encode_layer([workloads.normal_tensor((20_000,), 0.02, 7)])
    o = _stripe0(blob)
    for off, val in [(o, 0), (o + 8, 0x21), (o + 12, 9), (o + 28, 0x11)]:
        bad = blob.copy()
        bad[off] = val
        assert _decode_device_copy(blob, bad) & k3.ST_HEADER, off


def test_fault_device_table_oversubscribed():
    blob = oracle.encode_layer([workloads.normal_tensor((20_000,), 0.02, 8)])
    bad = blob.copy()
    bad[64:64 + 256] = 1
    assert _decode_device_copy(blob, bad) & k3.ST_HEADER


@pytest.mark.parametrize("seed", range(4))
def test_fault_random_bitstream(seed):
    blob = oracle.encode_layer([workloads.normal_tensor((50_000,), 0.02, 10 + seed)])
    o = _stripe0(blob)
    bits_off = int.from_bytes(blob[o + 24:o + 28].tobytes(), "little")
    even_off = int.from_bytes(blob[o + 28:o + 32].tobytes(), "little")
    bad = blob.copy()
    rng = np.random.default_rng(seed)
    bad[o + bits_off:o + even_off] = rng.integers(0, 256, even_off - bits_off, dtype=np.uint8)
    assert _decode_device_copy(blob, bad) != 0


def test_fault_random_bitstream_pooled():
    """A corrupt stretch of the bit stream of a layer large enough that every
    CTA pools items (the work-area instantiation): a status bit, the guard
    bytes intact, and the work area zero again after each launch."""
    blob = oracle.encode_layer([workloads.normal_tensor((1 << 25,), 0.02, 31)])
    info = k3.layer_info(blob)
    o = _stripe0(blob)
    bits_off = int.from_bytes(blob[o + 24:o + 28].tobytes(), "little")
    even_off = int.from_bytes(blob[o + 28:o + 32].tobytes(), "little")
    bad = blob.copy()
    rng = np.random.default_rng(31)
    lo = bits_off + (even_off - bits_off) * 15 // 16         # inside the last, pooled, items
    hi = even_off - 64                                        # the stream's padding stays zero
    bad[lo:hi] = rng.integers(0, 256, hi - lo, dtype=np.uint8)
    d_blob = torch.from_numpy(bad).cuda()
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    for _ in range(2):
        buf = torch.full((info["out_bytes"] + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, buf[GUARD:GUARD + info["out_bytes"]], st, work=work)
        torch.cuda.synchronize()
        h = buf.cpu().numpy()
        assert (h[:GUARD] == SENTINEL).all() and (h[GUARD + info["out_bytes"]:] == SENTINEL).all()
        assert int(st.item()) & (k3.ST_BADCODE | k3.ST_INDEX)
        assert int(work.abs().sum().item()) == 0


def test_host_side_errors_raise():
    blob = oracle.encode_layer([workloads.tiny()])
    info = k3.layer_info(blob)
    d_blob = torch.from_numpy(blob).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    small = torch.zeros(info["out_bytes"] - 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(k3.K3HufError):
        k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, small, st)
    out = torch.zeros(info["out_bytes"] + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(k3.K3HufError):
        k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, out[1:], st, out_bytes=info["out_bytes"])


# --- streaming ring ------------------------------------------------------------------

def test_ring_small_layers():
    layers = [[workloads.normal_tensor((3000 + i, 64), 0.05, 40 + i)] for i in range(5)]
    layers.append([workloads.normal_tensor((7,), 0.3, 99), workloads.normal_tensor((4097,), 0.02, 98)])
    blobs = [k3.encode_layer(ts) for ts in layers]
    h = [torch.from_numpy(b).pin_memory() for b in blobs]
    outs = [torch.zeros(k3.layer_info(b)["out_bytes"], dtype=torch.uint8, device="cuda") for b in blobs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ring = k3.Ring(max(b.size for b in blobs), 2)
    stats = ring.run(h, outs, st)
    ring.close()
    assert st.item() == 0
    assert stats["h2d_bytes"] == sum(b.size for b in blobs)
    for ts, b, o in zip(layers, blobs, outs):
        oc = o.cpu().numpy()
        for t, x in zip(tensor_regions(b), ts):
            a = t["out_offset"]
            assert np.array_equal(oc[a:a + 2 * t["n_values"]].view(np.uint16), x.reshape(-1))


def test_ring_from_file(tmp_path):
    """Storage feed: containers written to a file are read back through the
    staged ring (more layers than slots) and decode to the oracle's bytes."""
    layers = [[workloads.normal_tensor((2000 + 13 * i, 64), 0.05, 60 + i)] for i in range(4)]
    layers.append([workloads.normal_tensor((5,), 0.3, 70), workloads.normal_tensor((4097,), 0.02, 71)])
    blobs = [oracle.encode_layer(ts) for ts in layers]
    path = str(tmp_path / "layers.bin")
    offs = k3.write_layers(path, blobs)
    feed = k3.Feed(path, threads=3)
    ring = k3.Ring(max(b.size for b in blobs), 2, staged=True)
    outs = [torch.full((k3.layer_info(b)["out_bytes"],), SENTINEL, dtype=torch.uint8, device="cuda") for b in blobs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = ring.run_file(feed, offs, [b.size for b in blobs], outs, st)
    ring.close()
    feed.close()
    assert st.item() == 0
    assert stats["read_bytes"] == sum(b.size for b in blobs)
    assert stats["out_bytes"] == sum(k3.layer_info(b)["raw_bytes"] for b in blobs)
    for ts, b, o in zip(layers, blobs, outs):
        rc, ref = oracle.decode_layer(b)
        assert rc == 0
        oc = o.cpu().numpy()
        for t, x in zip(tensor_regions(b), ts):
            a0, a1 = t["out_offset"], t["out_offset"] + 2 * t["n_values"]
            assert np.array_equal(oc[a0:a1], ref[a0:a1])
            assert np.array_equal(oc[a0:a1].view(np.uint16), x.reshape(-1))


def test_ring_from_file_needs_staged_ring(tmp_path):
    blob = oracle.encode_layer([workloads.tiny()])
    path = str(tmp_path / "one.bin")
    offs = k3.write_layers(path, [blob])
    feed = k3.Feed(path)
    ring = k3.Ring(blob.size, 2)
    out = torch.empty(k3.layer_info(blob)["out_bytes"], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(k3.K3HufError) as e:
        ring.run_file(feed, offs, [blob.size], [out], st)
    assert e.value.code == k3.E_ARG
    ring.close()
    feed.close()


# --- full-size workloads, launched as the benchmark launches them -------------------

def _sampled_parity(blob, tensors, out_dev, n_sample=24, seed=0):
    """Every output byte equals the original tensor (checked on the GPU);
    sampled chunks equal the oracle's bit-serial decode of those chunks."""
    info = k3.layer_info(blob)
    regions = tensor_regions(blob)
    for t, x in zip(regions, tensors):
        a = t["out_offset"]
        ref = torch.from_numpy(np.asarray(x, np.uint16).reshape(-1).view(np.int16)).cuda()
        got = out_dev[a:a + 2 * t["n_values"]].view(torch.int16)
        assert torch.equal(got, ref)
        del ref
    out_host = None
    rng = np.random.default_rng(seed)
    cs = info["chunk_syms"]
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    for s in range(info["n_stripes"]):
        e = sdir + 32 * s
        nv = int.from_bytes(blob[e + 24:e + 28].tobytes(), "little")
        sout = int.from_bytes(blob[e + 16:e + 24].tobytes(), "little")
        nch = -(-nv // cs)
        picks = sorted(set([0, nch - 1] + list(rng.integers(0, nch, n_sample))))
        for c in picks:
            scratch = np.zeros(info["out_bytes"], dtype=np.uint8) if out_host is None else out_host
            out_host = scratch
            assert oracle.decode_chunks(blob, s, c, 1, scratch) == 0
            a = sout + 2 * c * cs
            b = sout + 2 * min(nv, (c + 1) * cs)
            got = out_dev[a:b].cpu().numpy()
            assert np.array_equal(got, scratch[a:b]), (s, c)


def _full_size(tensors):
    blob = k3.encode_layer(tensors)
    info = k3.layer_info(blob)
    d_blob = torch.from_numpy(blob).cuda()
    out = torch.empty(info["out_bytes"], dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3.set_decoder_variant(0)
    k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, out, st)
    # then twice as the benchmark launches it (work-area pools, early start):
    # the first of the two starts while the plain decode above finishes
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2 = torch.empty_like(out)
    for _ in range(2):
        k3.decode_layer(blob[: info["hdr_bytes"]], d_blob, out2, st2, work=work, early_start=True)
    torch.cuda.synchronize()
    assert st.item() == 0 and st2.item() == 0
    assert int(work.abs().sum().item()) == 0
    assert torch.equal(out, out2)
    _sampled_parity(blob, tensors, out)
    # the oracle encoder's tables equal the product encoder's
    for t, x in zip(tensor_regions(blob), tensors):
        assert np.array_equal(blob[64 + 256 * t["table"]: 64 + 256 * (t["table"] + 1)],
                              oracle.code_lengths(oracle.histogram(x)).astype(np.uint8))


@pytest.mark.slow
def test_full_projection():
    _full_size([workloads.projection()])


@pytest.mark.slow
def test_full_heavy_tail():
    _full_size([workloads.heavy_tail()])


@pytest.mark.slow
def test_full_trunk_layer():
    _full_size(workloads.trunk_layer())


@pytest.mark.slow
def test_full_ring_trunk_layers():
    """Three trunk layers (9 tensors, 9 code tables and 28 stripes each,
    seeds 10-12 of the streaming ring) go from pinned host memory through
    the ring's two device slots, more layers than slots: every byte of every
    layer equals its input tensors (checked on the GPU) and sampled chunks of
    every stripe equal the oracle's bit-serial decode of those chunks."""
    seeds = workloads.ring_layers(n_layers=3)
    layers = [workloads.trunk_layer(seed=s) for s in seeds]
    blobs = [k3.encode_layer(ts) for ts in layers]
    h = [torch.from_numpy(b).pin_memory() for b in blobs]
    outs = [torch.full((k3.layer_info(b)["out_bytes"],), SENTINEL, dtype=torch.uint8, device="cuda") for b in blobs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ring = k3.Ring(max(b.size for b in blobs), 2)
    stats = ring.run(h, outs, st)
    ring.close()
    assert st.item() == 0
    assert stats["h2d_bytes"] == sum(b.size for b in blobs)
    assert stats["out_bytes"] == sum(2 * sum(t.size for t in ts) for ts in layers)
    for i, (ts, b, o) in enumerate(zip(layers, blobs, outs)):
        info = k3.layer_info(b)
        assert info["n_tables"] == 9 and info["n_tensors"] == 9 and info["n_stripes"] == 28
        _sampled_parity(b, ts, o, n_sample=6, seed=i)


def test_random_layers_every_launch_path():
    """24 seeded random layers (alphabet size and skew, 1-4 tensors of
    1-300,000 values, chunk and sub-stream sizes, shared or per-tensor
    tables) decoded three ways on the GPU: plain, with a work area, and
    with a work area and early start back to back.  Every tensor's bytes
    equal the input's."""
    rng = np.random.default_rng(2026)
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device="cuda")
    for case in range(24):
        tensors = []
        for _ in range(int(rng.integers(1, 5))):
            n = int(rng.integers(1, 300_001))
            n_sym = int(rng.integers(1, 257))
            syms = rng.choice(256, size=n_sym, replace=False)
            w = float(rng.uniform(0.05, 1.0)) ** np.arange(n_sym, dtype=np.float64)
            hi = rng.choice(syms, size=n, p=w / w.sum()).astype(np.uint16)
            tensors.append((hi << 8) | rng.integers(0, 256, size=n, dtype=np.uint16))
        chunk_syms = int(rng.choice([64, 256, 1000, 4096, 8192]))
        sub_syms = int(rng.choice([0, 8, 64, 256, 512]))
        blob = oracle.encode_layer(tensors, chunk_syms=chunk_syms, sub_syms=sub_syms,
                                   shared_table=bool(rng.integers(0, 2)))
        info = k3.layer_info(blob)
        hdr = blob[: info["hdr_bytes"]]
        d_blob = torch.from_numpy(blob).cuda()
        outs = [torch.empty(info["out_bytes"], dtype=torch.uint8, device="cuda") for _ in range(3)]
        st = torch.zeros(3, dtype=torch.int32, device="cuda")
        k3.decode_layer(hdr, d_blob, outs[0], st[0:1])
        k3.decode_layer(hdr, d_blob, outs[1], st[1:2], work=work)
        k3.decode_layer(hdr, d_blob, outs[2], st[2:3], work=work, early_start=True)
        torch.cuda.synchronize()
        assert int(st.abs().sum().item()) == 0, case
        assert int(work.abs().sum().item()) == 0, case
        for t, x in enumerate(tensors):
            ti = k3.tensor_info(hdr, t)
            a, b = ti["out_offset"], ti["out_offset"] + 2 * ti["n_values"]
            ref = torch.from_numpy(x.view(np.uint8)).cuda()
            for o in outs:
                assert torch.equal(o[a:b], ref), (case, t)
