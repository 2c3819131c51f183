"""Pins of the oracle's container writer and bit-serial decoder.

The decoder is an exact inverse, so the plain definition of its result is
the input itself: decode(encode(x)) == x byte for byte (article "Kimi K3 纯
CPU 推理中的无损 Trunk 压缩：一次被解码速度判死刑的 Huffman 压缩实验",
section 验证结果).  The bit stream is checked against an independent packing
of the codes written here, and the sizes against closed forms."""
import numpy as np
import pytest

import oracle
import workloads

STRIPE_VALUES = 1 << 25


def _u32(b, off):
    return int.from_bytes(b[off:off + 4].tobytes(), "little")


def _u64(b, off):
    return int.from_bytes(b[off:off + 8].tobytes(), "little")


def parse(blob):
    """Walk the container by its documented layout (version 1)."""
    h = {
        "magic": blob[0:4].tobytes(), "version": int.from_bytes(blob[4:6].tobytes(), "little"),
        "maxlen": int.from_bytes(blob[6:8].tobytes(), "little"), "chunk_syms": _u32(blob, 8),
        "n_tables": _u32(blob, 12), "n_tensors": _u32(blob, 16), "n_stripes": _u32(blob, 20),
        "raw_bytes": _u64(blob, 24), "blob_bytes": _u64(blob, 32), "stripe_values": _u32(blob, 40),
        "hdr_bytes": _u32(blob, 44), "out_bytes": _u64(blob, 48), "sub_syms": _u32(blob, 56),
    }
    t0 = 64 + 256 * h["n_tables"]
    h["tables"] = [blob[64 + 256 * i: 64 + 256 * (i + 1)].copy() for i in range(h["n_tables"])]
    h["tensors"] = []
    for i in range(h["n_tensors"]):
        e = t0 + 32 * i
        h["tensors"].append(dict(table=_u32(blob, e), first_stripe=_u32(blob, e + 4), n_stripes=_u32(blob, e + 8),
                                 n_values=_u64(blob, e + 16), out_offset=_u64(blob, e + 24)))
    s0 = t0 + 32 * h["n_tensors"]
    h["stripes"] = []
    for i in range(h["n_stripes"]):
        e = s0 + 32 * i
        st = dict(blob_offset=_u64(blob, e), stripe_bytes=_u64(blob, e + 8), out_offset=_u64(blob, e + 16),
                  n_values=_u32(blob, e + 24), table=_u32(blob, e + 28))
        o = st["blob_offset"]
        st.update(magic=blob[o:o + 4].tobytes(), hdr_table=_u32(blob, o + 4), hdr_n_values=_u32(blob, o + 8),
                  n_chunks=_u32(blob, o + 12), huff_bits=_u64(blob, o + 16), bits_offset=_u32(blob, o + 24),
                  even_offset=_u32(blob, o + 28))
        st["chunk_bitoff"] = np.frombuffer(blob[o + 32: o + 32 + 4 * st["n_chunks"]].tobytes(), dtype="<u4")
        S = h["chunk_syms"] // h["sub_syms"]
        so = o + 32 + 4 * st["n_chunks"]
        st["sub_bitoff"] = np.frombuffer(blob[so: so + 2 * st["n_chunks"] * (S - 1)].tobytes(),
                                         dtype="<u2").reshape(st["n_chunks"], S - 1)
        h["stripes"].append(st)
    return h


def _independent_bits(hi, lens, codes):
    """Bit string (uint8 0/1 per bit) of the symbols' codes, MSB first."""
    L = lens[hi]
    C = codes[hi]
    total = int(L.sum())
    bits = np.zeros(total, dtype=np.uint8)
    starts = np.concatenate([[0], np.cumsum(L)[:-1]])
    for b in range(int(L.max())):
        m = L > b
        bits[starts[m] + b] = (C[m] >> (L[m] - 1 - b)) & 1
    return bits


def roundtrip(tensors, **kw):
    blob = oracle.encode_layer(tensors, **kw)
    rc, out = oracle.decode_layer(blob)
    assert rc == 0
    h = parse(blob)
    for t, x in zip(h["tensors"], tensors):
        got = out[t["out_offset"]: t["out_offset"] + 2 * t["n_values"]].view(np.uint16)
        assert np.array_equal(got, np.asarray(x, dtype=np.uint16).reshape(-1))
    return blob, h


def _expected_sub_syms(chunk_syms, sub_syms):
    if sub_syms == 0 or chunk_syms % sub_syms or chunk_syms * 12 > 65535:
        return chunk_syms
    return sub_syms


def check_layout(blob, tensors, chunk_syms=4096, shared=False, sub_syms=256):
    h = parse(blob)
    ss = _expected_sub_syms(chunk_syms, sub_syms)
    assert h["sub_syms"] == ss
    S = chunk_syms // ss
    assert h["magic"] == b"K3HF" and h["version"] == 1 and h["maxlen"] == 12
    assert h["chunk_syms"] == chunk_syms and h["stripe_values"] == STRIPE_VALUES
    assert h["blob_bytes"] == blob.size and h["hdr_bytes"] % 256 == 0
    assert h["raw_bytes"] == sum(2 * np.asarray(t).size for t in tensors)
    assert h["n_tables"] == (1 if shared else len(tensors))
    sid = 0
    prev_end = h["hdr_bytes"]
    for ti, (t, x) in enumerate(zip(h["tensors"], tensors)):
        x = np.asarray(x, dtype=np.uint16).reshape(-1)
        assert t["out_offset"] % 256 == 0 and t["first_stripe"] == sid
        assert t["n_stripes"] == -(-x.size // STRIPE_VALUES)
        lens = h["tables"][t["table"]].astype(np.int64)
        assert oracle.check_codelen(lens) == 0
        codes, _, _ = oracle.canonical(lens)
        codes = codes.astype(np.int64)
        if not shared:
            assert (lens == oracle.code_lengths(oracle.histogram(x))).all()
        for k in range(t["n_stripes"]):
            st = h["stripes"][sid + k]
            v0 = k * STRIPE_VALUES
            xs = x[v0: v0 + STRIPE_VALUES]
            hi = (xs >> 8).astype(np.int64)
            lo = (xs & 0xFF).astype(np.uint8)
            assert st["magic"] == b"K3HS" and st["hdr_n_values"] == xs.size == st["n_values"]
            assert st["table"] == st["hdr_table"] == t["table"]
            assert st["blob_offset"] % 256 == 0 and st["blob_offset"] >= prev_end
            assert st["out_offset"] == t["out_offset"] + 2 * v0
            assert st["n_chunks"] == -(-xs.size // chunk_syms)
            assert st["huff_bits"] == int(lens[hi].sum())                   # closed form
            per_chunk = np.add.reduceat(lens[hi], np.arange(0, xs.size, chunk_syms))
            assert np.array_equal(st["chunk_bitoff"].astype(np.int64), np.concatenate([[0], np.cumsum(per_chunk)[:-1]]))
            assert st["bits_offset"] % 16 == 0 and st["even_offset"] % 16 == 0
            assert st["bits_offset"] == -(-(32 + 4 * st["n_chunks"] + 2 * st["n_chunks"] * (S - 1)) // 16) * 16
            # sub-stream index: relative bit offset of value min(k*ss, len) of each chunk
            cum = np.concatenate([[0], np.cumsum(lens[hi])])
            for c in range(st["n_chunks"]):
                a = c * chunk_syms
                ln_c = min(chunk_syms, xs.size - a)
                for k in range(1, S):
                    assert st["sub_bitoff"][c, k - 1] == cum[a + min(k * ss, ln_c)] - cum[a], (c, k)
            o = st["blob_offset"]
            nbytes = (st["huff_bits"] + 7) // 8
            assert st["even_offset"] == st["bits_offset"] + (-(-nbytes // 16)) * 16 + 32
            assert st["stripe_bytes"] == st["even_offset"] + (-(-xs.size // 16)) * 16
            stream = blob[o + st["bits_offset"]: o + st["even_offset"]]
            assert not stream[nbytes:].any()                                 # zero padding
            if xs.size <= 1 << 21:
                ref = np.packbits(_independent_bits(hi, lens, codes))
                assert np.array_equal(stream[:nbytes], ref)
            assert np.array_equal(blob[o + st["even_offset"]: o + st["even_offset"] + xs.size], lo)
            prev_end = o + st["stripe_bytes"]
        sid += t["n_stripes"]
    assert sid == h["n_stripes"]
    return h


def test_tiny_roundtrip_and_layout():
    x = workloads.tiny()
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    rate = blob.size / (2 * x.size)
    assert 0.6 < rate < 0.75


@pytest.mark.parametrize("n", [1, 2, 3, 15, 16, 17, 4095, 4096, 4097, 8191, 12289, 100_003])
def test_ragged_sizes(n):
    x = workloads.normal_tensor((n,), 0.02, seed=n)
    blob, _ = roundtrip([x])
    check_layout(blob, [x])


@pytest.mark.parametrize("chunk_syms", [1, 7, 256, 1000, 4096, 65536])
def test_chunk_sizes(chunk_syms):
    x = workloads.normal_tensor((50_001,), 0.05, seed=9)
    blob, _ = roundtrip([x], chunk_syms=chunk_syms)
    check_layout(blob, [x], chunk_syms=chunk_syms)


def test_single_symbol_plane():
    x = workloads.single_symbol(10_000)
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    st = h["stripes"][0]
    assert st["huff_bits"] == x.size                                         # 1 bit per value
    lens = h["tables"][0]
    assert lens[0x3F] == 1 and lens.sum() == 1
    for w in (0, 1, 2047):
        assert oracle.decode_window(lens, w) == (0x3F, 1)
    for w in (2048, 4095):
        assert oracle.decode_window(lens, w) == (-1, 0)


def test_two_symbol_plane():
    x = workloads.two_symbol(10_000)
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    lens = h["tables"][0]
    assert lens[0x3F] == 1 and lens[0xBF] == 1 and lens.sum() == 2


def test_uniform_bytes_all_symbols():
    x = workloads.uniform_bytes(300_000)
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    assert (h["tables"][0] > 0).all()


def test_dyadic_plane_gets_dyadic_lengths():
    # symbol probabilities 2^-l give Huffman lengths l exactly (the entropy
    # bound is met with equality), here 1, 2, 3, 4, 6, 6 and 128 codes of 12
    x = workloads.dyadic_long_codes(1 << 19)
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    lens = h["tables"][0].astype(int)
    assert sorted(lens[lens > 0].tolist()) == [1, 2, 3, 4, 6, 6] + [12] * 128


def test_heavy_tail_sample_fires_limiter():
    x = workloads.heavy_tail(n=1 << 21)
    cnt = oracle.histogram(x)
    assert oracle.huffman_lengths(cnt).max() > 12
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    assert h["tables"][0].max() == 12


def test_multi_tensor_layer_and_shared_table():
    ts = [workloads.normal_tensor((64, 96), 1 / 96 ** 0.5, 3, tag=0),
          workloads.normal_tensor((5,), 0.3, 3, tag=1),
          workloads.normal_tensor((96, 640), 1 / 640 ** 0.5, 3, tag=2)]
    blob, h = roundtrip(ts)
    check_layout(blob, ts)
    assert [t["out_offset"] for t in h["tensors"]] == [0, 12288, 12544]
    blob2, h2 = roundtrip(ts, shared_table=True)
    check_layout(blob2, ts, shared=True)
    allx = np.concatenate([np.asarray(t).reshape(-1) for t in ts])
    assert (h2["tables"][0] == oracle.code_lengths(oracle.histogram(allx))).all()


def test_multi_stripe_tensor():
    """A tensor one stripe plus a ragged tail long: two stripes, the second
    starting at value 2^25 and output byte 2^26."""
    n = STRIPE_VALUES + 5003
    x = np.tile(workloads.tiny(), n // (1 << 21) + 1)[:n]
    blob, h = roundtrip([x])
    check_layout(blob, [x])
    assert h["n_stripes"] == 2
    assert h["stripes"][1]["out_offset"] == 2 * STRIPE_VALUES
    assert h["stripes"][1]["n_values"] == 5003


@pytest.mark.parametrize("chunk_syms,sub_syms", [(4096, 512), (4096, 256), (4096, 4096), (4096, 0), (4096, 1000),
                                                (1024, 8), (8192, 512), (64, 16), (8, 1)])
@pytest.mark.parametrize("n", [1, 4095, 4097, 30_001])
def test_sub_stream_index(chunk_syms, sub_syms, n):
    x = workloads.normal_tensor((n,), 0.03, seed=n + chunk_syms)
    blob, _ = roundtrip([x], chunk_syms=chunk_syms, sub_syms=sub_syms)
    check_layout(blob, [x], chunk_syms=chunk_syms, sub_syms=sub_syms)


def test_corrupt_sub_index_is_rejected():
    x = workloads.normal_tensor((20_000,), 0.02, seed=66)
    blob = oracle.encode_layer([x])
    h = parse(blob)
    st = h["stripes"][0]
    so = st["blob_offset"] + 32 + 4 * st["n_chunks"]
    for entry in (0, 6, 7 * 4 + 6):                   # first, last of chunk 0, last of the short chunk 4
        bad = blob.copy()
        bad[so + 2 * entry] ^= 1
        assert oracle.decode_layer(bad)[0] == oracle.E_FORMAT, entry


def test_decode_chunks_matches_full_decode():
    x = workloads.normal_tensor((40_000,), 0.02, seed=4)
    blob = oracle.encode_layer([x])
    _, full = oracle.decode_layer(blob)
    part = np.zeros_like(full)
    assert oracle.decode_chunks(blob, 0, 3, 2, part) == 0
    a, b = 2 * 3 * 4096, 2 * 5 * 4096
    assert np.array_equal(part[a:b], full[a:b])
    assert not part[:a].any() and not part[b:].any()


def test_corruptions_are_rejected():
    x = workloads.normal_tensor((20_000,), 0.02, seed=6)
    blob = oracle.encode_layer([x])
    h = parse(blob)
    st = h["stripes"][0]
    o = st["blob_offset"]
    # chunk index entry off by one bit -> chunk end mismatch
    bad = blob.copy()
    bad[o + 32 + 4] ^= 1
    assert oracle.decode_layer(bad)[0] == oracle.E_FORMAT
    # bit count one short -> the last code runs past the end
    bad = blob.copy()
    bad[o + 16] = (int(bad[o + 16]) - 1) & 0xFF
    assert oracle.decode_layer(bad)[0] == oracle.E_FORMAT
    # over-subscribed table in the header -> table error
    bad = blob.copy()
    bad[64: 64 + 256] = 1
    assert oracle.decode_layer(bad)[0] == oracle.E_OVERSUB
    # empty table
    bad = blob.copy()
    bad[64: 64 + 256] = 0
    assert oracle.decode_layer(bad)[0] == oracle.E_EMPTY
    # wrong magic
    bad = blob.copy()
    bad[0] ^= 0xFF
    with pytest.raises(ValueError):
        oracle.decode_layer(bad)


def test_incomplete_code_invalid_window_is_rejected():
    """An incomplete table (E4: {0:1, 1:2}, codes sym1=00, sym0=1) leaves the
    windows starting with 01 undecodable.  The encoder never writes such a
    table for two symbols, so the container is patched by hand."""
    x = np.array([0x0000, 0x0100, 0x0000, 0x0000], dtype=np.uint16)
    blob = oracle.encode_layer([x])
    h = parse(blob)
    assert list(h["tables"][0][:2]) == [1, 1]
    st = h["stripes"][0]
    o = st["blob_offset"]
    blob[64 + 1] = 2                                   # table {0:1, 1:2}
    blob[o + 16: o + 24] = np.frombuffer((5).to_bytes(8, "little"), np.uint8)
    blob[o + st["bits_offset"]] = 0b10011000           # 1 00 1 1
    so = o + 32 + 4 * st["n_chunks"]                   # sub-stream starts past the end: all at bit 5
    k = h["chunk_syms"] // h["sub_syms"] - 1
    blob[so: so + 2 * k] = np.frombuffer(np.full(k, 5, "<u2").tobytes(), np.uint8)
    rc, out = oracle.decode_layer(blob)
    assert rc == 0 and np.array_equal(out[:8].view(np.uint16), x)
    bad = blob.copy()
    bad[o + st["bits_offset"]] = 0b01011000            # starts with 01: no code
    assert oracle.decode_layer(bad)[0] == oracle.E_FORMAT


@pytest.mark.parametrize("case", ["ragged", "chunks", "multi", "shared", "two_stripes"])
def test_container_bytes_is_the_written_size(case):
    """The oracle's sizing pass (no bits packed) gives the size of the
    container its writer produces, whose layout check_layout walks field by
    field against the closed forms."""
    kw = {}
    if case == "ragged":
        ts = [workloads.normal_tensor((12289,), 0.02, seed=21)]
    elif case == "chunks":
        ts = [workloads.normal_tensor((50_001,), 0.05, seed=22)]
        kw = {"chunk_syms": 1000}
    elif case in ("multi", "shared"):
        ts = [workloads.normal_tensor((700, 33), 0.02, seed=23), workloads.single_symbol(5),
              workloads.dyadic_long_codes(40_000)]
        kw = {"shared_table": case == "shared"}
    else:
        ts = [np.tile(workloads.tiny(), 17)[: STRIPE_VALUES + 4097]]
    blob = oracle.encode_layer(ts, **kw)
    check_layout(blob, ts, chunk_syms=kw.get("chunk_syms", 4096), shared=kw.get("shared_table", False))
    assert oracle.container_bytes(ts, **kw) == blob.size
