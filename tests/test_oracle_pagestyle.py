"""Pins of the article-style CPU decoder (oracle/k3huf_pagestyle.c), the
like-for-like CPU timing beside the bit-serial oracle.

Its table is checked window by window against the hand-worked examples
in tests/golden/canonical_examples.txt and against the oracle's bit-serial
code walk, its stripe decode byte for byte against the oracle's decode of the
same containers (and both against the original tensors), and its error
paths on streams the oracle rejects."""
import numpy as np
import pytest

import oracle
import workloads
from conftest import golden_lines


def _stripe0(blob):
    info = oracle.layer_info(blob)
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    return int.from_bytes(blob[sdir:sdir + 8].tobytes(), "little")


def _tables():
    yield "normal", oracle.code_lengths(oracle.histogram(workloads.tiny()))
    yield "heavy tail (limiter fired)", oracle.code_lengths(oracle.histogram(workloads.heavy_tail(n=1 << 20)))
    yield "dyadic, 12-bit codes", oracle.code_lengths(oracle.histogram(workloads.dyadic_long_codes(1 << 16)))
    yield "uniform bytes (all length 8)", oracle.code_lengths(oracle.histogram(workloads.uniform_bytes(1 << 16)))
    one = np.zeros(256, np.int64)
    one[0x3C] = 1
    yield "single symbol", one
    inc = np.zeros(256, np.int64)
    inc[0], inc[1] = 1, 2                              # incomplete: half of the code space unused
    yield "incomplete", inc


@pytest.mark.parametrize("name,codelen", list(_tables()), ids=[n for n, _ in _tables()])
def test_table_matches_bit_serial_walk(name, codelen):
    """Entry w equals the oracle's bit-serial decode of window w: symbol and
    length of the code it starts with, or 0 where no code starts."""
    cl = np.asarray(codelen, np.uint8)
    lut = oracle.pagestyle_table(cl)
    for w in range(4096):
        sym, used = oracle.decode_window(cl, w)
        want = 0 if sym < 0 else (sym << 4) | used
        assert int(lut[w]) == want, (name, w)


@pytest.mark.parametrize("row", list(golden_lines("canonical_examples.txt")), ids=lambda r: r[0])
def test_table_matches_hand_worked_ranges(row):
    """The hand-worked examples E1-E6 (canonical codes worked out by hand and
    the 12-bit window ranges they imply): every window of the article-style
    table holds the symbol and length its range says, 0 where no code
    starts."""
    name, maxlen, lens_s, _codes, ranges_s = row
    cl = np.zeros(256, np.uint8)
    for tok in lens_s.split():
        sym, ln = tok.split(":")
        cl[int(sym)] = int(ln)
    lut = oracle.pagestyle_table(cl)
    covered = 0
    for tok in ranges_s.split():
        sym, rng = tok.split(":")
        lo, hi = (int(x) for x in rng.strip("[)").split(","))
        want = 0 if sym == "x" else (int(sym) << 4) | int(cl[int(sym)])
        assert (lut[lo:hi] == want).all(), (name, sym, lo, hi)
        covered += hi - lo
    assert covered == 4096, name


def test_table_rejects_long_lengths():
    cl = np.zeros(256, np.uint8)
    cl[0] = 13
    with pytest.raises(ValueError):
        oracle.pagestyle_table(cl)


CASES = {
    "tiny": lambda: [workloads.tiny()],
    "ragged": lambda: [workloads.normal_tensor((n,), 0.02, 5) for n in (1, 4095, 4097, 33)],
    "single symbol": lambda: [workloads.single_symbol(10_000)],
    "two symbols": lambda: [workloads.two_symbol(10_000)],
    "uniform bytes": lambda: [workloads.uniform_bytes(50_000)],
    "dyadic long codes": lambda: [workloads.dyadic_long_codes(1 << 16)],
    "heavy tail": lambda: [workloads.heavy_tail(n=1 << 21)],
    "several tables": lambda: [workloads.normal_tensor((64, 96), 0.1, 3, 0), workloads.normal_tensor((5,), 0.3, 3, 1),
                               workloads.normal_tensor((96, 640), 0.04, 3, 2)],
    "two stripes": lambda: [np.tile(workloads.tiny(), 17)[: (1 << 25) + 5003]],
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_equals_oracle_and_input(name):
    tensors = CASES[name]()
    blob = oracle.encode_layer(tensors)
    rc, ref = oracle.decode_layer(blob)
    assert rc == 0
    rc2, out = oracle.pagestyle_decode_layer(blob)
    assert rc2 == 0
    assert np.array_equal(out, ref)
    info = oracle.layer_info(blob)
    sdir = 64 + 256 * info["n_tables"]
    for t, x in enumerate(tensors):
        e = sdir + 32 * t
        off = int.from_bytes(blob[e + 24:e + 32].tobytes(), "little")     # the tensor's output offset
        flat = np.asarray(x, np.uint16).reshape(-1)
        assert np.array_equal(out[off:off + 2 * flat.size].view(np.uint16), flat)


def test_undecodable_window_is_an_error():
    """An incomplete table {0: 1 bit, 1: 2 bits} and a stream that starts
    with 01 (no code): the oracle rejects it, and so does this decoder."""
    x = np.array([0x0000, 0x0100, 0x0000, 0x0000] * 3, dtype=np.uint16)
    blob = oracle.encode_layer([x])
    o = _stripe0(blob)
    bits_off = int.from_bytes(blob[o + 24:o + 28].tobytes(), "little")
    blob[64 + 1] = 2
    blob[o + 16:o + 24] = np.frombuffer((15).to_bytes(8, "little"), np.uint8)
    blob[o + bits_off:o + bits_off + 2] = [0b10011100, 0b11100110]
    so = o + 32 + 4 * 1
    k = int.from_bytes(blob[8:12].tobytes(), "little") // int.from_bytes(blob[56:60].tobytes(), "little") - 1
    blob[so:so + 2 * k] = np.frombuffer(np.full(k, 15, "<u2").tobytes(), np.uint8)
    assert oracle.decode_layer(blob)[0] == 0
    rc, out = oracle.pagestyle_decode_layer(blob)
    assert rc == 0 and np.array_equal(out[:24].view(np.uint16), x)
    bad = blob.copy()
    bad[o + bits_off] = 0b01011100
    assert oracle.decode_layer(bad)[0] != 0
    assert oracle.pagestyle_decode_layer(bad)[0] == oracle.E_FORMAT


def test_stream_shorter_than_its_codes_is_an_error():
    """A recorded bit length below what the values need: decoding reads
    past it, which is an error."""
    blob = oracle.encode_layer([workloads.normal_tensor((20_000,), 0.02, 9)])
    o = _stripe0(blob)
    bits = int.from_bytes(blob[o + 16:o + 24].tobytes(), "little")
    bad = blob.copy()
    bad[o + 16:o + 24] = np.frombuffer((bits - 9).to_bytes(8, "little"), np.uint8)
    assert oracle.decode_layer(bad)[0] != 0
    assert oracle.pagestyle_decode_layer(bad)[0] == oracle.E_FORMAT
