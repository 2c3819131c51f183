"""Property tests on CPU: random layers (alphabet size and skew, tensor
sizes, chunk and sub-stream sizes, shared or per-tensor tables) through
the product's CPU encoder, the oracle's encoder and both CPU decoders.

For every drawn layer: the two encoders write the same bytes; the oracle's
bit-serial decoder and the article-style decoder both give back the input
bytes exactly; the library's size bound holds; the library and the oracle
read the same header fields."""
import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
k3 = pytest.importorskip("lossless_bf16_weight_k3huf_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    k3._build.build()


def _tensor(seed: int, n: int, n_sym: int, skew: float) -> np.ndarray:
    """bf16 bit patterns: high bytes from n_sym symbols with geometric
    weights (ratio skew), low bytes uniform."""
    rng = np.random.default_rng(seed)
    syms = rng.choice(256, size=n_sym, replace=False)
    w = skew ** np.arange(n_sym, dtype=np.float64)
    hi = rng.choice(syms, size=n, p=w / w.sum()).astype(np.uint16)
    lo = rng.integers(0, 256, size=n, dtype=np.uint16)
    return (hi << 8) | lo


layers = st.lists(
    st.tuples(st.integers(0, 2**31 - 1), st.integers(1, 20_000), st.integers(1, 256),
              st.floats(0.05, 1.0)),
    min_size=1, max_size=4)


@hyp.settings(max_examples=120, deadline=None, derandomize=True)
@hyp.given(spec=layers, chunk_syms=st.sampled_from([1, 7, 64, 256, 1000, 4096]),
           sub_syms=st.sampled_from([0, 8, 16, 200, 256, 512]), shared=st.booleans())
def test_random_layers_round_trip_and_encoders_agree(spec, chunk_syms, sub_syms, shared):
    tensors = [_tensor(*t) for t in spec]
    kw = dict(chunk_syms=chunk_syms, sub_syms=sub_syms, shared_table=shared)
    blob = k3.encode_layer(tensors, threads=2, **kw)
    ref = oracle.encode_layer(tensors, **kw)
    assert np.array_equal(blob, ref)
    assert blob.size <= k3.encode_bound([t.size for t in tensors], **kw)

    info, oinfo = k3.layer_info(blob), oracle.layer_info(blob)
    for key in ("chunk_syms", "n_tables", "n_tensors", "n_stripes", "raw_bytes", "blob_bytes", "hdr_bytes",
                "out_bytes", "sub_syms"):
        assert info[key] == oinfo[key], key

    rc, out = oracle.decode_layer(blob)
    assert rc == 0
    rc2, out2 = oracle.pagestyle_decode_layer(blob)
    assert rc2 == 0
    hdr = blob[: info["hdr_bytes"]]
    for t, x in enumerate(tensors):
        ti = k3.tensor_info(hdr, t)
        a, b = ti["out_offset"], ti["out_offset"] + 2 * ti["n_values"]
        assert np.array_equal(out[a:b].view(np.uint16), x)
        assert np.array_equal(out2[a:b].view(np.uint16), x)
