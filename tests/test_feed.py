"""Storage feed (host side, no GPU): a container file read back through
k3huf_feed_read with parallel preads, O_DIRECT where the filesystem allows
it, equals the file's bytes; misaligned or out-of-range requests are
refused before any read."""
import os

import numpy as np
import pytest

k3 = pytest.importorskip("lossless_bf16_weight_k3huf_gb300")

MiB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    k3._build.build()


@pytest.fixture(scope="module")
def data_file(tmp_path_factory):
    rng = np.random.default_rng(7)
    data = rng.integers(0, 256, 21 * MiB + 777, dtype=np.uint8)
    p = tmp_path_factory.mktemp("feed") / "blob.bin"
    p.write_bytes(data.tobytes())
    return str(p), data


@pytest.mark.parametrize("threads", [1, 3, 8])
@pytest.mark.parametrize("offset,nbytes", [(0, 1), (0, 4095), (0, 4096), (4096, 4097), (8 * MiB, 8 * MiB + 1),
                                           (12288, 21 * MiB + 777 - 12288), (0, 21 * MiB + 777)])
def test_read_matches_file(data_file, threads, offset, nbytes):
    path, data = data_file
    f = k3.Feed(path, threads=threads)
    assert f.direct in (True, False)
    buf = k3.aligned_host(-(-nbytes // 4096) * 4096)
    buf[:] = 0xCC
    f.read(offset, nbytes, buf)
    assert np.array_equal(buf[:nbytes], data[offset: offset + nbytes])
    f.close()


def test_read_refuses_bad_requests(data_file):
    path, data = data_file
    f = k3.Feed(path, threads=2)
    buf = k3.aligned_host(2 * MiB)
    with pytest.raises(k3.K3HufError) as e:
        f.read(100, 4096, buf)                                   # offset not 4096-aligned
    assert e.value.code == k3.E_ARG
    with pytest.raises(k3.K3HufError) as e:
        f.read(0, 4096, buf.ctypes.data + 8, 4096)               # buffer not aligned
    assert e.value.code == k3.E_ARG
    with pytest.raises(k3.K3HufError) as e:
        f.read(0, 4097, buf[:4096])                              # buffer shorter than whole blocks
    assert e.value.code == k3.E_ARG
    with pytest.raises(k3.K3HufError) as e:
        f.read(20 * MiB, 2 * MiB, buf)                           # past the end of the file
    assert e.value.code == k3.E_IO
    f.close()
    with pytest.raises(k3.K3HufError) as e:
        k3.Feed(os.path.join(os.path.dirname(path), "missing.bin"))
    assert e.value.code == k3.E_IO


def test_write_layers_aligns_offsets(tmp_path):
    rng = np.random.default_rng(3)
    blobs = [rng.integers(0, 256, n, dtype=np.uint8) for n in (5000, 4096, 1, 70000)]
    p = str(tmp_path / "layers.bin")
    offs = k3.write_layers(p, blobs)
    assert all(o % 4096 == 0 for o in offs)
    f = k3.Feed(p, threads=4)
    for o, b in zip(offs, blobs):
        buf = k3.aligned_host(-(-b.size // 4096) * 4096)
        f.read(o, b.size, buf)
        assert np.array_equal(buf[:b.size], b)
    f.close()
