"""Decode fused into its consumer: y += W x with W held as a k3huf container
and decoded on chip.  Compared with the oracle's decode of W multiplied by x
in float64.  The GPU sums in fp32: each lane adds about sub_syms products in
order, a warp reduction adds 5 levels and the row's work items are added
atomically, so the error is below (256 + 5 + items per row) x 2^-24 of
sum |W| |x|; the test allows 1e-4 of it."""
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


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_gemv(blob, tensor, cols, x_bits, y0=None):
    info = k3.layer_info(blob)
    d_blob = torch.from_numpy(blob).cuda()
    n = k3.tensor_info(blob, tensor)["n_values"]
    y = torch.zeros(n // cols, dtype=torch.float32, device="cuda") if y0 is None else y0
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3.gemv_layer(blob[: info["hdr_bytes"]], d_blob, tensor, cols, x, y, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return y.cpu().numpy().astype(np.float64)


def reference(blob, tensor, cols, x_bits):
    rc, out = oracle.decode_layer(blob)
    assert rc == 0
    t = k3.tensor_info(blob, tensor)
    w = out[t["out_offset"]: t["out_offset"] + 2 * t["n_values"]].view(np.uint16)
    W = bf16_to_f64(w).reshape(-1, cols)
    x = bf16_to_f64(x_bits)
    return W @ x, np.abs(W) @ np.abs(x)


def x_vector(cols, seed):
    return workloads.normal_tensor((cols,), 1.0, seed).reshape(-1)


@pytest.mark.parametrize("rows,cols", [(1, 8192), (7, 8192), (64, 16384), (3, 24576)])
def test_gemv_matches_oracle(rows, cols):
    w = workloads.normal_tensor((rows, cols), 0.02, rows + cols)
    blob = oracle.encode_layer([w])
    x = x_vector(cols, 5)
    y = run_gemv(blob, 0, cols, x)
    ref, mag = reference(blob, 0, cols, x)
    assert np.all(np.abs(y - ref) <= 1e-4 * mag + 1e-30)


def test_gemv_multi_stripe_tensor_and_heavy_tail():
    rows, cols = 4097, 8192                     # 2^25 + 8192 values: two stripes, the second one row
    w = workloads.heavy_tail(n=rows * cols).reshape(rows, cols)
    blob = oracle.encode_layer([w])
    assert k3.layer_info(blob)["n_stripes"] == 2
    x = x_vector(cols, 6)
    y = run_gemv(blob, 0, cols, x)
    ref, mag = reference(blob, 0, cols, x)
    assert np.all(np.abs(y - ref) <= 1e-4 * mag + 1e-30)


def test_gemv_picks_the_tensor_and_accumulates():
    ts = [workloads.normal_tensor((5, 8192), 0.1, 1), workloads.normal_tensor((9, 16384), 0.03, 2),
          workloads.normal_tensor((77,), 0.3, 3)]
    blob = oracle.encode_layer(ts)
    x = x_vector(16384, 7)
    y0 = torch.full((9,), 0.5, dtype=torch.float32, device="cuda")
    y = run_gemv(blob, 1, 16384, x, y0=y0)
    ref, mag = reference(blob, 1, 16384, x)
    assert np.all(np.abs(y - (ref + 0.5)) <= 1e-4 * mag + 1e-6)


def test_gemv_refuses_unsupported_shapes():
    blob = oracle.encode_layer([workloads.normal_tensor((24, 576), 0.02, 4), workloads.normal_tensor((2, 8192), 0.02, 5)])
    info = k3.layer_info(blob)
    d_blob = torch.from_numpy(blob).cuda()
    x = torch.zeros(8192, dtype=torch.int16, device="cuda")
    y = torch.zeros(64, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tensor, cols in [(0, 576), (1, 4096), (1, 3000), (2, 8192)]:
        with pytest.raises(k3.K3HufError) as e:
            k3.gemv_layer(blob[: info["hdr_bytes"]], d_blob, tensor, cols, x, y, st)
        assert e.value.code == k3.E_ARG


def test_gemv_ex_zero_y_and_early_start_back_to_back():
    """k3huf_gemv_layer_ex with both flags, calls back to back on one
    stream: every call gives y = W x for its own x although y starts as
    garbage and the call before it is still adding into y (its zeroing
    waits for that call, its GEMV for the zeroing), interleaved with an
    early-start decode; a multi-stripe heavy-tail matrix and a two-table
    layer."""
    rows, cols = 4097, 8192
    heavy = workloads.heavy_tail(n=rows * cols).reshape(rows, cols)
    blob_a = oracle.encode_layer([heavy])
    blob_b = oracle.encode_layer([workloads.normal_tensor((5, 8192), 0.1, 1), workloads.normal_tensor((96, 16384), 0.03, 2)])
    cases = [(blob_a, 0, cols), (blob_b, 1, 16384)]
    xs = {(i, s): x_vector(c, 20 + s + 7 * i) for i, (_, _, c) in enumerate(cases) for s in range(3)}
    refs = {key: reference(cases[key[0]][0], cases[key[0]][1], cases[key[0]][2], x) for key, x in xs.items()}
    dev = [(torch.from_numpy(b).cuda(), b[: k3.layer_info(b)["hdr_bytes"]]) for b, _, _ in cases]
    dec_out = torch.empty(k3.layer_info(blob_b)["out_bytes"], dtype=torch.uint8, device="cuda")
    dec_ref = torch.from_numpy(oracle.decode_layer(blob_b)[1]).cuda()
    for _ in range(2):
        ys, sts = {}, []
        for s in range(3):
            for i, (b, t, c) in enumerate(cases):
                d_blob, hdr = dev[i]
                y = torch.full((k3.tensor_info(b, t)["n_values"] // c,), float("nan"), dtype=torch.float32, device="cuda")
                st = torch.zeros(1, dtype=torch.int32, device="cuda")
                x = torch.from_numpy(xs[(i, s)].view(np.int16)).cuda()
                k3.gemv_layer(hdr, d_blob, t, c, x, y, st, zero_y=True, early_start=True)
                ys[(i, s)] = y
                sts.append(st)
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            k3.decode_layer(dev[1][1], dev[1][0], dec_out, st, early_start=True)
            sts.append(st)
        torch.cuda.synchronize()
        assert all(int(st.item()) == 0 for st in sts)
        for t in (k3.tensor_info(blob_b, j) for j in range(2)):      # (the gaps between tensors are not written)
            a0, a1 = t["out_offset"], t["out_offset"] + 2 * t["n_values"]
            assert torch.equal(dec_out[a0:a1], dec_ref[a0:a1])
        for key, y in ys.items():
            ref, mag = refs[key]
            assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - ref) <= 1e-4 * mag + 1e-30), key


def test_gemv_ex_reads_x_after_the_kernel_that_writes_it():
    """x is written by the kernel right before an early-start call (with and
    without the zeroing kernel between them): every result uses the new x,
    since the GEMV reads x only after the kernel before it has completed."""
    rows, cols = 512, 16384
    w = workloads.normal_tensor((rows, cols), 0.02, 31)
    blob = oracle.encode_layer([w])
    info = k3.layer_info(blob)
    d_blob, hdr = torch.from_numpy(blob).cuda(), blob[: info["hdr_bytes"]]
    srcs = [torch.from_numpy(x_vector(cols, 40 + i).view(np.int16)).cuda() for i in range(4)]
    x = torch.zeros(cols, dtype=torch.int16, device="cuda")
    for zero_y in (True, False):
        ys = []
        for i, src in enumerate(srcs):
            y = torch.zeros(rows, dtype=torch.float32, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            x.copy_(src)                                  # the kernel before the call writes x
            k3.gemv_layer(hdr, d_blob, 0, cols, x, y, st, zero_y=zero_y, early_start=True)
            ys.append((y, st))
        torch.cuda.synchronize()
        for i, (y, st) in enumerate(ys):
            assert int(st.item()) == 0
            ref, mag = reference(blob, 0, cols, x_vector(cols, 40 + i))
            assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - ref) <= 1e-4 * mag + 1e-30), (zero_y, i)


@pytest.mark.parametrize("n_vec", [2, 4, 8])
def test_gemv_batch_matches_oracle(n_vec):
    """Y = W X for several vectors with one decode of W, each vector's y
    against the oracle's decode of W times that vector in float64."""
    rows, cols = 48, 16384
    w = workloads.normal_tensor((rows, cols), 0.02, 40 + n_vec)
    blob = oracle.encode_layer([w])
    info = k3.layer_info(blob)
    xs = [x_vector(cols, 50 + b) for b in range(n_vec)]
    X = torch.from_numpy(np.concatenate(xs).view(np.int16)).cuda()
    Y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_blob = torch.from_numpy(blob).cuda()
    k3.gemv_layer_batch(blob[: info["hdr_bytes"]], d_blob, 0, cols, X, Y, st, zero_y=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = Y.cpu().numpy().astype(np.float64)
    for b in range(n_vec):
        ref, mag = reference(blob, 0, cols, xs[b])
        assert np.all(np.abs(got[b] - ref) <= 1e-4 * mag + 1e-30), b


def test_gemv_batch_refuses_other_counts():
    rows, cols = 8, 8192
    blob = oracle.encode_layer([workloads.normal_tensor((rows, cols), 0.02, 77)])
    info = k3.layer_info(blob)
    d_blob = torch.from_numpy(blob).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    X = torch.zeros((3, cols), dtype=torch.int16, device="cuda")
    Y = torch.zeros((3, rows), dtype=torch.float32, device="cuda")
    with pytest.raises(k3.K3HufError) as e:
        k3.gemv_layer_batch(blob[: info["hdr_bytes"]], d_blob, 0, cols, X, Y, st)
    assert e.value.code == k3.E_ARG
