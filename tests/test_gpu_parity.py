"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact: every Q4_0 / Q8_0 byte and every per-block int32 sum.
Outputs: |gpu - oracle| <= 1e-5 * sum_b |fp32(d_w d_x) isum_b| per element,
exactly zero where that sum is zero.
"""
import numpy as np
import pytest

import oracle
from q4_quantized_matmul_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def q4q():
    import __graft_entry__
    __graft_entry__.build()
    import q4_quantized_matmul_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    torch.cuda.set_device(0)
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref, scale):
    got = np.asarray(got, dtype=np.float32)
    assert got.shape == ref.shape
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = err > TOL * scale
    assert not bad.any(), "%d of %d outside tolerance; worst err %g at scale %g" % (
        bad.sum(), bad.size, err[bad].max(), scale[bad][np.argmax(err[bad])])
    zero = scale == 0
    assert np.all(got[zero] == 0)


def _special_weights(rng, ne01, ne00):
    w = (rng.standard_normal((ne01, ne00)) * 0.02).astype(np.float32)
    blocks = w.reshape(-1, 32)
    nb = blocks.shape[0]
    blocks[rng.integers(0, nb, size=max(1, nb // 10))] = 0.0                     # d = 0
    c = rng.integers(0, nb, size=max(1, nb // 10))
    blocks[c] = blocks[c, :1]                                                    # constant
    t = rng.integers(0, nb, size=max(1, nb // 10))
    k = rng.integers(-16, 16, size=(t.size, 32)).astype(np.float32)
    k[:, 0] = -16.0
    blocks[t] = k * np.float32(0.125) / 2                                         # exact .5 ties
    return w


# ---------------------------------------------------------------- quantizers --

@pytest.mark.parametrize("nrows,ncols", [(1, 32), (5, 96), (3, 768), (37, 4096), (2304, 768), (11, 14336)])
@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_quantize_bit_exact(q4q, nrows, ncols, kind):
    rng = np.random.default_rng([nrows, ncols])
    w = _special_weights(rng, nrows, ncols)
    if kind == "q8_0":
        w = w * np.float32(50.0)
    fn = q4q.q4q_quantize_q4_0 if kind == "q4_0" else q4q.q4q_quantize_q8_0
    ref = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    got = fn(dev(w)).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_quantize_misaligned_buffers(q4q, kind):
    # src offset by one float, dst by one byte: the generic (scalar) kernel
    rng = np.random.default_rng(77)
    nrows, ncols = 9, 320
    w = _special_weights(rng, nrows, ncols)
    src = torch.zeros(nrows * ncols + 1, dtype=torch.float32, device="cuda")
    src[1:] = dev(w.reshape(-1))
    bpr = ncols // 32 * (18 if kind == "q4_0" else 34)
    dst = torch.zeros(nrows * bpr + 1, dtype=torch.uint8, device="cuda")
    lib = q4q._lib.load()
    fn = lib.q4q_quantize_q4_0 if kind == "q4_0" else lib.q4q_quantize_q8_0
    import ctypes
    st = fn(ctypes.c_void_p(src.data_ptr() + 4), ctypes.c_void_p(dst.data_ptr() + 1), ncols, nrows,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    ref = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(dst[1:].cpu().numpy().reshape(nrows, bpr), ref)
    assert dst[0].item() == 0


def _near_tie_rows(rng, levels, nrows):
    """Blocks whose quotients x/d sit within a few ulps of half-integers (the
    places where round-half-away-from-zero is decided), for random scales."""
    rows = []
    for _ in range(nrows):
        amax = np.float32(rng.uniform(0.01, 100.0))
        d = np.float32(amax / np.float32(levels))
        blk = np.empty(32, np.float32)
        blk[0] = -amax if levels == 8 else amax
        for j in range(1, 32):
            k = rng.integers(-levels, levels) + 0.5
            x = np.float32(k * np.float64(d))
            for _ in range(int(rng.integers(-3, 4))):
                x = np.nextafter(x, np.float32(np.inf) if rng.random() < 0.5 else np.float32(-np.inf))
            blk[j] = x if abs(x) <= amax else np.float32(np.sign(x) * amax)
        rows.append(blk)
    return np.stack(rows).reshape(nrows // 8, 256)


def _band_edge_rows(rng, levels, nrows):
    """Blocks whose quotients x/d lie at distances 1e-6 .. 2e-3 (log-uniform, either
    side) from half-integers: across the band the kernels treat as a possible tie,
    so that a quotient approximation worse than its stated bound would round some
    of them to the wrong side."""
    rows = []
    for _ in range(nrows):
        amax = np.float32(rng.uniform(0.01, 100.0))
        d = np.float32(amax / np.float32(levels))
        blk = np.empty(32, np.float32)
        blk[0] = -amax if levels == 8 else amax
        k = rng.integers(-levels, levels, size=31) + 0.5
        delta = np.exp(rng.uniform(np.log(1e-6), np.log(2e-3), size=31)) * rng.choice([-1.0, 1.0], size=31)
        x = ((k + delta) * np.float64(d)).astype(np.float32)
        blk[1:] = np.clip(x, -amax, amax)
        rows.append(blk)
    return np.stack(rows).reshape(nrows // 8, 256)


@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_quantize_band_edges_bit_exact(q4q, kind):
    rng = np.random.default_rng(33)
    levels = 8 if kind == "q4_0" else 127
    w = _band_edge_rows(rng, levels, 8192)
    fn = q4q.q4q_quantize_q4_0 if kind == "q4_0" else q4q.q4q_quantize_q8_0
    ref = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(fn(dev(w)).cpu().numpy(), ref)


def test_mul_mat_band_edge_activations(q4q):
    # Q4_0 weights with a single nonzero code per block (+1 at one element), so that
    # every output isolates activation codes: a code off by one changes the output
    # by d_w * d_x, far above the tolerance
    rng = np.random.default_rng(34)
    ne00, ne01 = 4096, 64
    x = _band_edge_rows(rng, 127, 16 * ne00 // 32).reshape(16, ne00)
    wq_rows = np.zeros((ne01, ne00 // 32, 18), np.uint8)
    wq_rows[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    wq_rows[:, :, 2:] = 0x88                                      # every nibble 8: value 0
    sel = rng.integers(0, 32, size=(ne01, ne00 // 32))
    for r in range(ne01):
        for b in range(ne00 // 32):
            j = sel[r, b]
            byte = 2 + j // 2
            wq_rows[r, b, byte] = (0x89 if j % 2 == 0 else 0x98)    # nibble 9: value +1 * d
    wq = wq_rows.reshape(-1)
    for ne11 in (1, 3, 7, 16):
        got = q4q.q4q_mul_mat(dev(wq), ne00, ne01, dev(x[:ne11])).cpu().numpy()
        ref, scale = oracle.mul_mat(wq, ne00, ne01, x[:ne11])
        assert_close(got, ref, scale)


@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_quantize_near_ties_bit_exact(q4q, kind):
    rng = np.random.default_rng(31)
    levels = 8 if kind == "q4_0" else 127
    w = _near_tie_rows(rng, levels, 4096)
    fn = q4q.q4q_quantize_q4_0 if kind == "q4_0" else q4q.q4q_quantize_q8_0
    ref = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(fn(dev(w)).cpu().numpy(), ref)


def test_mul_mat_near_tie_activations(q4q):
    # the activation quantization inside both mul_mat paths meets the same ties
    rng = np.random.default_rng(32)
    x = _near_tie_rows(rng, 127, 512).reshape(-1, 1024)
    assert x.shape == (16, 1024)
    ne00 = 1024
    w = (rng.standard_normal((300, ne00)) * 0.02).astype(np.float32)
    wq = oracle.quantize_q4_0(w)
    for ne11 in (1, 3, 16):
        got = q4q.q4q_mul_mat(dev(wq), ne00, 300, dev(x[:ne11])).cpu().numpy()
        ref, scale = oracle.mul_mat(wq, ne00, 300, x[:ne11])
        assert_close(got, ref, scale)
    xq = oracle.quantize_q8_0(x[:16])
    for path in (0, 1):
        got = q4q.q4q_debug_block_isums(dev(wq), dev(xq), ne00, 300, 16, path=path).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.block_isums(wq, xq, ne00, 300, 16))


def test_quantize_hand_block(q4q):
    w = ((np.arange(32) - 16) * 0.25).astype(np.float32).reshape(1, 32)
    got = q4q.q4q_quantize_q4_0(dev(w)).cpu().numpy()
    assert bytes(got[0]) == bytes.fromhex("0038001122334455667798a9bacbdcedfeff")


# ------------------------------------------------------------ block int sums --

@pytest.mark.parametrize("ne00,ne01,ne11", [(64, 1, 1), (256, 5, 3), (768, 37, 2), (4096, 9, 1), (160 * 2, 4, 4)])
def test_block_isums_gemv_routine(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 1])
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[:, ::7] *= 30
    wq = oracle.quantize_q4_0(w)
    xq = oracle.quantize_q8_0(x)
    ref = oracle.block_isums(wq, xq, ne00, ne01, ne11)
    got = q4q.q4q_debug_block_isums(dev(wq), dev(xq), ne00, ne01, ne11, path=0).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def test_block_isums_extremes(q4q):
    # nibble 0 (-8) against -127 and nibble 15 (+7) against +127 in every position
    ne00, ne01, ne11 = 64, 2, 2
    wq = np.zeros((ne01, 2 * 18), np.uint8)
    wq[0, 2:18] = 0x00
    wq[0, 20:36] = 0xFF
    wq[1, 2:18] = 0xF0
    wq[1, 20:36] = 0x0F
    xq = np.zeros((ne11, 2 * 34), np.uint8)
    xq[0, 2:34] = np.int8(-127).view(np.uint8)
    xq[0, 36:68] = np.int8(127).view(np.uint8)
    xq[1, 2:34] = np.int8(127).view(np.uint8)
    xq[1, 36:68] = np.int8(-127).view(np.uint8)
    ref = oracle.block_isums(wq, xq, ne00, ne01, ne11)
    assert ref[0, 0, 0] == 32 * 8 * 127
    got = q4q.q4q_debug_block_isums(dev(wq), dev(xq), ne00, ne01, ne11, path=0).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("ne00,ne01,ne11", [(256, 1, 1), (256, 5, 3), (512, 130, 9), (1024, 200, 17),
                                            (4096, 64, 40), (768, 37, 130)])
def test_block_isums_mma_routine(q4q, ne00, ne01, ne11):
    # one 32-wide K block per fresh TMEM accumulator, read back as exact integers
    rng = np.random.default_rng([ne00, ne01, ne11, 4])
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[:, ::5] *= 40
    wq = oracle.quantize_q4_0(w)
    xq = oracle.quantize_q8_0(x)
    ref = oracle.block_isums(wq, xq, ne00, ne01, ne11)
    got = q4q.q4q_debug_block_isums(dev(wq), dev(xq), ne00, ne01, ne11, path=1).cpu().numpy()
    np.testing.assert_array_equal(got, ref)
    assert q4q.q4q_device_status() == 0


def test_block_isums_mma_extremes(q4q):
    ne00, ne01, ne11 = 256, 3, 2
    wq = np.zeros((ne01, 8 * 18), np.uint8)
    wq[0, :] = 0x00
    wq[1, :] = 0xFF
    wq[2, :] = 0x0F
    xq = np.zeros((ne11, 8 * 34), np.uint8)
    xq[0, :] = np.int8(-127).view(np.uint8)
    xq[1, :] = np.int8(127).view(np.uint8)
    ref = oracle.block_isums(wq, xq, ne00, ne01, ne11)
    got = q4q.q4q_debug_block_isums(dev(wq), dev(xq), ne00, ne01, ne11, path=1).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------- mul_mat --

# (14336, 1): a CTA pair where one CTA has no rows; (8448, 129), (2816, 50) at 7
# tokens: pairs whose two halves of the blocks split inside a token; (4096, 1216): one
# full 8-row unit on each of 152 CTAs (one dot pass), (4096, 1217): one row more, two
# units a CTA again; (768, 153): one row past one-row units
GEMV_SHAPES = [(256, 1), (256, 3), (768, 2304), (768, 1000), (3072, 768), (4096, 1024), (14336, 64),
               (512, 33), (1024, 4099), (14336, 1), (8448, 129), (2816, 50), (4096, 1216), (4096, 1217),
               (768, 153)]


@pytest.mark.parametrize("ne00,ne01", GEMV_SHAPES)
@pytest.mark.parametrize("ne11", [1, 2, 7])
def test_mul_mat_gemv(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 2])
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    wq_d = q4q.q4q_quantize_q4_0(dev(w))
    got = q4q.q4q_mul_mat(wq_d, ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(oracle.quantize_q4_0(w), ne00, ne01, x, nthreads=8)
    assert_close(got, ref, scale)


@pytest.mark.parametrize("ne00,ne01,ne11", [(32, 3, 1), (96, 17, 2), (800, 65, 5), (160, 40, 9), (256, 70, 8),
                                            (768, 130, 17), (4096, 64, 16)])
def test_mul_mat_other_paths(q4q, ne00, ne01, ne11):
    # ne00 % 256 != 0 (generic path) and ne11 >= 8 (GEMM path where it applies)
    rng = np.random.default_rng([ne00, ne01, ne11, 3])
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    got = q4q.q4q_mul_mat(q4q.q4q_quantize_q4_0(dev(w)), ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(oracle.quantize_q4_0(w), ne00, ne01, x, nthreads=8)
    assert_close(got, ref, scale)


MMA_SHAPES = [(256, 128, 8), (512, 300, 16), (768, 130, 17), (4096, 1024, 64), (4096, 257, 129), (1024, 64, 200),
              (14336, 256, 512)]


@pytest.mark.parametrize("ne00,ne01,ne11", MMA_SHAPES)
def test_mul_mat_tensor_core(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 5])
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[ne11 // 2] = 0.0
    got = q4q.q4q_mul_mat(q4q.q4q_quantize_q4_0(dev(w)), ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(oracle.quantize_q4_0(w), ne00, ne01, x, nthreads=8)
    assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0


def _min_mma_workspace(ne00, ne11):
    # the split-free minimum of the tensor-core path: fp16 operand + block scales + control word
    return (ne11 * ne00 * 2 + 255) // 256 * 256 + (ne00 // 32) * ((ne11 + 127) // 128 * 128) * 4 + 256


@pytest.mark.parametrize("ne00,ne01,ne11,split", [(4096, 1024, 8, True), (4096, 300, 64, True),
                                                  (14336, 256, 16, True), (1024, 64, 200, False)])
@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_mul_mat_split_k(q4q, ne00, ne01, ne11, split, kind):
    """Split-K (few output tiles): with the workspace q4q_mul_mat_workspace_size asks for,
    the K loop is split and the partial sums added in order; with the split-free minimum
    it runs unsplit.  Both are within tolerance of the oracle."""
    rng = np.random.default_rng([ne00, ne01, ne11, 11])
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[ne11 // 3] = 0.0
    if kind == "q4_0":
        wq = oracle.quantize_q4_0(w)
        full = q4q.q4q_mul_mat_workspace_size(ne00, ne01, ne11)
        call = q4q.q4q_mul_mat
        ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    else:
        wq = oracle.quantize_q8_0(w)
        full = q4q.q4q_mul_mat_q8_0_workspace_size(ne00, ne01, ne11)
        call = q4q.q4q_mul_mat_q8_0
        ref, scale = oracle.mul_mat_w8(wq, ne00, ne01, x, nthreads=8)
    least = _min_mma_workspace(ne00, ne11)
    assert (full > least) == split
    wq_d, x_d = dev(wq), dev(x)
    for nbytes in (full, least):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        got = call(wq_d, ne00, ne01, x_d, workspace=ws).cpu().numpy()
        assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0


def test_mul_mat_pdl_chain(q4q):
    # y1 = W1 x, y2 = W2 y1, y3 = W3 y2 with programmatic dependent launch: every
    # call must see its predecessor's output (same kernels, so results are identical)
    rng = np.random.default_rng(9)
    dims = [1024, 2048, 768, 1536]
    ws = [q4q.q4q_quantize_q4_0(dev((rng.standard_normal((dims[i + 1], dims[i])) * 0.02).astype(np.float32)))
          for i in range(3)]
    x = dev(rng.standard_normal((1, dims[0])).astype(np.float32))
    outs = {}
    for flags in (0, q4q.Q4Q_MUL_MAT_PDL):
        y = x
        for i in range(3):
            y = q4q.q4q_mul_mat(ws[i], dims[i], dims[i + 1], y, flags=flags)
        outs[flags] = y.cpu().numpy()
    np.testing.assert_array_equal(outs[0], outs[q4q.Q4Q_MUL_MAT_PDL])
    # and every step against the oracle at the 1e-5 S bar, on the input the GPU step read
    y = x
    for i in range(3):
        got = q4q.q4q_mul_mat(ws[i], dims[i], dims[i + 1], y, flags=q4q.Q4Q_MUL_MAT_PDL)
        ref, scale = oracle.mul_mat(ws[i].cpu().numpy(), dims[i], dims[i + 1], y.cpu().numpy())
        assert_close(got.cpu().numpy(), ref, scale)
        y = got
    np.testing.assert_array_equal(y.cpu().numpy(), outs[0])


def test_mul_mat_misaligned_weights_take_generic_path(q4q):
    ne00, ne01, ne11 = 512, 40, 1
    rng = np.random.default_rng(5)
    w = _special_weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    wq = oracle.quantize_q4_0(w)
    buf = torch.zeros(wq.size + 2, dtype=torch.uint8, device="cuda")
    buf[2:] = dev(wq.reshape(-1))
    src0 = buf[2:]
    assert src0.data_ptr() % 16 != 0
    got = q4q.q4q_mul_mat(src0, ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x)
    assert_close(got, ref, scale)


def test_mul_mat_zero_rows_and_tokens(q4q):
    ne00, ne01, ne11 = 1024, 50, 3
    rng = np.random.default_rng(6)
    w = _special_weights(rng, ne01, ne00)
    w[7] = 0.0
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[1] = 0.0
    got = q4q.q4q_mul_mat(q4q.q4q_quantize_q4_0(dev(w)), ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(oracle.quantize_q4_0(w), ne00, ne01, x)
    assert np.all(got[1] == 0) and np.all(got[:, 7] == 0)
    assert_close(got, ref, scale)


def test_mul_mat_hand_block(q4q):
    w = ((np.arange(32) - 16) * 0.25).astype(np.float32)
    w = np.tile(w, 8).reshape(1, 256)
    x = np.ones((1, 256), np.float32)
    got = q4q.q4q_mul_mat(q4q.q4q_quantize_q4_0(dev(w)), 256, 1, dev(x)).cpu().numpy()
    assert got[0, 0] == np.float32(8 * -4.499725341796875)


def test_mul_mat_empty(q4q):
    wq = torch.zeros(18 * 8, dtype=torch.uint8, device="cuda")
    out = q4q.q4q_mul_mat(wq, 256, 0, torch.zeros(3, 256, device="cuda"))
    assert out.shape == (3, 0)
    out = q4q.q4q_mul_mat(wq, 256, 1, torch.zeros(0, 256, device="cuda"))
    assert out.shape == (0, 1)


def test_no_device_errors_recorded(q4q):
    assert q4q.q4q_device_status() == 0


def test_bounded_wait_reports_timeout_and_context_stays_usable(q4q):
    # a wait that nothing completes gives up after 2 ms and records Q4Q_ERR_TIMEOUT;
    # the status is read (and cleared) on the host, and the next call works
    assert q4q.q4q_device_status() == 0
    q4q.q4q_debug_wait_timeout(2_000_000)
    assert q4q.q4q_device_status() == 6
    assert q4q.q4q_device_status() == 0
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((300, 1024)) * 0.02).astype(np.float32)
    x = rng.standard_normal((1, 1024)).astype(np.float32)
    wq = oracle.quantize_q4_0(w)
    got = q4q.q4q_mul_mat(dev(wq), 1024, 300, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(wq, 1024, 300, x)
    assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0


# ---------------------------------------------------- full-size workloads ----

def _sample_rows(ne01, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(ne01, size=min(n, ne01), replace=False), [0, ne01 - 1]]))
    return rows


@pytest.mark.parametrize("name", ["gpt2_c_attn_1tok", "gpt2_decode_step", "llama3_8b_decode"])
def test_full_size_decode_workloads(q4q, name):
    """Every distinct matrix of the workload at full size, in the launch
    configuration the benchmark times: Q4_0 bytes bit-exact and outputs within
    tolerance on up to 4096 sampled rows (plus the first and last) for every token."""
    wl = workloads.WORKLOADS[name]
    seen = set()
    for i, (ne00, ne01) in enumerate(wl.shapes):
        if name == "gpt2_decode_step" and (ne00, ne01) in seen:
            continue           # the 12 layers repeat 4 shapes; one of each + lm_head
        seen.add((ne00, ne01))
        w, x = workloads.problem(name, i)
        wq_d = q4q.q4q_quantize_q4_0(dev(w))
        got = q4q.q4q_mul_mat(wq_d, ne00, ne01, dev(x)).cpu().numpy()
        rows = _sample_rows(ne01, 4096, i)
        wq_rows = oracle.quantize_q4_0(w[rows])
        np.testing.assert_array_equal(wq_d.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy(), wq_rows)
        ref, scale = oracle.mul_mat(wq_rows, ne00, rows.size, x, nthreads=8)
        assert_close(got[:, rows], ref, scale)
    assert q4q.q4q_device_status() == 0


@pytest.mark.parametrize("name,ne11", [("llama3_8b_batched", 8), ("llama3_8b_batched", 64),
                                       ("llama3_8b_batched", 512), ("stress_prefill", 2048)])
def test_full_size_batched_workloads(q4q, name, ne11):
    """The tensor-core path at full size: every matrix of the workload, outputs on
    up to 1024 sampled rows (plus first and last) for every token."""
    wl = workloads.WORKLOADS[name]
    for i, (ne00, ne01) in enumerate(wl.shapes):
        if name == "llama3_8b_batched" and i in (2, 3, 5):
            continue           # v = k, o = q, up = gate in shape
        w, x = workloads.problem(name, i, ne11)
        wq_d = q4q.q4q_quantize_q4_0(dev(w))
        got = q4q.q4q_mul_mat(wq_d, ne00, ne01, dev(x)).cpu().numpy()
        rows = _sample_rows(ne01, 1024, 100 + i)
        wq_rows = wq_d.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy()
        np.testing.assert_array_equal(wq_rows, oracle.quantize_q4_0(w[rows]))
        ref, scale = oracle.mul_mat(wq_rows, ne00, rows.size, x, nthreads=16)
        assert_close(got[:, rows], ref, scale)
        del wq_d
    assert q4q.q4q_device_status() == 0


# ------------------------------------------------------------ tiny block scales --

def _tiny_scale_rows(rng, levels, nblocks):
    """Blocks whose scale d32 = amax / levels sits around the smallest fp16 normal
    (2^-14) and the smallest fp16 subnormal (2^-24, with 2^-25 rounding to zero),
    blocks whose amax is itself an fp32 subnormal (d32 may underflow to zero; a
    reciprocal that flushes subnormals gives infinity, so the exact division must
    decide), and blocks just above the smallest fp32 normal.  Each block holds
    +-amax, exact ties (k + 1/2) d32 where they are representable, and uniform
    values."""
    lo_hi = [(-16.0, -13.0), (-27.0, -23.0), (-149.0 + np.log2(levels), -126.0), (-126.0, -120.0)]
    exact = [2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14 * (1 - 2.0 ** -11)]
    out = np.empty((nblocks, 32), np.float32)
    for i in range(nblocks):
        if i < len(exact) * 4:
            d = exact[i % len(exact)]
            amax = np.float32(d * levels)
        else:
            lo, hi = lo_hi[i % len(lo_hi)]
            amax = np.float32(2.0 ** rng.uniform(lo, hi) * (levels if hi > -126.0 else 1.0))
        d32 = np.float32(amax / np.float32(levels))
        blk = (rng.uniform(-1.0, 1.0, 32) * np.float64(amax)).astype(np.float32)
        blk[rng.integers(0, 32)] = amax if rng.random() < 0.5 else -amax
        if d32 > 0:
            k = rng.integers(-levels, levels, size=6) + 0.5
            t = (k * np.float64(d32)).astype(np.float32)
            ok = (np.abs(t) <= amax) & (t.astype(np.float64) == k * np.float64(d32))
            blk[1:7][ok] = t[ok]
        out[i] = blk
    return out


@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_quantize_tiny_scales_bit_exact(q4q, kind):
    import ctypes
    levels = 8 if kind == "q4_0" else 127
    rng = np.random.default_rng(71 + levels)
    w = _tiny_scale_rows(rng, levels, 4096).reshape(-1, 256)
    assert np.any(w != 0) and np.any((np.abs(w) < 2.0 ** -126) & (w != 0))
    fn = q4q.q4q_quantize_q4_0 if kind == "q4_0" else q4q.q4q_quantize_q8_0
    ref = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(fn(dev(w)).cpu().numpy(), ref)
    # the same rows through the scalar kernel (misaligned buffers)
    nrows, ncols = w.shape
    src = torch.zeros(w.size + 1, dtype=torch.float32, device="cuda")
    src[1:] = dev(w.reshape(-1))
    bpr = ncols // 32 * (18 if kind == "q4_0" else 34)
    dst = torch.zeros(nrows * bpr + 1, dtype=torch.uint8, device="cuda")
    lib = q4q._lib.load()
    cfn = lib.q4q_quantize_q4_0 if kind == "q4_0" else lib.q4q_quantize_q8_0
    assert cfn(ctypes.c_void_p(src.data_ptr() + 4), ctypes.c_void_p(dst.data_ptr() + 1), ncols, nrows,
               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    np.testing.assert_array_equal(dst[1:].cpu().numpy().reshape(nrows, bpr), ref)


def test_mul_mat_tiny_activation_scales(q4q):
    # The activation quantization fused into the GEMV (1..7 tokens) and into the
    # tensor-core path's operand kernel (16 tokens) on tiny-scale blocks, against
    # weights with one nonzero code per block so that every output isolates codes.
    rng = np.random.default_rng(72)
    ne00, ne01 = 4096, 64
    x = _tiny_scale_rows(rng, 127, 16 * ne00 // 32).reshape(16, ne00)
    # token 2: every block scale below half the smallest fp16 subnormal, so every
    # d_x is stored as zero (nonzero codes, S = 0): those outputs must be exactly 0
    x[2] = (x[2].astype(np.float64) * 2.0 ** -120).astype(np.float32)
    wq_rows = np.zeros((ne01, ne00 // 32, 18), np.uint8)
    wq_rows[:, :, 0:2] = np.frombuffer(np.float16(0.5).tobytes(), np.uint8)
    wq_rows[:, :, 2:] = 0x88
    sel = rng.integers(0, 32, size=(ne01, ne00 // 32))
    for r in range(ne01):
        for b in range(ne00 // 32):
            j = sel[r, b]
            wq_rows[r, b, 2 + j // 2] = (0x8F if j % 2 == 0 else 0xF8)    # nibble 15: value +7 d
    wq = wq_rows.reshape(-1)
    for ne11 in (1, 3, 7, 16):
        got = q4q.q4q_mul_mat(dev(wq), ne00, ne01, dev(x[:ne11])).cpu().numpy()
        ref, scale = oracle.mul_mat(wq, ne00, ne01, x[:ne11])
        assert np.all(scale[:2] > 0) and (ne11 < 3 or np.all(scale[2] == 0))
        assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0


# --------------------------------------------- the kernels' own bounded waits --

@pytest.mark.parametrize("path,ne00,ne01,ne11", [(0, 4096, 1024, 1), (0, 1024, 300, 3), (0, 4096, 128256, 1),
                                                 (1, 4096, 1024, 16), (1, 1024, 256, 130), (1, 4096, 2048, 64),
                                                 (3, 4096, 1024, 8), (3, 1024, 300, 32), (3, 4096, 128256, 2)])
def test_kernel_timeout_path(q4q, path, ne00, ne01, ne11):
    """A matmul kernel whose first CTA never receives its first stage (a hand-off left
    out on purpose, with every wait bounded by 5 ms): the waits run out, the device
    status reports Q4Q_ERR_TIMEOUT once, and the CTAs wind down (their copies landed,
    tensor memory freed), so the same kernel then runs normally, twice in a row, and
    matches the oracle.  No GPU fault or hang is involved."""
    assert q4q.q4q_device_status() == 0
    rng = np.random.default_rng([path, ne00, ne01, ne11])
    w = (rng.standard_normal((ne01, ne00)) * 0.02).astype(np.float32)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    wq_d = q4q.q4q_quantize_q4_0(dev(w))
    x_d = dev(x)
    q4q.q4q_debug_mul_mat_timeout(wq_d, ne00, ne01, x_d, path, 5_000_000)
    assert q4q.q4q_device_status() == 6
    assert q4q.q4q_device_status() == 0
    rows = _sample_rows(ne01, 2048, 7)
    ref, scale = oracle.mul_mat(wq_d.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy(), ne00, rows.size, x,
                                nthreads=8)
    for _ in range(2):
        got = q4q.q4q_mul_mat(wq_d, ne00, ne01, x_d).cpu().numpy()
        assert_close(got[:, rows], ref, scale)
    assert q4q.q4q_device_status() == 0


def test_kernel_timeout_argument_errors(q4q):
    wq = torch.zeros(64 * 8 * 18, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 256), device="cuda")
    with pytest.raises(q4q.Q4QError):            # path 1 needs ne11 >= 8
        q4q.q4q_debug_mul_mat_timeout(wq, 256, 64, x, 1, 1_000_000)
    with pytest.raises(q4q.Q4QError):            # limit above one second
        q4q.q4q_debug_mul_mat_timeout(wq, 256, 64, x, 0, 2_000_000_000)
    with pytest.raises(q4q.Q4QError):            # unknown path
        q4q.q4q_debug_mul_mat_timeout(wq, 256, 64, x, 4, 1_000_000)
    with pytest.raises(q4q.Q4QError):            # path 3 takes at most 32 tokens
        q4q.q4q_debug_mul_mat_timeout(wq, 256, 64, torch.zeros((33, 256), device="cuda"), 3, 1_000_000)
    assert q4q.q4q_device_status() == 0


def test_mul_mat_tensor_core_weight_scale_extremes(q4q):
    """The tensor-core path at 130 tokens (128-token tiles) on rows that mix blocks whose
    stored weight scales are fp16 subnormals, ordinary, exactly 8188, exactly 8192 and far
    above (weights up to ~1e5, block scales up to ~5e4): every output within 1e-5 S of
    the oracle."""
    rng = np.random.default_rng(91)
    ne00, ne01, ne11 = 1024, 256, 130
    z = rng.standard_normal((ne01, ne00 // 32, 32))
    scales = np.array([3e-7, 2e-5, 1e-3, 0.02, 1.0, 300.0, 4e4, 1.2e5])
    pick = rng.integers(0, scales.size, size=(ne01, ne00 // 32))
    w = (z * scales[pick][..., None]).astype(np.float32)
    # blocks whose stored scale is exactly 8188 (amax 65504) and exactly 8192 (amax 65536)
    w[3, :, :] = 0.0
    w[3, :, 0] = 65504.0
    w[3, :, 1:] = rng.uniform(-65504.0, 65504.0, size=(ne00 // 32, 31)).astype(np.float32)
    w[4, :, 0] = -65536.0
    w = w.reshape(ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[5] = 0.0
    wq = oracle.quantize_q4_0(w)
    d = oracle.f32_from_fp16(wq.reshape(-1, 18)[:, :2].copy().view(np.uint16).reshape(-1))
    assert np.any(d > 8188) and np.any((d > 0) & (d < 2.0 ** -14)) and np.any(d == 8188) and np.any(d == 8192)
    got = q4q.q4q_mul_mat(dev(wq), ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0
