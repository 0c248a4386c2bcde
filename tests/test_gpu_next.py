"""GPU parity of the operations next to the matmul, through the C ABI, against
the CPU oracle: the Q4_0 / Q8_0 row gather, the bias / GELU and SwiGLU
epilogues, and the Q8_0-weight matmul.

Bars:
  * get_rows: bit-exact (the decode (nibble - 8) * d, resp. q * d, is exact in fp32).
  * Q8_0-weight block sums: bit-exact; outputs within 1e-5 * S, S = sum_b
    |fp32(d_w d_x) isum_b|, exactly zero where S is zero (the matmul's own bar).
  * bias: the matmul's error (1e-5 * S) plus one fp32 rounding of the add on each
    side (2^-23 |ref|).
  * GELU: the pre-activation error above times max |GELU'| (< 1.13), plus the fp32
    evaluation: erfcf (<= 4 ulp) of an argument rounded once, which moves erfc by
    up to 2 x^2 ulp for x = v / sqrt 2 (x^2 < 85 before erfc underflows), so
    1e-5 |ref|; 1e-30 absolute for the underflowed tail.
  * SwiGLU: |silu(g') u' - silu(g) u| <= max|silu'| (< 1.1) e_g (|u| + e_u) +
    |silu(g)| e_u with e_g = 1e-5 S_g and e_u = 1e-5 S_u, plus 1e-6 |ref| for the
    fp32 evaluation (expf, add, divide, multiply: a few ulp); exactly zero where
    S_g or S_u is zero.
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


def _check(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float32)
    assert got.shape == ref.shape, what
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = err > tol
    assert not bad.any(), "%s: %d of %d outside tolerance; worst err %g (tol %g)" % (
        what, bad.sum(), bad.size, err[bad].max(), tol[bad][np.argmax(err[bad])])


def _weights(rng, ne01, ne00, scale=0.02):
    w = (rng.standard_normal((ne01, ne00)) * scale).astype(np.float32)
    blocks = w.reshape(-1, 32)
    nb = blocks.shape[0]
    blocks[rng.integers(0, nb, size=max(1, nb // 10))] = 0.0          # d = 0 blocks
    c = rng.integers(0, nb, size=max(1, nb // 10))
    blocks[c] = blocks[c, :1]                                         # constant blocks
    return w


def _sample_rows(ne01, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(ne01, size=min(n, ne01), replace=False), [0, ne01 - 1]]))


# ---------------------------------------------------------------- get_rows --

@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
@pytest.mark.parametrize("ne00,ne01,n_ids", [(32, 5, 7), (96, 13, 20), (768, 50257, 9), (4096, 1000, 513),
                                             (14336, 3, 5)])
def test_get_rows_bit_exact(q4q, kind, ne00, ne01, n_ids):
    rng = np.random.default_rng([ne00, ne01, n_ids])
    w = _weights(rng, ne01, ne00)
    quant = oracle.quantize_q4_0 if kind == "q4_0" else oracle.quantize_q8_0
    table = quant(w)
    ids = rng.integers(0, ne01, size=n_ids).astype(np.int32)
    ids[0], ids[-1] = 0, ne01 - 1
    if n_ids > 3:
        ids[1] = ids[2]                                               # a repeated token
    fn = q4q.q4q_get_rows_q4_0 if kind == "q4_0" else q4q.q4q_get_rows_q8_0
    got = fn(dev(table), ne00, ne01, ids=dev(ids)).cpu().numpy()
    ref, ok = oracle.get_rows(table, ne00, ids, kind)
    assert ok
    np.testing.assert_array_equal(got, ref)
    assert q4q.q4q_device_status() == 0


@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_get_rows_whole_table_and_bad_ids(q4q, kind):
    rng = np.random.default_rng(51)
    ne00, ne01 = 256, 37
    w = _weights(rng, ne01, ne00)
    table = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    fn = q4q.q4q_get_rows_q4_0 if kind == "q4_0" else q4q.q4q_get_rows_q8_0
    # ids = NULL: rows 0 .. n-1, i.e. the decode of the table
    got = fn(dev(table), ne00, ne01).cpu().numpy()
    deq = oracle.dequantize_q4_0(table, ne00) if kind == "q4_0" else oracle.dequantize_q8_0(table, ne00)
    np.testing.assert_array_equal(got, deq)
    assert q4q.q4q_device_status() == 0
    # ids outside [0, ne01): zero rows, the table is not read there, and the device status says so
    ids = np.array([3, ne01, -1, 36, 2 ** 31 - 1], np.int32)
    out = torch.full((ids.size, ne00), 7.0, device="cuda")
    fn(dev(table), ne00, ne01, ids=dev(ids), dst=out)
    got = out.cpu().numpy()
    ref, ok = oracle.get_rows(table, ne00, ids, kind)
    assert not ok
    np.testing.assert_array_equal(got, ref)
    assert q4q.q4q_device_status() == 7            # Q4Q_ERR_ARG, then cleared
    assert q4q.q4q_device_status() == 0


def test_get_rows_full_size_token_embedding(q4q):
    # the Llama-3-8B-shaped token embedding 4096 x 128256 stored as Q4_0, 512 token ids
    ne00, ne01 = 4096, 128256
    w, _ = workloads.problem("llama3_8b_decode", 7)                  # an lm_head-shaped table
    table = q4q.q4q_quantize_q4_0(dev(w))
    rng = np.random.default_rng(52)
    ids = rng.integers(0, ne01, size=512).astype(np.int32)
    got = q4q.q4q_get_rows_q4_0(table, ne00, ne01, ids=dev(ids)).cpu().numpy()
    rows = table.view(ne01, -1)[torch.from_numpy(ids.astype(np.int64)).cuda()].cpu().numpy()
    np.testing.assert_array_equal(rows, oracle.quantize_q4_0(w[ids]))
    ref, ok = oracle.get_rows(rows, ne00, np.arange(ids.size, dtype=np.int32))
    assert ok
    np.testing.assert_array_equal(got, ref)


# --------------------------------------------------------- bias / GELU ------

BIAS_SHAPES = [(256, 3, 1), (768, 2304, 1), (768, 3072, 2), (3072, 768, 7), (4096, 1000, 1), (14336, 64, 1),
               (1024, 4099, 3), (768, 130, 17), (4096, 257, 64), (96, 17, 2), (800, 65, 9)]


@pytest.mark.parametrize("ne00,ne01,ne11", BIAS_SHAPES)
@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("with_bias", [True, False])
def test_mul_mat_bias_act(q4q, ne00, ne01, ne11, act, with_bias):
    if not with_bias and act == 0:
        pytest.skip("plain mul_mat")
    rng = np.random.default_rng([ne00, ne01, ne11, act, with_bias])
    w = _weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    bias = (rng.standard_normal(ne01) * 0.5).astype(np.float32) if with_bias else None
    wq = oracle.quantize_q4_0(w)
    got = q4q.q4q_mul_mat_bias_act(dev(wq), ne00, ne01, dev(x), bias=dev(bias) if with_bias else None,
                                   act=act).cpu().numpy()
    ref, pre, scale = oracle.mul_mat_epilogue(wq, ne00, ne01, x, bias=bias, act=act, nthreads=8)
    e_pre = TOL * scale + 2.0 ** -23 * np.abs(pre)
    tol = e_pre if act == 0 else 1.13 * e_pre + 1e-5 * np.abs(ref) + 1e-30
    _check(got, ref, tol, "bias=%s act=%d" % (with_bias, act))
    assert q4q.q4q_device_status() == 0


def test_mul_mat_bias_act_pdl_chain(q4q):
    # GPT-2 MLP at one token, PDL-chained: fc (+ bias, GELU) then proj (+ bias)
    rng = np.random.default_rng(53)
    wfc = q4q.q4q_quantize_q4_0(dev((rng.standard_normal((3072, 768)) * 0.02).astype(np.float32)))
    wpj = q4q.q4q_quantize_q4_0(dev((rng.standard_normal((768, 3072)) * 0.02).astype(np.float32)))
    bfc = dev((rng.standard_normal(3072) * 0.1).astype(np.float32))
    bpj = dev((rng.standard_normal(768) * 0.1).astype(np.float32))
    x = dev(rng.standard_normal((1, 768)).astype(np.float32))
    outs = {}
    for flags in (0, q4q.Q4Q_MUL_MAT_PDL):
        h = q4q.q4q_mul_mat_bias_act(wfc, 768, 3072, x, bias=bfc, act=q4q.Q4Q_ACT_GELU, flags=flags)
        y = q4q.q4q_mul_mat_bias_act(wpj, 3072, 768, h, bias=bpj, flags=flags)
        outs[flags] = (h.cpu().numpy(), y.cpu().numpy())
    np.testing.assert_array_equal(outs[0][0], outs[q4q.Q4Q_MUL_MAT_PDL][0])
    np.testing.assert_array_equal(outs[0][1], outs[q4q.Q4Q_MUL_MAT_PDL][1])
    # each step against the oracle on the same input the GPU step read, at the
    # epilogue's own bar (the matmul's 1e-5 S, one fp32 rounding of the bias add,
    # GELU's slope and its own error)
    h_gpu, y_gpu = outs[0]
    ref_h, pre_h, s_h = oracle.mul_mat_epilogue(wfc.cpu().numpy(), 768, 3072, x.cpu().numpy(), bias=bfc.cpu().numpy(),
                                                act=oracle.ACT_GELU)
    e_h = TOL * s_h + 2.0 ** -23 * np.abs(pre_h)
    _check(h_gpu, ref_h, 1.13 * e_h + 1e-5 * np.abs(ref_h) + 1e-30, "pdl fc")
    ref_y, pre_y, s_y = oracle.mul_mat_epilogue(wpj.cpu().numpy(), 3072, 768, h_gpu, bias=bpj.cpu().numpy())
    _check(y_gpu, ref_y, TOL * s_y + 2.0 ** -23 * np.abs(pre_y), "pdl proj")


# ------------------------------------------------------------------ SwiGLU --

SWIGLU_SHAPES = [(256, 3, 1), (4096, 1000, 1), (4096, 1000, 2), (4096, 1000, 7), (768, 3072, 1), (3072, 768, 3),
                 (14336, 64, 1), (1024, 4099, 1), (512, 33, 5), (1024, 300, 8), (768, 130, 17), (4096, 257, 64),
                 (96, 17, 2), (800, 65, 1)]


def _swiglu_tol(ref, g, u, sg, su):
    eg, eu = TOL * sg, TOL * su
    s = np.abs(g.astype(np.float64)) / (1.0 + np.exp(-np.clip(g.astype(np.float64), -700, 700)))
    return 1.1 * eg * (np.abs(u) + eu) + eu * s + 1e-6 * np.abs(ref) + 1e-30


@pytest.mark.parametrize("ne00,ne01,ne11", SWIGLU_SHAPES)
def test_mul_mat_swiglu(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 60])
    wg, wu = _weights(rng, ne01, ne00), _weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    if ne11 > 2:
        x[1] = 0.0
    gq, uq = oracle.quantize_q4_0(wg), oracle.quantize_q4_0(wu)
    got = q4q.q4q_mul_mat_swiglu(dev(gq), dev(uq), ne00, ne01, dev(x)).cpu().numpy()
    ref, g, u, sg, su = oracle.mul_mat_swiglu(gq, uq, ne00, ne01, x, nthreads=8)
    _check(got, ref, _swiglu_tol(ref, g, u, sg, su), "swiglu")
    zero = (sg == 0) | (su == 0)
    assert np.all(got[zero] == 0)
    assert q4q.q4q_device_status() == 0


def test_mul_mat_swiglu_misaligned_takes_the_two_pass_path(q4q):
    rng = np.random.default_rng(61)
    ne00, ne01 = 512, 40
    wg, wu = _weights(rng, ne01, ne00), _weights(rng, ne01, ne00)
    x = rng.standard_normal((1, ne00)).astype(np.float32)
    gq, uq = oracle.quantize_q4_0(wg), oracle.quantize_q4_0(wu)
    buf = torch.zeros(uq.size + 2, dtype=torch.uint8, device="cuda")
    buf[2:] = dev(uq.reshape(-1))
    got = q4q.q4q_mul_mat_swiglu(dev(gq), buf[2:], ne00, ne01, dev(x)).cpu().numpy()
    ref, g, u, sg, su = oracle.mul_mat_swiglu(gq, uq, ne00, ne01, x)
    _check(got, ref, _swiglu_tol(ref, g, u, sg, su), "swiglu two-pass")


def test_mul_mat_swiglu_full_size(q4q):
    """Llama-3-8B gate and up (4096 -> 14336) at one token, in the launch the
    benchmark times (PDL), on 4096 sampled rows plus the first and last."""
    ne00, ne01 = 4096, 14336
    wg, x = workloads.problem("llama3_8b_decode", 4)
    wu, _ = workloads.problem("llama3_8b_decode", 5)
    gd, ud = q4q.q4q_quantize_q4_0(dev(wg)), q4q.q4q_quantize_q4_0(dev(wu))
    got = q4q.q4q_mul_mat_swiglu(gd, ud, ne00, ne01, dev(x), flags=q4q.Q4Q_MUL_MAT_PDL).cpu().numpy()
    rows = _sample_rows(ne01, 4096, 62)
    gq, uq = oracle.quantize_q4_0(wg[rows]), oracle.quantize_q4_0(wu[rows])
    np.testing.assert_array_equal(gd.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy(), gq)
    ref, g, u, sg, su = oracle.mul_mat_swiglu(gq, uq, ne00, rows.size, x, nthreads=8)
    _check(got[:, rows], ref, _swiglu_tol(ref, g, u, sg, su), "swiglu full size")
    assert q4q.q4q_device_status() == 0


# ------------------------------------------------------------ Q8_0 weights --

def _assert_close(got, ref, scale):
    _check(got, ref, TOL * scale, "q8_0 weights")
    assert np.all(np.asarray(got)[scale == 0] == 0)


@pytest.mark.parametrize("ne00,ne01,ne11,path", [(64, 1, 1, 0), (256, 5, 3, 0), (768, 37, 2, 0), (4096, 9, 1, 0),
                                                 (320, 4, 4, 0), (256, 5, 3, 1), (512, 130, 9, 1), (4096, 64, 40, 1),
                                                 (768, 37, 130, 1), (1024, 200, 17, 1)])
def test_block_isums_w8_routine(q4q, ne00, ne01, ne11, path):
    # path 0: the GEMV's block dot; path 1: the tensor-core GEMM with the Q8_0
    # dequantizer (one 32-wide K block per fresh TMEM accumulator, read back exactly)
    rng = np.random.default_rng([ne00, ne01, ne11, 70])
    w = _weights(rng, ne01, ne00, scale=1.0)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[:, ::7] *= 30
    wq, xq = oracle.quantize_q8_0(w), oracle.quantize_q8_0(x)
    got = q4q.q4q_debug_block_isums_q8_0(dev(wq), dev(xq), ne00, ne01, ne11, path=path).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.block_isums_w8(wq, xq, ne00, ne01, ne11))
    assert q4q.q4q_device_status() == 0


def test_block_isums_w8_extremes(q4q):
    ne00, ne01, ne11 = 64, 2, 2
    wq = np.zeros((ne01, 2 * 34), np.uint8)
    wq[0, 2:34] = np.int8(-127).view(np.uint8)
    wq[0, 36:68] = np.int8(127).view(np.uint8)
    wq[1, 2:34] = np.int8(127).view(np.uint8)
    wq[1, 36:68] = np.int8(-127).view(np.uint8)
    xq = wq.copy()
    ref = oracle.block_isums_w8(wq, xq, ne00, ne01, ne11)
    assert ref[0, 0, 0] == 32 * 127 * 127 and ref[1, 0, 0] == -32 * 127 * 127
    got = q4q.q4q_debug_block_isums_q8_0(dev(wq), dev(xq), ne00, ne01, ne11).cpu().numpy()
    np.testing.assert_array_equal(got, ref)
    # the same extremes through the tensor-core routine (K = 256: four copies of the pair)
    wq4, xq4 = np.tile(wq, (1, 4)), np.tile(xq, (1, 4))
    got = q4q.q4q_debug_block_isums_q8_0(dev(wq4), dev(xq4), 256, ne01, ne11, path=1).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.block_isums_w8(wq4, xq4, 256, ne01, ne11))


W8_SHAPES = [(256, 1), (256, 3), (768, 2304), (3072, 768), (4096, 1024), (14336, 64), (512, 33), (1024, 4099),
             (14336, 1), (8448, 129)]


@pytest.mark.parametrize("ne00,ne01", W8_SHAPES)
@pytest.mark.parametrize("ne11", [1, 2, 7])
def test_mul_mat_q8_0_gemv(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 71])
    w = _weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    wq_d = q4q.q4q_quantize_q8_0(dev(w))
    got = q4q.q4q_mul_mat_q8_0(wq_d, ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat_w8(oracle.quantize_q8_0(w), ne00, ne01, x, nthreads=8)
    _assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0


@pytest.mark.parametrize("ne00,ne01,ne11", [(1024, 300, 8), (768, 130, 15), (4096, 64, 64), (96, 17, 3),
                                            (800, 65, 9), (32, 3, 1), (512, 130, 9), (4096, 257, 129),
                                            (1024, 64, 200), (14336, 256, 512), (768, 37, 130)])
def test_mul_mat_q8_0_batches_and_generic(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 72])
    w = _weights(rng, ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[ne11 // 2] = 0.0
    wq = oracle.quantize_q8_0(w)
    got = q4q.q4q_mul_mat_q8_0(dev(wq), ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat_w8(wq, ne00, ne01, x, nthreads=8)
    _assert_close(got, ref, scale)


def test_mul_mat_q8_0_misaligned_weights(q4q):
    rng = np.random.default_rng(73)
    ne00, ne01 = 512, 40
    w = _weights(rng, ne01, ne00)
    x = rng.standard_normal((2, ne00)).astype(np.float32)
    wq = oracle.quantize_q8_0(w)
    buf = torch.zeros(wq.size + 2, dtype=torch.uint8, device="cuda")
    buf[2:] = dev(wq.reshape(-1))
    got = q4q.q4q_mul_mat_q8_0(buf[2:], ne00, ne01, dev(x)).cpu().numpy()
    ref, scale = oracle.mul_mat_w8(wq, ne00, ne01, x)
    _assert_close(got, ref, scale)


def test_mul_mat_q8_0_full_size_decode_set(q4q):
    """Every distinct matrix of the Llama-3-8B decode set with Q8_0 weights at one
    token, as the benchmark launches them (PDL): Q8_0 bytes bit-exact and outputs
    within tolerance on up to 4096 sampled rows plus the first and last."""
    wl = workloads.WORKLOADS["llama3_8b_decode"]
    for i, (ne00, ne01) in enumerate(wl.shapes):
        if i in (2, 3, 5):
            continue                      # same shapes as k, q, gate
        w, x = workloads.problem("llama3_8b_decode", i)
        wq_d = q4q.q4q_quantize_q8_0(dev(w))
        got = q4q.q4q_mul_mat_q8_0(wq_d, ne00, ne01, dev(x), flags=q4q.Q4Q_MUL_MAT_PDL).cpu().numpy()
        rows = _sample_rows(ne01, 4096, 80 + i)
        wq_rows = oracle.quantize_q8_0(w[rows])
        np.testing.assert_array_equal(wq_d.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy(), wq_rows)
        ref, scale = oracle.mul_mat_w8(wq_rows, ne00, rows.size, x, nthreads=8)
        _assert_close(got[:, rows], ref, scale)
        del wq_d
    assert q4q.q4q_device_status() == 0


# ----------------------------------------------- projections of one input --

GROUP_CASES = [(4096, [4096, 1024, 1024]), (768, [2304]), (768, [768, 3072, 50257]), (3072, [768, 100, 1, 37]),
               (14336, [64, 4096]), (1024, [4099, 33])]


@pytest.mark.parametrize("ne00,rows", GROUP_CASES)
@pytest.mark.parametrize("ne11", [1, 3, 7, 16])
def test_mul_mat_group(q4q, ne00, rows, ne11):
    rng = np.random.default_rng([ne00, len(rows), ne11, 90])
    ws = [_weights(rng, r, ne00) for r in rows]
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    wqs = [q4q.q4q_quantize_q4_0(dev(w)) for w in ws]
    outs = q4q.q4q_mul_mat_group(wqs, rows, ne00, dev(x))
    for m, r in enumerate(rows):
        got = outs[m].cpu().numpy()
        # the same per-row arithmetic as a call of its own on the same path (below 8
        # tokens the GEMV, which a call without workspace takes)
        alone = q4q.q4q_mul_mat(wqs[m], ne00, r, dev(x), workspace=(
            torch.empty(0, dtype=torch.uint8, device="cuda") if ne11 < 8 else None))
        np.testing.assert_array_equal(got, alone.cpu().numpy())
        sel = _sample_rows(r, 2048, m) if r > 2048 else np.arange(r)
        ref, scale = oracle.mul_mat(oracle.quantize_q4_0(ws[m][sel]), ne00, sel.size, x, nthreads=8)
        _assert_close(got[:, sel], ref, scale)
    assert q4q.q4q_device_status() == 0


def test_mul_mat_group_skips_empty_and_takes_misaligned(q4q):
    rng = np.random.default_rng(91)
    ne00 = 512
    rows = [40, 0, 7]
    ws = [_weights(rng, r, ne00) if r else np.zeros((0, ne00), np.float32) for r in rows]
    x = rng.standard_normal((2, ne00)).astype(np.float32)
    wq = [oracle.quantize_q4_0(w) for w in ws]
    buf = torch.zeros(wq[2].size + 2, dtype=torch.uint8, device="cuda")
    buf[2:] = dev(wq[2].reshape(-1))
    src = [dev(wq[0]), torch.zeros(16, dtype=torch.uint8, device="cuda"), buf[2:]]
    outs = q4q.q4q_mul_mat_group(src, rows, ne00, dev(x))
    assert outs[1].shape == (2, 0)
    for m in (0, 2):
        ref, scale = oracle.mul_mat(wq[m], ne00, rows[m], x)
        _assert_close(outs[m].cpu().numpy(), ref, scale)


@pytest.mark.parametrize("ne11", [8, 64, 512])
def test_mul_mat_q8_0_full_size_batched(q4q, ne11):
    """The tensor-core path with Q8_0 weights at full size: the Llama-3-8B-shaped
    lm_head (4096 -> 128256) and down (14336 -> 4096) projections, outputs on up to
    1024 sampled rows (plus the first and last) for every token."""
    for i in (7, 6):
        ne00, ne01 = workloads.WORKLOADS["llama3_8b_batched"].shapes[i]
        w, x = workloads.problem("llama3_8b_batched", i, ne11)
        wq_d = q4q.q4q_quantize_q8_0(dev(w))
        got = q4q.q4q_mul_mat_q8_0(wq_d, ne00, ne01, dev(x)).cpu().numpy()
        rows = _sample_rows(ne01, 1024, 200 + i)
        wq_rows = wq_d.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy()
        np.testing.assert_array_equal(wq_rows, oracle.quantize_q8_0(w[rows]))
        ref, scale = oracle.mul_mat_w8(wq_rows, ne00, rows.size, x, nthreads=16)
        _assert_close(got[:, rows], ref, scale)
        del wq_d
    assert q4q.q4q_device_status() == 0
