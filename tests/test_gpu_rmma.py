"""GPU parity of the warp-MMA kernel (q4q_rmma.cu) at 1..32 tokens, run through
q4q_debug_mul_mat_path (path 3) whatever q4q_mul_mat would pick for the shape, and of
q4q_mul_mat's own choice between it, the GEMV and the tensor-core GEMM.

Every output is checked against the oracle at the library's bar, |gpu - oracle| <=
1e-5 * sum_b |fp32(d_w d_x) isum_b|, and is exactly zero where that sum is zero.
A mistake in the K order of either operand, a fragment lane, a block scale or a
split's partial sum moves an output by a sizeable part of that sum, far outside the
bar.  The shapes cover one and several 128-row tiles with a ragged last tile, one
and many 256-K stages, every token count of the path (one to four n8 token groups,
full and partial), and the K splits the workspace allows.
"""
import numpy as np
import pytest

import oracle

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
    assert np.all(got[scale == 0] == 0)


def _weights(rng, ne01, ne00):
    """Gaussian weights with blocks that are all zero (d = 0), constant, or hold exact
    rounding ties."""
    w = (rng.standard_normal((ne01, ne00)) * 0.02).astype(np.float32)
    blocks = w.reshape(-1, 32)
    nb = blocks.shape[0]
    blocks[rng.integers(0, nb, size=max(1, nb // 10))] = 0.0
    c = rng.integers(0, nb, size=max(1, nb // 10))
    blocks[c] = blocks[c, :1]
    t = rng.integers(0, nb, size=max(1, nb // 10))
    k = rng.integers(-16, 16, size=(t.size, 32)).astype(np.float32)
    k[:, 0] = -16.0
    blocks[t] = k * np.float32(0.125) / 2
    return w


def _acts(rng, ne11, ne00):
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[ne11 // 2] = 0.0                                   # a token whose every block has d = 0
    return x


def _least_workspace(ne00, ne11):
    # the warp-MMA kernel's split-free minimum: fp16 codes and scale quads for the tokens
    # padded to a multiple of 8, then the control words
    r256 = lambda b: (b + 255) // 256 * 256
    n8 = (ne11 + 7) // 8 * 8
    return r256(ne00 * n8 * 2) + r256((ne00 // 32) * (n8 // 2) * 16) + 256


def _run(q4q, wq, ne00, ne01, x, workspace=None):
    return q4q.q4q_debug_mul_mat_path(dev(wq), ne00, ne01, dev(x), 3, workspace=workspace).cpu().numpy()


# (ne00, ne01): one row; one ragged tile; several tiles with a ragged last one; the
# Llama-3-8B k/v projection (8 tiles, many K splits); a long row (56 stages) on two
# tiles; a 33-tile matrix whose last tile holds 3 rows
SHAPES = [(256, 1), (512, 300), (768, 130), (4096, 1024), (14336, 200), (1024, 4099)]


@pytest.mark.parametrize("ne00,ne01", SHAPES)
@pytest.mark.parametrize("ne11", [1, 2, 7, 8, 17, 24, 32])
def test_rmma_matches_oracle(q4q, ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 41])
    wq = oracle.quantize_q4_0(_weights(rng, ne01, ne00))
    x = _acts(rng, ne11, ne00)
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    assert_close(_run(q4q, wq, ne00, ne01, x), ref, scale)
    assert q4q.q4q_device_status() == 0


def test_rmma_every_token_count(q4q):
    # 1..32 tokens on one shape: each count of full and partial n8 token groups, on the
    # warp-MMA kernel and on whatever path q4q_mul_mat picks
    rng = np.random.default_rng(42)
    ne00, ne01 = 512, 300
    wq = oracle.quantize_q4_0(_weights(rng, ne01, ne00))
    x = rng.standard_normal((32, ne00)).astype(np.float32)
    wq_d = dev(wq)
    for ne11 in range(1, 33):
        ref, scale = oracle.mul_mat(wq, ne00, ne01, x[:ne11], nthreads=8)
        assert_close(q4q.q4q_debug_mul_mat_path(wq_d, ne00, ne01, dev(x[:ne11]), 3).cpu().numpy(), ref, scale)
        assert_close(q4q.q4q_mul_mat(wq_d, ne00, ne01, dev(x[:ne11])).cpu().numpy(), ref, scale)
    assert q4q.q4q_device_status() == 0


@pytest.mark.parametrize("ne00,ne01,ne11", [(4096, 1024, 8), (4096, 1024, 32), (14336, 256, 5), (4096, 300, 16)])
def test_rmma_split_counts_are_deterministic(q4q, ne00, ne01, ne11):
    """With the workspace q4q_mul_mat_workspace_size asks for, K is split (partial sums
    added by the last split of each slab, in split order); with less, fewer splits;
    with the split-free minimum, none.  Every result is within the bar, and a repeat
    with the same workspace gives identical bits."""
    rng = np.random.default_rng([ne00, ne01, ne11, 43])
    wq = oracle.quantize_q4_0(_weights(rng, ne01, ne00))
    x = _acts(rng, ne11, ne00)
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    full = q4q.q4q_debug_mul_mat_path_workspace_size(ne00, ne01, ne11, 3)
    least = _least_workspace(ne00, ne11)
    assert full > least
    wq_d, x_d = dev(wq), dev(x)
    for nbytes in (full, (full + least) // 2, least):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        a = q4q.q4q_debug_mul_mat_path(wq_d, ne00, ne01, x_d, 3, workspace=ws).cpu().numpy()
        b = q4q.q4q_debug_mul_mat_path(wq_d, ne00, ne01, x_d, 3, workspace=ws).cpu().numpy()
        assert_close(a, ref, scale)
        np.testing.assert_array_equal(a, b)
    assert q4q.q4q_device_status() == 0


@pytest.mark.parametrize("ne11", [3, 8, 32])
def test_rmma_split_tail_tiles(q4q, ne11):
    """More 128-row tiles than resident CTAs (on 152 SMs: 351 tiles, 304 CTAs): the
    whole waves run whole and the last wave's tiles in K splits, summed by the reduce
    kernel.  Every row of the split tiles and a sample of the others against the oracle,
    with the planned workspace and with the split-free minimum."""
    rng = np.random.default_rng([ne11, 48])
    ne00, ne01 = 1024, 350 * 128 + 37
    wq = oracle.quantize_q4_0(_weights(rng, ne01, ne00))
    x = _acts(rng, ne11, ne00)
    rows = np.unique(np.concatenate([np.arange(280 * 128, ne01), rng.choice(280 * 128, 2048, replace=False)]))
    ref, scale = oracle.mul_mat(wq.reshape(ne01, -1)[rows], ne00, rows.size, x, nthreads=8)
    wq_d, x_d = dev(wq), dev(x)
    full = q4q.q4q_debug_mul_mat_path_workspace_size(ne00, ne01, ne11, 3)
    least = _least_workspace(ne00, ne11)
    assert full > least
    for nbytes in (full, least):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        got = q4q.q4q_debug_mul_mat_path(wq_d, ne00, ne01, x_d, 3, workspace=ws).cpu().numpy()
        assert_close(got[:, rows], ref, scale)
    assert q4q.q4q_device_status() == 0


def test_rmma_scale_extremes(q4q):
    """Rows mixing weight blocks whose stored scales are fp16 subnormals, ordinary,
    exactly 8188, exactly 8192 and far above; a token scaled by 2^-120 (its fp32 block
    scales round to fp16 zero, so its outputs are exactly zero), one scaled by 2^-12
    (fp16-subnormal activation scales) and an all-zero one."""
    rng = np.random.default_rng(44)
    ne00, ne01, ne11 = 1024, 256, 24
    z = rng.standard_normal((ne01, ne00 // 32, 32))
    scales = np.array([3e-7, 2e-5, 1e-3, 0.02, 1.0, 300.0, 4e4, 1.2e5])
    w = (z * scales[rng.integers(0, scales.size, size=(ne01, ne00 // 32))][..., None]).astype(np.float32)
    w[3] = 0.0
    w[3, :, 0] = 65504.0
    w[4, :, 0] = -65536.0
    w = w.reshape(ne01, ne00)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    x[2] *= np.float32(2.0 ** -120)
    x[3] *= np.float32(2.0 ** -12)
    x[5] = 0.0
    wq = oracle.quantize_q4_0(w)
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    assert np.all(scale[2] == 0) and np.all(scale[5] == 0) and np.all(scale[3] > 0)
    assert_close(_run(q4q, wq, ne00, ne01, x), ref, scale)
    assert q4q.q4q_device_status() == 0


def test_rmma_without_workspace_falls_back(q4q):
    """Below 8 tokens a call without workspace takes the GEMV; with it, the faster of the
    GEMV and the warp-MMA kernel for the shape (here the warp-MMA kernel).  Both are
    within the bar of the oracle."""
    rng = np.random.default_rng(45)
    ne00, ne01, ne11 = 4096, 4096, 5
    wq = oracle.quantize_q4_0(_weights(rng, ne01, ne00))
    x = _acts(rng, ne11, ne00)
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    dst = torch.empty((ne11, ne01), device="cuda")
    q4q.q4q_mul_mat(dev(wq), ne00, ne01, dev(x), dst=dst, workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    assert_close(dst.cpu().numpy(), ref, scale)
    assert_close(_run(q4q, wq, ne00, ne01, x), ref, scale)
    assert q4q.q4q_device_status() == 0


def test_rmma_pdl_flag_chain(q4q):
    """y1 = W1 x, y2 = W2 y1, y3 = W3 y2 at 12 tokens with the PDL flag: the activation
    kernel of each call is launched behind the previous call and must see its output
    (same kernels, so the results equal those of calls without the flag)."""
    rng = np.random.default_rng(46)
    dims = [2048, 1024, 3072, 512]
    ne11 = 12
    wqs = [oracle.quantize_q4_0(_weights(rng, dims[i + 1], dims[i])) for i in range(3)]
    x = _acts(rng, ne11, dims[0])
    outs = {}
    for flags in (0, q4q.Q4Q_MUL_MAT_PDL):
        y = dev(x)
        ys = []
        for i in range(3):
            y = q4q.q4q_mul_mat(dev(wqs[i]), dims[i], dims[i + 1], y, flags=flags)
            ys.append(y)
        torch.cuda.synchronize()
        outs[flags] = [t.cpu().numpy() for t in ys]
    for a, b in zip(outs[0], outs[q4q.Q4Q_MUL_MAT_PDL]):
        np.testing.assert_array_equal(a, b)
    xin = x
    for i in range(3):
        ref, scale = oracle.mul_mat(wqs[i], dims[i], dims[i + 1], xin, nthreads=8)
        assert_close(outs[0][i], ref, scale)
        xin = outs[0][i]
    assert q4q.q4q_device_status() == 0


@pytest.mark.parametrize("ne00,ne01,ne11", [(256, 128, 8), (512, 300, 16), (768, 130, 17), (4096, 1024, 32)])
def test_tensor_core_path_at_few_tokens(q4q, ne00, ne01, ne11):
    """The tensor-core GEMM at 8..32 tokens, which q4q_mul_mat no longer picks for Q4_0
    weights but still runs for Q8_0 weights: forced through the path entry."""
    rng = np.random.default_rng([ne00, ne01, ne11, 47])
    wq = oracle.quantize_q4_0(_weights(rng, ne01, ne00))
    x = _acts(rng, ne11, ne00)
    ref, scale = oracle.mul_mat(wq, ne00, ne01, x, nthreads=8)
    got = q4q.q4q_debug_mul_mat_path(dev(wq), ne00, ne01, dev(x), 1).cpu().numpy()
    assert_close(got, ref, scale)
    assert q4q.q4q_device_status() == 0
