"""GPU parity of q4q_mul_mat_chain: dependent one-token projections in one launch.

The decode step of the "ggml GPT-2 117M inference walkthrough" (gpt2_eval: every
layer's QKV projection §3.2, output projection and MLP §3.5, the lm_head §3.6)
runs its ggml_mul_mat calls one after another, each on what an earlier one wrote.
Every link is checked against the oracle on the very input the GPU link read, at
the library's bar (|gpu - oracle| <= 1e-5 sum_b |fp32(d_w d_x) isum_b|, exact 0
where that sum is 0), and against q4q_mul_mat on the same input (the chain
computes each row exactly as the GEMV does, so the outputs are bit-identical).
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
    err = np.abs(np.asarray(got, np.float64) - ref.astype(np.float64))
    bad = err > TOL * scale
    assert not bad.any(), "%d of %d outside tolerance; worst %g" % (bad.sum(), bad.size, err[bad].max())
    assert np.all(np.asarray(got)[scale == 0] == 0)


def _weights(q4q, rng, ne01, ne00):
    w = (rng.standard_normal((ne01, ne00)) * 0.02).astype(np.float32)
    return q4q.q4q_quantize_q4_0(dev(w))


def _check_links(q4q, links, sample_rows=4096):
    """Each link against the oracle on the input the GPU read, and against q4q_mul_mat."""
    for i, (w, ne00, ne01, x, y) in enumerate(links):
        xin = x.reshape(1, ne00)
        got = y.cpu().numpy().reshape(1, ne01)
        rows = np.arange(ne01) if ne01 <= sample_rows else np.unique(np.concatenate([
            np.random.default_rng(i).choice(ne01, sample_rows, replace=False), [0, ne01 - 1]]))
        wq_rows = w.view(ne01, -1)[torch.from_numpy(rows).cuda()].cpu().numpy()
        ref, scale = oracle.mul_mat(wq_rows, ne00, rows.size, xin.cpu().numpy(), nthreads=8)
        assert_close(got[:, rows], ref, scale)
        plain = q4q.q4q_mul_mat(w, ne00, ne01, xin).cpu().numpy()
        np.testing.assert_array_equal(got, plain, err_msg="link %d" % i)


def test_chain_three_dependent_links(q4q):
    rng = np.random.default_rng(81)
    dims = [1024, 2048, 768, 1536]
    ws = [_weights(q4q, rng, dims[i + 1], dims[i]) for i in range(3)]
    x = dev(rng.standard_normal(dims[0]).astype(np.float32))
    ys = [torch.full((dims[i + 1],), float("nan"), device="cuda") for i in range(3)]
    links = [(ws[0], dims[0], dims[1], x, ys[0]), (ws[1], dims[1], dims[2], ys[0], ys[1]),
             (ws[2], dims[2], dims[3], ys[1], ys[2])]
    for _ in range(2):                                  # the same workspace twice: counters restart
        q4q.q4q_mul_mat_chain(links)
        torch.cuda.synchronize()
        _check_links(q4q, links)
    assert q4q.q4q_device_status() == 0


def test_chain_gpt2_decode_step_fully_dependent(q4q):
    # 12 layers of c_attn (768 -> 2304), c_proj (768 -> 768, reading the first 768 of
    # c_attn's output), c_fc (768 -> 3072), c_proj of the MLP (3072 -> 768), then the
    # lm_head (768 -> 50257): every link reads the previous link's output
    rng = np.random.default_rng(82)
    shapes = workloads.WORKLOADS["gpt2_decode_step"].shapes
    assert len(shapes) == 49
    x0 = dev(rng.standard_normal(768).astype(np.float32))
    links, prev = [], x0
    for (ne00, ne01) in shapes:
        w = _weights(q4q, rng, ne01, ne00)
        y = torch.full((ne01,), float("nan"), device="cuda")
        links.append((w, ne00, ne01, prev[:ne00], y))
        prev = y
    q4q.q4q_mul_mat_chain(links)
    torch.cuda.synchronize()
    _check_links(q4q, links)
    assert q4q.q4q_device_status() == 0


def test_chain_independent_inputs_llama_shapes(q4q):
    # the Llama-3-8B decode set with one input per link (the benchmark's form): the
    # links still run in order, each after the previous one completed everywhere
    rng = np.random.default_rng(83)
    links = []
    for (ne00, ne01) in workloads.WORKLOADS["llama3_8b_decode"].shapes:
        w = _weights(q4q, rng, ne01, ne00)
        x = dev(rng.standard_normal(ne00).astype(np.float32))
        links.append((w, ne00, ne01, x, torch.empty(ne01, device="cuda")))
    q4q.q4q_mul_mat_chain(links)
    torch.cuda.synchronize()
    _check_links(q4q, links, sample_rows=2048)
    assert q4q.q4q_device_status() == 0


def test_chain_single_link_and_row_counts(q4q):
    # one link; links whose row counts leave most CTAs without a unit; a long row
    rng = np.random.default_rng(84)
    for spec in [((256, 1),), ((256, 3), (512, 1), (256, 7)), ((768, 33), (256, 4099), (14336, 2), (4096, 300))]:
        links = []
        for (ne00, ne01) in spec:
            w = _weights(q4q, rng, ne01, ne00)
            x = dev(rng.standard_normal(ne00).astype(np.float32))
            links.append((w, ne00, ne01, x, torch.full((ne01,), float("nan"), device="cuda")))
        q4q.q4q_mul_mat_chain(links)
        torch.cuda.synchronize()
        _check_links(q4q, links)
    assert q4q.q4q_device_status() == 0


def test_chain_wait_timeout_path(q4q):
    """A chain whose first CTA never reports its first link finished (the debug entry,
    5 ms limit): the other CTAs' waits before the second link run out, the status
    reports Q4Q_ERR_TIMEOUT once, and the next chain runs normally."""
    rng = np.random.default_rng(85)
    w = _weights(q4q, rng, 4096, 4096)
    x = dev(rng.standard_normal((1, 4096)).astype(np.float32))
    assert q4q.q4q_device_status() == 0
    q4q.q4q_debug_mul_mat_timeout(w, 4096, 4096, x, 2, 5_000_000)
    assert q4q.q4q_device_status() == 6
    assert q4q.q4q_device_status() == 0
    ys = [torch.empty(4096, device="cuda") for _ in range(2)]
    links = [(w, 4096, 4096, x.reshape(-1), ys[0]), (w, 4096, 4096, ys[0], ys[1])]
    q4q.q4q_mul_mat_chain(links)
    torch.cuda.synchronize()
    _check_links(q4q, links)
    assert q4q.q4q_device_status() == 0
