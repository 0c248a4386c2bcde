"""q4q_mul_mat_noalloc: the matmul for callers that cannot allocate device memory.

Some callers (a plugin inside an application that owns every device allocation,
a runtime that forbids allocation after start-up) cannot hand the library a
workspace.  q4q_mul_mat_noalloc takes only inputs and outputs and uses a static
scratch array that the library owns.  These tests call it through the C ABI and
check it against q4q_mul_mat, which gets a workspace from the caller, on two
calls in a row (the second call finds the first call's data in the scratch array).
This file is collected last so that a stop-at-first-failure run has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

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


def _problem(ne00, ne01, ne11, seed):
    rng = np.random.default_rng([ne00, ne01, ne11, seed])
    w = (rng.standard_normal((ne01, ne00)) * 0.02).astype(np.float32)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    return w, x


def _call_noalloc_abi(lib, wq, ne00, ne01, x, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.q4q_mul_mat_noalloc(ctypes.c_void_p(wq.data_ptr()), ne00, ne01, ctypes.c_void_p(x.data_ptr()),
                                   ne00, x.shape[0], ctypes.c_void_p(out.data_ptr()), stream)


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(q4q):
    lib = q4q._lib.load()
    # the tensor-core path (ne11 >= 8) twice with different shapes, the generic path
    # (ne00 % 256 != 0: Q8_0 activations in the scratch array) twice, then the GEMV,
    # which needs no scratch; each against the workspace entry point and the oracle
    cases = [(4096, 1000, 64, 1), (768, 130, 17, 2), (800, 200, 12, 4), (96, 33, 9, 5), (1024, 300, 3, 3)]
    for ne00, ne01, ne11, seed in cases:
        w, x = _problem(ne00, ne01, ne11, seed)
        wq = q4q.q4q_quantize_q4_0(torch.from_numpy(w).cuda())
        xd = torch.from_numpy(x).cuda()
        ref_dev = q4q.q4q_mul_mat(wq, ne00, ne01, xd)            # caller-provided workspace
        got = torch.full((ne11, ne01), float("nan"), device="cuda")
        assert _call_noalloc_abi(lib, wq, ne00, ne01, xd, got) == 0
        torch.cuda.synchronize()
        ref_dev = ref_dev.cpu().numpy()
        got = got.cpu().numpy()
        want, scale = oracle.mul_mat(wq.cpu().numpy(), ne00, ne01, x, nthreads=8)
        assert np.all(np.abs(got.astype(np.float64) - ref_dev) <= TOL * scale)
        assert np.all(np.abs(got.astype(np.float64) - want) <= TOL * scale)
        assert np.all(got[scale == 0] == 0)
    assert q4q.q4q_device_status() == 0


def test_noalloc_rejects_problems_beyond_the_static_scratch(q4q):
    lib = q4q._lib.load()
    ne00, ne01, ne11 = 4096, 256, 2048            # needs ~17 MB of scratch, the array holds 8 MiB
    assert q4q.q4q_mul_mat_workspace_size(ne00, ne01, ne11) > q4q.Q4Q_NOALLOC_SCRATCH_BYTES
    wq = torch.zeros(ne01 * ne00 // 32 * 18, dtype=torch.uint8, device="cuda")
    x = torch.zeros((ne11, ne00), device="cuda")
    out = torch.full((ne11, ne01), 7.0, device="cuda")
    assert _call_noalloc_abi(lib, wq, ne00, ne01, x, out) == 4        # Q4Q_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    with pytest.raises(q4q.Q4QError):
        q4q.q4q_mul_mat_noalloc(wq, ne00, ne01, x)
