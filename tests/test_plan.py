"""Host logic of the launch planning, on the CPU (no GPU needed).

q4q_debug_gemv_plan returns the GEMV plan the library would launch on a device
described by its SM count and opt-in shared memory; q4q_debug_mma_splits the
tensor-core GEMM's split-K count.  The tests check the invariants the kernels
rely on (shared memory within the limit, two or more ring stages wherever a CTA
reuses one, 16-byte
aligned stage offsets for the bulk copies, every row in exactly one unit, lanes
per row dividing the block pairs) over a grid of shapes, and a few plans whose
launch shapes ncu recorded on a GB300 (152 SMs, 227 KB of opt-in shared memory).
"""
import ctypes
import itertools

import pytest

SMS = 152
OPTIN = 232448          # cudaDevAttrMaxSharedMemoryPerBlockOptin on GB300
LIMIT = min(OPTIN, 227 * 1024) - 1024
FIELDS = ["G", "S", "stage", "smem", "grid", "cl", "lpr", "ppl_reg", "units", "act_off", "stage_off", "half_off",
          "row_bytes", "dy_off", "sy_off"]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from q4_quantized_matmul_gb300 import _lib
    return _lib.load()


def plan(lib, ne00, ne01, ne11, block_bytes=18, mats=1, sms=SMS, optin=OPTIN):
    out = (ctypes.c_int64 * len(FIELDS))()
    st = lib.q4q_debug_gemv_plan(ne00, ne01, ne11, block_bytes, mats, sms, optin, out)
    return (dict(zip(FIELDS, list(out))) if st == 0 else None), st


def check_invariants(p, ne00, ne01, ne11, block_bytes, mats):
    nb, npairs = ne00 // 32, ne00 // 64
    assert p["row_bytes"] == nb * block_bytes and p["row_bytes"] % 16 == 0
    # at least two ring stages, except in the small-matrix plan, where the stages
    # hold every unit of every CTA at once (nothing waits for a stage to free up)
    assert 1 <= p["S"] <= 8
    assert p["S"] >= 2 or p["units"] <= p["grid"] * p["S"]
    assert p["stage"] % 128 == 0 and p["stage"] >= p["G"] * mats * p["row_bytes"]
    assert p["half_off"] == p["G"] * p["row_bytes"] and p["half_off"] % 16 == 0
    assert p["act_off"] == 256
    assert p["dy_off"] == p["act_off"] + ne11 * npairs * 64
    assert p["sy_off"] == p["dy_off"] + ne11 * nb * 4
    assert p["stage_off"] % 128 == 0 and p["stage_off"] >= p["sy_off"] + ne11 * nb * 4
    assert p["smem"] == p["stage_off"] + p["S"] * p["stage"] and p["smem"] <= LIMIT
    assert 1 <= p["G"] <= max(1, ne01)
    assert p["units"] == -(-ne01 // p["G"])
    assert 1 <= p["grid"] <= p["units"]
    assert p["lpr"] in (4, 8, 16, 32) and npairs % p["lpr"] == 0
    ppl = npairs // p["lpr"]
    assert p["ppl_reg"] == (ppl if ne11 == 1 and ppl <= 8 else 0)
    assert p["cl"] in (1, 2) and (mats == 1 or p["cl"] == 1)
    # one phase of the ring's mbarrier counts at most 2^20 - 1 bytes
    assert mats * p["G"] * p["row_bytes"] < (1 << 20)


@pytest.mark.parametrize("block_bytes,mats", [(18, 1), (18, 2), (34, 1)])
def test_plans_keep_the_kernel_invariants(lib, block_bytes, mats):
    found = 0
    for ne00, ne01, ne11 in itertools.product([256, 512, 768, 1024, 3072, 4096, 8448, 14336, 16384],
                                              [1, 3, 33, 1000, 4099, 14336, 50257, 128256], range(1, 8)):
        p, st = plan(lib, ne00, ne01, ne11, block_bytes, mats)
        if p is None:
            assert st == 2                      # Q4Q_ERR_SHAPE: the generic kernel takes it
            continue
        found += 1
        check_invariants(p, ne00, ne01, ne11, block_bytes, mats)
    assert found > 300


def test_every_decode_shape_of_the_workloads_has_a_plan(lib):
    from q4_quantized_matmul_gb300 import workloads
    for name in ("gpt2_decode_step", "llama3_8b_decode"):
        for ne00, ne01 in set(workloads.WORKLOADS[name].shapes):
            for bb in (18, 34):
                for t in range(1, 8):
                    p, st = plan(lib, ne00, ne01, t, bb)
                    assert p is not None, (name, ne00, ne01, t, bb)


def test_plans_recorded_by_ncu(lib):
    # lm_head 4096 -> 128256, 1 token: 8-row units, 4 stages, two CTAs per SM (grid 304);
    # two such CTAs leave room for a small matrix's CTA (the q projection, 68 KB), three
    # do not fit
    p, _ = plan(lib, 4096, 128256, 1)
    assert (p["G"], p["S"], p["stage"], p["grid"], p["cl"], p["lpr"], p["ppl_reg"]) == (8, 4, 18432, 304, 1, 32, 2)
    q, _ = plan(lib, 4096, 4096, 1)
    per_cta = 1024   # shared memory the SM reserves for every resident CTA
    assert 2 * (p["smem"] + per_cta) + q["smem"] + per_cta <= 228 * 1024 < 3 * (p["smem"] + per_cta)
    # down 14336 -> 4096, 1 token: CTA pairs share the activation quantization; 7-row
    # units (586 of them, at most 4 on a CTA: 28 rows) balance the 152 CTAs better than
    # 8-row units (512, at most 4: 32 rows)
    p, _ = plan(lib, 14336, 4096, 1)
    assert (p["cl"], p["ppl_reg"], p["G"], p["units"]) == (2, 7, 7, 586)
    # the same with Q8_0 rows (15 KB): 4-row units so that three stages fit
    p, _ = plan(lib, 14336, 4096, 1, 34)
    assert (p["G"], p["S"], p["cl"]) == (4, 3, 2)
    # SwiGLU gate + up 4096 -> 14336: both matrices' rows in one stage, grid 152
    p, _ = plan(lib, 4096, 14336, 1, 18, 2)
    assert (p["G"], p["stage"], p["grid"], p["cl"]) == (8, 36864, 152, 1)
    # k 4096 -> 1024 (2.4 MB): the small-matrix plan, every unit in flight at once; one
    # 7-row unit a CTA (one dot pass of the 8 row groups)
    p, _ = plan(lib, 4096, 1024, 1)
    assert (p["G"], p["S"], p["units"], p["grid"]) == (7, 1, 147, 147)


def test_small_plans_run_one_pass(lib):
    # A small matrix (at most 96 KB of weights per SM) whose rows fit one pass of the
    # row groups on every SM gets one unit per CTA: ceil(ne01 / SMs) rows, one dot pass.
    for ne00 in (256, 768, 1024, 3072, 4096):
        for ne01 in (1, 7, 100, 152, 153, 768, 1000, 1024, 1216, 2304):
            for t in (1, 2, 3):
                p, st = plan(lib, ne00, ne01, t)
                assert st == 0, (ne00, ne01, t)
                rp = 256 // p["lpr"]
                g1 = -(-ne01 // SMS)
                if ne01 * p["row_bytes"] <= 96 * 1024 * SMS and g1 <= rp and p["ppl_reg"] <= 3:
                    assert p["G"] == g1 and p["units"] <= p["grid"] and p["S"] == 1, (ne00, ne01, t, p)


def test_shapes_the_gemv_does_not_take(lib):
    assert plan(lib, 800, 10, 1)[1] == 2            # ne00 % 256 != 0
    assert plan(lib, 4096, 10, 8)[1] == 2           # 8 tokens: the tensor-core path
    assert plan(lib, 4096, 0, 1)[1] == 2
    out = (ctypes.c_int64 * len(FIELDS))()
    assert lib.q4q_debug_gemv_plan(4096, 10, 1, 20, 1, SMS, OPTIN, out) == 7
    assert lib.q4q_debug_gemv_plan(4096, 10, 1, 18, 3, SMS, OPTIN, out) == 7
    assert lib.q4q_debug_gemv_plan(4096, 10, 1, 18, 1, SMS, OPTIN, None) == 1


def splits(lib, ne00, ne01, ne11, sms=SMS):
    s = ctypes.c_int(0)
    st = lib.q4q_debug_mma_splits(ne00, ne01, ne11, sms, ctypes.byref(s))
    assert st == 0
    return s.value


def test_split_k_rule(lib):
    for ne00, ne01, ne11 in itertools.product([256, 512, 1024, 4096, 14336], [1, 64, 300, 1024, 4096, 14336, 128256],
                                              [8, 16, 33, 64, 100, 512, 2048]):
        s = splits(lib, ne00, ne01, ne11)
        n_raw = ne00 // 256
        assert s == 1 or 4 <= s <= n_raw // 2           # every split keeps >= 512 K
        nt = 16 if ne11 <= 16 else 32 if ne11 <= 32 else 64 if ne11 <= 64 else 128
        tiles = -(-ne11 // nt) * -(-ne01 // 128)
        target = SMS * (2 if nt <= 32 else 1)
        if s > 1:
            assert tiles * 3 < target                   # only where the tiles leave most SMs idle
    # the Llama set: k/v and down split at 8 tokens, gate/up and lm_head do not
    assert splits(lib, 4096, 1024, 8) == 8
    assert splits(lib, 14336, 4096, 8) == 10
    assert splits(lib, 4096, 14336, 8) == 1
    assert splits(lib, 4096, 128256, 8) == 1
    assert splits(lib, 4096, 4096, 512) == 1           # 128 tiles: two splits would not pay
    assert splits(lib, 4096, 1024, 512) == 5


def test_split_k_argument_errors(lib):
    s = ctypes.c_int(0)
    assert lib.q4q_debug_mma_splits(4096, 1024, 4, SMS, ctypes.byref(s)) == 7     # GEMV range
    assert lib.q4q_debug_mma_splits(800, 1024, 64, SMS, ctypes.byref(s)) == 7     # ne00 % 256
    assert lib.q4q_debug_mma_splits(4096, 1024, 64, SMS, None) == 1
