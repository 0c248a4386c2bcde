"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one oracle function to a value the pages fix, a closed form, a
library routine or brute force, so that a plausible slip (dropped -8 offset,
swapped nibbles, /128 instead of /127, round-half-even, transposed operands)
fails at least one of them.

Method: "llama.cpp 深度解读" (luoboask.github.io) §2 "量化数据结构 — Q4_0 格式详解"
and §3 "量化矩阵乘法 — 核心算子".
"""
import os

import numpy as np
import pytest

import oracle
from q4_quantized_matmul_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            out[k.strip()] = v.strip()
    return out


# ------------------------------------------------------------------ layout --

def test_block_sizes_and_compression():
    # §2: 18 bytes hold 32 weights (fp16 d + 16 nibble bytes); "7.1x" vs fp32.
    assert oracle.sizeof_block_q4_0() == 18
    assert oracle.sizeof_block_q8_0() == 34
    assert round(32 * 4 / oracle.sizeof_block_q4_0(), 1) == 7.1
    w = np.zeros((3, 256), np.float32)
    assert oracle.quantize_q4_0(w).nbytes == 3 * 8 * 18
    assert oracle.quantize_q8_0(w).nbytes == 3 * 8 * 34


# ------------------------------------------------------------- hand block --

def test_hand_worked_block():
    g = _golden("hand_block.txt")
    w = ((np.arange(32) - 16) * 0.25).astype(np.float32).reshape(1, 32)
    blk = oracle.quantize_q4_0(w)[0]
    want = bytes(int(t, 16) for t in g["q4_0_bytes"].split())
    assert bytes(blk) == want
    assert int.from_bytes(bytes(blk[:2]), "little") == int(g["weights_scale_fp16"], 16)
    # decode gives the hand-derived q values times d = 0.5
    q = np.array([int(t) for t in g["weights_q"].split()], dtype=np.float32)
    np.testing.assert_array_equal(oracle.dequantize_q4_0(blk, 32)[0], q * 0.5)

    x = np.ones((1, 32), np.float32)
    q8 = oracle.quantize_q8_0(x)[0]
    assert int.from_bytes(bytes(q8[:2]), "little") == int(g["act_scale_fp16"], 16)
    assert np.all(q8[2:].view(np.int8) == int(g["act_q"]))

    assert oracle.block_isums(blk, q8, 32, 1, 1)[0, 0, 0] == int(g["isum"])
    assert oracle.vec_dot_q4_0_q8_0(32, blk, q8) == float(g["dst"])
    dst, scale = oracle.mul_mat(blk, 32, 1, x)
    assert dst[0, 0] == np.float32(float(g["dst"]))
    assert scale[0, 0] == abs(float(g["dst"]))
    # the true (unquantized) dot is -4.0: quantization error is ~0.5, not zero
    assert float(np.dot(w[0].astype(np.float64), x[0])) == float(g["dst_unquantized"])



def test_two_block_tolerance_scale():
    # The tolerance scale S = sum_b |fp32(d_w d_x) * isum_b| on a row whose two
    # block sums have opposite signs (the hand block followed by its negation,
    # tests/golden/two_block_scale.txt): S is the sum of the absolute block terms,
    # not the absolute value of their sum, and dst keeps its sign.
    g = _golden("two_block_scale.txt")
    a = ((np.arange(32) - 16) * 0.25).astype(np.float32)
    w = np.concatenate([a, -a]).reshape(1, 64)
    blocks = oracle.quantize_q4_0(w)[0]
    assert bytes(blocks[18:]) == bytes(int(t, 16) for t in g["block_b_bytes"].split())
    q = np.array([int(t) for t in g["block_b_q"].split()], dtype=np.float32)
    np.testing.assert_array_equal(oracle.dequantize_q4_0(blocks[18:], 32)[0], q * 0.5)
    x = np.ones((1, 64), np.float32)
    q8 = oracle.quantize_q8_0(x)
    np.testing.assert_array_equal(oracle.block_isums(blocks, q8, 64, 1, 1)[0, 0],
                                  [int(g["isum_a"]), int(g["isum_b"])])
    dst, scale = oracle.mul_mat(blocks, 64, 1, x)
    assert dst[0, 0] == np.float32(float(g["dst"]))
    assert scale[0, 0] == float(g["scale"])
    # the same through the already-quantized entry point, and with the blocks swapped
    dst2, scale2 = oracle.mul_mat_q8(blocks, 64, 1, q8, 1)
    assert dst2[0, 0] == dst[0, 0] and scale2[0, 0] == scale[0, 0]
    swapped = np.concatenate([blocks[18:], blocks[:18]])
    dst3, scale3 = oracle.mul_mat(swapped, 64, 1, x)
    assert dst3[0, 0] == dst[0, 0] and scale3[0, 0] == scale[0, 0]


def test_tolerance_scale_closed_forms():
    # Where every block term has the same sign, S = |dst| up to dst's fp32 rounding.
    rng = np.random.default_rng(17)
    w = np.abs(rng.standard_normal((6, 256))).astype(np.float32)
    x = np.abs(rng.standard_normal((3, 256))).astype(np.float32)
    dst, scale = oracle.mul_mat(oracle.quantize_q4_0(w), 256, 6, x)
    assert np.all(np.abs(np.abs(dst) - scale) <= 8 * 2.0 ** -24 * scale)
    # A row whose second block repeats the first while the activations of the second
    # block are the negated first ones: Q8_0 quantization is symmetric (round half
    # away from zero, scale from |x|), so isum_b = -isum_a and the two terms cancel
    # exactly: dst = 0 while S is twice one block's term.
    wa = (rng.standard_normal((4, 32)) * 0.02).astype(np.float32)
    xa = rng.standard_normal((3, 32)).astype(np.float32)
    rows = oracle.quantize_q4_0(np.concatenate([wa, wa], axis=1))
    xx = np.concatenate([xa, -xa], axis=1)
    isums = oracle.block_isums(rows, oracle.quantize_q8_0(xx), 64, 4, 3)
    np.testing.assert_array_equal(isums[..., 1], -isums[..., 0])
    d, s = oracle.mul_mat(rows, 64, 4, xx)
    single_d, single_s = oracle.mul_mat(oracle.quantize_q4_0(wa), 32, 4, xa)
    assert np.all(d == 0.0)
    np.testing.assert_array_equal(s, 2 * single_s)
    # one block: S is |d * isum| in fp64, dst the same product rounded once to fp32
    assert np.all(np.abs(single_s - np.abs(single_d)) <= 2.0 ** -24 * single_s)

# -------------------------------------------------------------------- fp16 --

def _fp32_patterns(rng):
    pats = []
    mant = rng.integers(0, 1 << 23, size=2048, dtype=np.uint32)
    # half-way and neighbouring mantissas for binary16 normals (13 dropped bits)
    ties = np.array([0x1000, 0x0fff, 0x1001, 0x3000, 0x2fff, 0x3001, 0x7fffff, 0x7fe000,
                     0x7ff000, 0x7fefff, 0x0, 0x1, 0x2000], dtype=np.uint32)
    for e in range(256):
        for s in (0, 1):
            base = np.uint32((s << 31) | (e << 23))
            pats.append(base | mant)
            pats.append(base | ties)
            # binary16 subnormal range: ties at every possible drop position
            sh = np.arange(13, 24, dtype=np.uint32)
            pats.append(base | (np.uint32(1) << (sh - 1)))
            pats.append(base | (np.uint32(3) << (sh - 1)))
            pats.append(base | ((np.uint32(1) << (sh - 1)) + 1))
            pats.append(base | ((np.uint32(1) << (sh - 1)) - 1))
    pats.append(rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32))
    return np.concatenate(pats)


def test_fp16_narrowing_matches_numpy():
    # numpy's float32 -> float16 cast is IEEE round-to-nearest-even with subnormals.
    rng = np.random.default_rng(1234)
    bits = _fp32_patterns(rng)
    x = bits.view(np.float32)
    ours = oracle.fp16_from_f32(x)
    ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN
    assert np.all((ours[nan] & 0x7c00) == 0x7c00) and np.all((ours[nan] & 0x3ff) != 0)


def test_fp16_widening_all_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f32_from_fp16(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(ours[nan]))


# ------------------------------------------------ exact-grid closed forms --

def _grid_q4_blocks(rng, nblocks, log2_scales):
    k = rng.integers(-8, 8, size=(nblocks, 32))
    k[:, rng.integers(0, 32, size=nblocks)] = -8           # amax = 8 * s in every block
    k[np.arange(nblocks), rng.integers(0, 32, size=nblocks)] = -8
    s = np.exp2(rng.choice(log2_scales, size=(nblocks, 1))).astype(np.float32)
    return k, s


def test_q4_0_exact_grid_round_trip():
    # Weights that already sit on the Q4_0 grid (integer k in [-8, 7] times a
    # power-of-two scale, -8 present so amax = 8s) must encode to nibble k + 8,
    # store d = s, and decode back bit-exactly.
    rng = np.random.default_rng(7)
    k, s = _grid_q4_blocks(rng, 4096, np.arange(-14, 10))
    w = (k * s).astype(np.float32).reshape(64, 64 * 32)
    blocks = oracle.quantize_q4_0(w).reshape(-1, 18)
    d = oracle.f32_from_fp16(blocks[:, :2].copy().view(np.uint16).reshape(-1))
    np.testing.assert_array_equal(d, s.reshape(-1))
    nib_lo = (blocks[:, 2:] & 0x0F).astype(np.int64) - 8
    nib_hi = (blocks[:, 2:] >> 4).astype(np.int64) - 8
    np.testing.assert_array_equal(nib_lo, k[:, 0::2])
    np.testing.assert_array_equal(nib_hi, k[:, 1::2])
    np.testing.assert_array_equal(oracle.dequantize_q4_0(blocks, 64 * 32), w)


def test_q8_0_exact_grid_round_trip():
    rng = np.random.default_rng(8)
    n = 4096
    k = rng.integers(-127, 128, size=(n, 32))
    k[np.arange(n), rng.integers(0, 32, size=n)] = rng.choice([-127, 127], size=n)
    s = np.exp2(rng.integers(-14, 8, size=(n, 1))).astype(np.float32)
    x = (k * s).astype(np.float32).reshape(64, 64 * 32)
    blocks = oracle.quantize_q8_0(x).reshape(-1, 34)
    d = oracle.f32_from_fp16(blocks[:, :2].copy().view(np.uint16).reshape(-1))
    # amax/127 = 127 s / 127 = s exactly
    np.testing.assert_array_equal(d, s.reshape(-1))
    np.testing.assert_array_equal(blocks[:, 2:].view(np.int8).astype(np.int64), k)
    np.testing.assert_array_equal(oracle.dequantize_q8_0(blocks, 64 * 32), x)


@pytest.mark.parametrize("ne00,ne01,ne11", [(32, 1, 1), (64, 3, 2), (256, 5, 3), (96, 7, 4)])
def test_lossless_inputs_give_plain_matmul(ne00, ne01, ne11):
    # With both operands on their quantization grids nothing is lost, so the
    # quantized matmul must equal numpy's float64 product W @ X^T of the raw
    # inputs (up to the oracle's fp32 accumulation).  A transposed operand, a
    # dropped -8, swapped nibbles or a wrong scale all break this.
    rng = np.random.default_rng([ne00, ne01, ne11])
    nbw = ne01 * ne00 // 32
    k, s = _grid_q4_blocks(rng, nbw, np.arange(-8, -3))
    w = (k * s).astype(np.float32).reshape(ne01, ne00)
    nbx = ne11 * ne00 // 32
    kx = rng.integers(-127, 128, size=(nbx, 32))
    kx[np.arange(nbx), rng.integers(0, 32, size=nbx)] = 127
    sx = np.exp2(rng.integers(-8, 2, size=(nbx, 1))).astype(np.float32)
    x = (kx * sx).astype(np.float32).reshape(ne11, ne00)
    blocks = oracle.quantize_q4_0(w)
    dst, scale = oracle.mul_mat(blocks, ne00, ne01, x)
    ref = x.astype(np.float64) @ w.astype(np.float64).T          # [ne11, ne01]
    assert dst.shape == (ne11, ne01)
    assert np.all(np.abs(dst - ref) <= 1e-6 * scale + 1e-30)


# ------------------------------------------------------- invariants ------

def test_round_trip_error_bound():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((128, 1024)) * 0.02).astype(np.float32)
    blocks = oracle.quantize_q4_0(w)
    deq = oracle.dequantize_q4_0(blocks, 1024)
    wb = w.reshape(-1, 32)
    d32 = (np.abs(wb).max(axis=1, keepdims=True) / np.float32(8)).astype(np.float32)
    err = np.abs(wb - deq.reshape(-1, 32))
    # rounding error <= d/2, fp16 scale error <= 8 * d * 2^-11; the clamped top element <= d
    assert np.all(err <= d32 * (1 + 2.0 ** -8) * (1 + 1e-6))
    inner = wb < 7.5 * d32
    assert np.all(err[inner] <= (d32 * (0.5 + 2.0 ** -8) * (1 + 1e-6) * np.ones_like(wb))[inner])

    x = rng.standard_normal((16, 1024)).astype(np.float32)
    q8 = oracle.quantize_q8_0(x)
    xd = oracle.dequantize_q8_0(q8, 1024).reshape(-1, 32)
    xb = x.reshape(-1, 32)
    dx = np.abs(xb).max(axis=1, keepdims=True) / np.float32(127)
    assert np.all(np.abs(xb - xd) <= dx * (0.5 + 127 * 2.0 ** -11) * (1 + 1e-6))


def test_special_blocks():
    z = np.zeros((1, 32), np.float32)
    b = oracle.quantize_q4_0(z)[0]
    assert list(b[:2]) == [0, 0] and np.all(b[2:] == 0x88)
    q = oracle.quantize_q8_0(z)[0]
    assert np.all(q == 0)
    # a positive constant block: c/(c/8) = 8 -> clamped to 7 -> nibble 15; error exactly c/8
    c = np.full((1, 32), 0.75, np.float32)
    b = oracle.quantize_q4_0(c)[0]
    assert np.all(b[2:] == 0xFF)
    assert np.all(oracle.dequantize_q4_0(b, 32) == np.float32(7 * 0.75 / 8))
    # a negative constant block sits exactly on -8
    b = oracle.quantize_q4_0(-c)[0]
    assert np.all(b[2:] == 0x00)
    assert np.all(oracle.dequantize_q4_0(b, 32) == np.float32(-0.75))
    # a zero weight row or a zero activation row gives exactly zero
    w = np.random.default_rng(3).standard_normal((4, 64)).astype(np.float32)
    dst, scale = oracle.mul_mat(oracle.quantize_q4_0(w), 64, 4, np.zeros((2, 64), np.float32))
    assert np.all(dst == 0) and np.all(scale == 0)


def test_half_away_from_zero_rounding():
    # w = (+-2.5, +-1.5, +-0.5) * d with amax = 8 d: ties go away from zero
    d = np.float32(0.25)
    vals = np.zeros(32, np.float32)
    vals[0] = -8 * d
    vals[1:7] = np.array([2.5, -2.5, 1.5, -1.5, 0.5, -0.5], np.float32) * d
    b = oracle.quantize_q4_0(vals.reshape(1, 32))[0]
    deq = oracle.dequantize_q4_0(b, 32)[0] / d
    np.testing.assert_array_equal(deq[1:7], [3, -3, 2, -2, 1, -1])



def test_q8_0_half_away_from_zero_rounding():
    # Q8_0 with amax = 127 s (s a power of two) has d32 = s exactly, so elements at
    # (k + 1/2) s are exact ties: they round away from zero (roundf), not to even.
    s = np.float32(2.0 ** -5)
    vals = np.zeros(32, np.float32)
    vals[0] = 127 * s
    ties = np.array([2.5, -2.5, 1.5, -1.5, 0.5, -0.5, 126.5, -126.5], np.float32)
    vals[1:9] = ties * s
    q = oracle.quantize_q8_0(vals.reshape(1, 32))[0]
    assert int.from_bytes(bytes(q[:2]), "little") == 0x2800          # fp16 2^-5
    np.testing.assert_array_equal(q[3:11].view(np.int8), [3, -3, 2, -2, 1, -1, 127, -127])

# ---------------------------------------------------------- brute force --

@pytest.mark.parametrize("ne00,ne01,ne11", [(32, 1, 1), (64, 2, 1), (256, 3, 2), (256, 5, 3), (160, 4, 3)])
def test_block_form_equals_decoded_brute_force(ne00, ne01, ne11):
    w, x = workloads.random_problem(ne00, ne01, ne11, seed=11)
    blocks = oracle.quantize_q4_0(w)
    q8 = oracle.quantize_q8_0(x)
    dst, scale = oracle.mul_mat(blocks, ne00, ne01, x)
    # fp64 over decoded reals, two independent ways
    bf = oracle.mul_mat_decoded_f64(blocks, ne00, ne01, q8, ne11)
    npref = (oracle.dequantize_q8_0(q8, ne00).astype(np.float64)
             @ oracle.dequantize_q4_0(blocks, ne00).astype(np.float64).T)
    np.testing.assert_allclose(bf, npref, rtol=0, atol=1e-12 * (1 + np.abs(npref).max()))
    assert np.all(np.abs(dst - bf) <= 1e-6 * scale + 1e-30)
    # and the integer block sums times the scales reproduce the fp64 value exactly
    isums = oracle.block_isums(blocks, q8, ne00, ne01, ne11).astype(np.float64)
    dw = oracle.f32_from_fp16(blocks.reshape(-1, 18)[:, :2].copy().view(np.uint16).reshape(-1)).reshape(ne01, -1)
    dx = oracle.f32_from_fp16(q8.reshape(-1, 34)[:, :2].copy().view(np.uint16).reshape(-1)).reshape(ne11, -1)
    blockform = np.einsum("tb,rb,trb->tr", dx.astype(np.float64), dw.astype(np.float64), isums)
    np.testing.assert_allclose(blockform, bf, rtol=1e-13, atol=1e-300)


def test_isum_brute_force_tiny():
    # every (nibble, int8) pair in one block position, summed by plain Python loops
    rng = np.random.default_rng(5)
    for _ in range(20):
        nib = rng.integers(0, 16, size=32)
        q = rng.integers(-127, 128, size=32)
        blk = np.zeros(18, np.uint8)
        blk[2:] = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
        y = np.zeros(34, np.uint8)
        y[2:] = q.astype(np.int8).view(np.uint8)
        want = sum(int(nib[i] - 8) * int(q[i]) for i in range(32))
        assert oracle.block_isums(blk, y, 32, 1, 1)[0, 0, 0] == want


def test_threads_do_not_change_results():
    w, x = workloads.random_problem(512, 300, 3, seed=2)
    blocks = oracle.quantize_q4_0(w)
    d1, s1 = oracle.mul_mat(blocks, 512, 300, x, nthreads=1)
    d4, s4 = oracle.mul_mat(blocks, 512, 300, x, nthreads=4)
    np.testing.assert_array_equal(d1, d4)
    np.testing.assert_array_equal(s1, s4)


# ------------------------------------------- independent numpy restatement --

def _np_quant(x, levels_lo, levels_hi, div):
    xb = x.reshape(-1, 32).astype(np.float32)
    amax = np.abs(xb).max(axis=1, keepdims=True)
    d = (amax / np.float32(div)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d > 0, xb / np.where(d > 0, d, 1), 0).astype(np.float32)
    r = np.sign(r) * np.floor(np.abs(r) + np.float32(0.5))        # half away from zero
    return np.clip(r, levels_lo, levels_hi).astype(np.int64), d.astype(np.float16).view(np.uint16)


def test_numpy_restatement_q4_0_and_q8_0():
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    k, d = _np_quant(w, -8, 7, 8)
    blocks = oracle.quantize_q4_0(w).reshape(-1, 18)
    np.testing.assert_array_equal(blocks[:, :2].copy().view(np.uint16), d)
    np.testing.assert_array_equal((blocks[:, 2:] & 0xF).astype(np.int64) - 8, k[:, 0::2])
    np.testing.assert_array_equal((blocks[:, 2:] >> 4).astype(np.int64) - 8, k[:, 1::2])
    x = rng.standard_normal((8, 512)).astype(np.float32)
    kq, dq = _np_quant(x, -127, 127, 127)
    q8 = oracle.quantize_q8_0(x).reshape(-1, 34)
    np.testing.assert_array_equal(q8[:, :2].copy().view(np.uint16), dq)
    np.testing.assert_array_equal(q8[:, 2:].view(np.int8).astype(np.int64), kq)
