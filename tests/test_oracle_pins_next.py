"""Pins of the oracle's functions next to the matmul (CPU only): the Q4_0 / Q8_0
row gather, the bias / GELU / SwiGLU epilogues and the Q8_0-weight contraction.

Each test ties an oracle function to something other than itself: closed forms
of the activation functions and textbook values of the normal CDF, scipy's
special functions, numpy fp64 products of lossless inputs, brute-force decoding
with plain Python loops.  Sources:
  * get_rows: the embedding lookup of the Llama graph in "llama.cpp 深度解读" §4
    (ggml_get_rows(tok_embeddings, inp_tokens)), the table stored as Q4_0 (§1's
    GGUF tensor-info example), decoded as §2 states.
  * bias: ggml_add(ggml_repeat(b, cur), cur) after every GPT-2 projection
    ("ggml GPT-2 117M inference walkthrough" §3.2, §3.5); GELU on the MLP's first
    projection (same page, §3.5 and its F1 equation).
  * SwiGLU: SiLU(gate) * up with SiLU(x) = x * sigmoid(x) ("llama.cpp 深度解读" §4, Step I).
  * Q8_0 weights: the Q8_0 type of §2's type table in the contraction of §3.
"""
import math
import os

import numpy as np
import pytest

import oracle

scipy_special = pytest.importorskip("scipy.special")


# ---------------------------------------------------------------- get_rows --

def _decode_q4_0_py(block: bytes) -> list:
    d = float(np.frombuffer(block[:2], dtype=np.float16)[0])
    out = []
    for j in range(16):
        byte = block[2 + j]
        out.append(((byte & 0x0F) - 8) * d)
        out.append(((byte >> 4) - 8) * d)
    return out


def _decode_q8_0_py(block: bytes) -> list:
    d = float(np.frombuffer(block[:2], dtype=np.float16)[0])
    return [int(np.int8(np.uint8(b))) * d for b in block[2:34]]


@pytest.mark.parametrize("kind", ["q4_0", "q8_0"])
def test_get_rows_brute_force(kind):
    rng = np.random.default_rng(41)
    ncols, nrows = 96, 13
    w = (rng.standard_normal((nrows, ncols)) * 0.02).astype(np.float32)
    table = oracle.quantize_q4_0(w) if kind == "q4_0" else oracle.quantize_q8_0(w)
    bpb = 18 if kind == "q4_0" else 34
    dec = _decode_q4_0_py if kind == "q4_0" else _decode_q8_0_py
    ids = np.array([0, 12, 5, 5, 7, 0, 11], np.int32)
    rows, ok = oracle.get_rows(table, ncols, ids, kind)
    assert ok and rows.shape == (ids.size, ncols)
    for i, r in enumerate(ids):
        want = []
        for b in range(ncols // 32):
            want += dec(bytes(table[r, b * bpb:(b + 1) * bpb]))
        np.testing.assert_array_equal(rows[i], np.array(want, np.float32))


def test_get_rows_lossless_table_returns_raw_rows():
    # a table already on the Q4_0 grid decodes back to the raw fp32 rows exactly
    rng = np.random.default_rng(42)
    nrows, ncols = 40, 256
    k = rng.integers(-8, 8, size=(nrows * ncols // 32, 32))
    k[:, 0] = -8
    s = np.exp2(rng.integers(-12, 4, size=(k.shape[0], 1))).astype(np.float32)
    w = (k * s).astype(np.float32).reshape(nrows, ncols)
    ids = rng.integers(0, nrows, size=100).astype(np.int32)
    rows, ok = oracle.get_rows(oracle.quantize_q4_0(w), ncols, ids)
    assert ok
    np.testing.assert_array_equal(rows, w[ids])


def test_get_rows_out_of_range_ids():
    w = np.ones((4, 64), np.float32)
    table = oracle.quantize_q4_0(w)
    rows, ok = oracle.get_rows(table, 64, np.array([1, 4, -1, 3], np.int32))
    assert not ok
    assert np.all(rows[1] == 0) and np.all(rows[2] == 0)
    assert np.all(rows[0] == np.float32(7 / 8)) and np.all(rows[3] == np.float32(7 / 8))


# --------------------------------------------------------------- epilogues --

def test_silu_and_gelu_closed_forms():
    assert oracle.silu(0.0) == 0.0 and oracle.gelu(0.0) == 0.0
    # sigmoid(ln 3) = 3/4
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) <= 1e-15
    for x in (0.1, 0.7, 1.0, 2.5, 6.0, 30.0):
        # silu(x) - silu(-x) = x (sigmoid(x) + sigmoid(-x) = 1), same for gelu (Phi(x) + Phi(-x) = 1)
        assert abs(oracle.silu(x) - oracle.silu(-x) - x) <= 1e-14 * max(1.0, x)
        assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) <= 1e-14 * max(1.0, x)
    # textbook values of the standard normal CDF: Phi(1), Phi(2), Phi(-3)
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) <= 1e-15
    assert abs(oracle.gelu(2.0) - 2 * 0.9772498680518208) <= 1e-15
    assert abs(oracle.gelu(-3.0) - (-3) * 0.0013498980316301) <= 1e-16
    # large |x|: silu -> x, gelu -> x (positive side) and -> 0 (negative side)
    assert oracle.silu(50.0) == 50.0 and oracle.gelu(50.0) == 50.0
    assert abs(oracle.silu(-50.0)) < 1e-19 and abs(oracle.gelu(-50.0)) < 1e-300


def test_activations_match_scipy():
    xs = np.concatenate([np.linspace(-20, 20, 4001), [-87.5, -60.0, 60.0, 1e-30, -1e-30]])
    for x in xs:
        # relative: a few ulps of the two libraries' exp / erfc apart, also where the
        # values are tiny, where rounding x/sqrt(2) moves erfc by up to ~2x^2 ulps
        # (the tanh approximation of GELU is ~1e-4 off, far outside)
        s_ref, g_ref = x * scipy_special.expit(x), x * scipy_special.ndtr(x)
        assert abs(oracle.silu(x) - s_ref) <= 1e-13 * abs(s_ref) + 1e-300
        assert abs(oracle.gelu(x) - g_ref) <= 1e-12 * abs(g_ref) + 1e-300


def _grid_w(rng, ne01, ne00):
    k = rng.integers(-8, 8, size=(ne01 * ne00 // 32, 32))
    k[:, 0] = -8
    s = np.exp2(rng.integers(-8, -3, size=(k.shape[0], 1))).astype(np.float32)
    return (k * s).astype(np.float32).reshape(ne01, ne00)


def _grid_x(rng, ne11, ne00):
    k = rng.integers(-127, 128, size=(ne11 * ne00 // 32, 32))
    k[:, 0] = 127
    s = np.exp2(rng.integers(-8, -2, size=(k.shape[0], 1))).astype(np.float32)
    return (k * s).astype(np.float32).reshape(ne11, ne00)


@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_GELU])
def test_bias_epilogue_lossless(act):
    # lossless operands: mul_mat is exact (a sum of few dyadic terms), so
    # act(mul_mat + bias) must equal the fp64 value rounded once to fp32 before
    # the activation; bias is [ne01] and repeats over the ne11 tokens
    rng = np.random.default_rng(43)
    ne00, ne01, ne11 = 64, 5, 3
    w, x = _grid_w(rng, ne01, ne00), _grid_x(rng, ne11, ne00)
    bias = (rng.integers(-64, 64, size=ne01) / 8.0).astype(np.float32)
    dst, pre, _ = oracle.mul_mat_epilogue(oracle.quantize_q4_0(w), ne00, ne01, x, bias=bias, act=act)
    exact = x.astype(np.float64) @ w.astype(np.float64).T + bias.astype(np.float64)[None, :]
    np.testing.assert_array_equal(pre, exact.astype(np.float32))
    want = pre if act == oracle.ACT_NONE else np.vectorize(lambda v: np.float32(v * scipy_special.ndtr(v)))(
        pre.astype(np.float64)).astype(np.float32)
    np.testing.assert_array_equal(dst, want)


def test_swiglu_epilogue_lossless_and_operand_order():
    rng = np.random.default_rng(44)
    ne00, ne01, ne11 = 96, 6, 2
    wg, wu, x = _grid_w(rng, ne01, ne00), _grid_w(rng, ne01, ne00), _grid_x(rng, ne11, ne00)
    dst, g, u, _, _ = oracle.mul_mat_swiglu(oracle.quantize_q4_0(wg), oracle.quantize_q4_0(wu), ne00, ne01, x)
    g64 = x.astype(np.float64) @ wg.astype(np.float64).T
    u64 = x.astype(np.float64) @ wu.astype(np.float64).T
    np.testing.assert_array_equal(g, g64.astype(np.float32))
    np.testing.assert_array_equal(u, u64.astype(np.float32))
    s = (g64 * scipy_special.expit(g64)).astype(np.float32)
    np.testing.assert_array_equal(dst, (s * u64.astype(np.float32)).astype(np.float32))
    # SiLU applies to the gate, not to up
    assert not np.array_equal(dst, oracle.swiglu(u, g))


def test_swiglu_elementwise_values():
    g = np.array([0.0, 1.0, -1.0, 4.0, -100.0, 30.0], np.float32)
    u = np.array([5.0, 2.0, 2.0, -1.0, 3.0, 0.5], np.float32)
    y = oracle.swiglu(g, u)
    assert y[0] == 0.0
    assert y[1] == np.float32(np.float32(1.0 / (1.0 + math.exp(-1.0))) * 2.0)
    assert y[2] == np.float32(np.float32(-1.0 / (1.0 + math.exp(1.0))) * 2.0)
    assert abs(y[4]) < 1e-40
    assert y[5] == np.float32(np.float32(30.0 / (1.0 + math.exp(-30.0))) * 0.5)


# ----------------------------------------------------------- Q8_0 weights --

@pytest.mark.parametrize("ne00,ne01,ne11", [(32, 1, 1), (64, 3, 2), (256, 5, 3), (96, 7, 4)])
def test_w8_lossless_inputs_give_plain_matmul(ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 8])
    w = _grid_x(rng, ne01, ne00)          # Q8_0 grid: integer codes times a power of two
    x = _grid_x(rng, ne11, ne00)
    dst, scale = oracle.mul_mat_w8(oracle.quantize_q8_0(w), ne00, ne01, x)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert dst.shape == (ne11, ne01)
    assert np.all(np.abs(dst - ref) <= 1e-6 * scale + 1e-30)


@pytest.mark.parametrize("ne00,ne01,ne11", [(32, 1, 1), (256, 4, 3), (160, 5, 2)])
def test_w8_block_form_equals_decoded_brute_force(ne00, ne01, ne11):
    rng = np.random.default_rng([ne00, ne01, ne11, 9])
    w = (rng.standard_normal((ne01, ne00)) * 0.02).astype(np.float32)
    x = rng.standard_normal((ne11, ne00)).astype(np.float32)
    wq, xq = oracle.quantize_q8_0(w), oracle.quantize_q8_0(x)
    dst, scale = oracle.mul_mat_w8(wq, ne00, ne01, x)
    ref = oracle.dequantize_q8_0(xq, ne00).astype(np.float64) @ oracle.dequantize_q8_0(wq, ne00).astype(np.float64).T
    assert np.all(np.abs(dst - ref) <= 1e-6 * scale + 1e-30)
    d2, _ = oracle.mul_mat_w8_q8(wq, ne00, ne01, xq, ne11)
    np.testing.assert_array_equal(d2, dst)


def test_w8_isum_brute_force_tiny():
    rng = np.random.default_rng(45)
    for _ in range(20):
        a = rng.integers(-127, 128, size=32)
        b = rng.integers(-127, 128, size=32)
        xa = np.zeros(34, np.uint8)
        xa[2:] = a.astype(np.int8).view(np.uint8)
        yb = np.zeros(34, np.uint8)
        yb[2:] = b.astype(np.int8).view(np.uint8)
        want = sum(int(a[i]) * int(b[i]) for i in range(32))
        assert oracle.block_isums_w8(xa, yb, 32, 1, 1)[0, 0, 0] == want
    # extremes: 32 * 127 * 127 and its negative
    xa = np.zeros(34, np.uint8)
    xa[2:] = np.int8(-127).view(np.uint8)
    yb = np.zeros(34, np.uint8)
    yb[2:] = np.int8(127).view(np.uint8)
    assert oracle.block_isums_w8(xa, yb, 32, 1, 1)[0, 0, 0] == -32 * 127 * 127


def _golden(name):
    out = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split("=", 1)
                out[k.strip()] = v.strip()
    return out


def test_w8_two_block_tolerance_scale():
    # The Q8_0-weight contraction's tolerance scale on a hand-worked row whose two
    # block sums have opposite signs (tests/golden/two_block_scale.txt): S sums the
    # absolute block terms, dst keeps the sign of their sum.
    g = _golden("two_block_scale.txt")
    w = np.zeros((1, 64), np.float32)
    w[0, 0] = 127.0 / 128.0
    w[0, 32] = -127.0 / 256.0
    x = np.zeros((1, 64), np.float32)
    x[0, 0] = x[0, 32] = 127.0 / 128.0
    wq = oracle.quantize_q8_0(w)
    assert int.from_bytes(bytes(wq[0, :2]), "little") == 0x2000          # 2^-7
    assert int.from_bytes(bytes(wq[0, 34:36]), "little") == 0x1C00       # 2^-8
    isums = oracle.block_isums_w8(wq, oracle.quantize_q8_0(x), 64, 1, 1)[0, 0]
    np.testing.assert_array_equal(isums, [int(g["w8_isum_a"]), int(g["w8_isum_b"])])
    dst, scale = oracle.mul_mat_w8(wq, 64, 1, x)
    assert dst[0, 0] == np.float32(float(g["w8_dst"]))
    assert scale[0, 0] == float(g["w8_scale"])
    d2, s2 = oracle.mul_mat_w8_q8(wq, 64, 1, oracle.quantize_q8_0(x), 1)
    assert d2[0, 0] == dst[0, 0] and s2[0, 0] == scale[0, 0]
