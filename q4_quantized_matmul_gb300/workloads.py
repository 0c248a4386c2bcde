"""Seeded synthetic inputs for the Q4_0 matmul workloads.

This module only draws random fp32 numbers; it holds none of the method's
arithmetic (no quantization, no dot products).  Both the CUDA path and the CPU
oracle consume what it produces, so they always see identical inputs.

Workload shapes follow the pages' models:
  * GPT-2 117M projections (d = 768, 4d = 3072, vocab 50257) from the "ggml GPT-2
    117M inference walkthrough" (aicoding.csdn.net), hyper-parameter list and
    §3.2 / §3.5 / §3.6 (c_attn 768->2304, c_proj 768->768, c_fc 768->3072,
    c_mlp_proj 3072->768, lm_head 768->50257).
  * Llama-3-8B-shaped projections (hidden 4096, vocab 128256, from the GGUF
    metadata example in "llama.cpp 深度解读" §1) with 8 kv heads x 128, FFN 14336.
Every matrix of a workload gets its own generator, seeded by (seed, index), so a
single matrix can be regenerated without drawing the others.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    shapes: Tuple[Tuple[int, int], ...]   # (ne00 = K, ne01 = rows) per projection
    ne11: Tuple[int, ...]                 # token counts to run
    seed: int
    weights: str                          # distribution recipe key
    acts: str

    @property
    def n_matrices(self) -> int:
        return len(self.shapes)

    def weight_count(self) -> int:
        return sum(k * n for k, n in self.shapes)


_GPT2_LAYER = ((768, 2304), (768, 768), (768, 3072), (3072, 768))
_LLAMA_SET = ((4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096),
              (4096, 14336), (4096, 14336), (14336, 4096), (4096, 128256))

WORKLOADS = {
    "gpt2_c_attn_1tok": Workload(
        "gpt2_c_attn_1tok",
        "GPT-2 117M c_attn 768->2304, 1 token; W ~ N(0,0.02), x ~ N(0,1); seed 0",
        ((768, 2304),), (1,), 0, "normal", "normal"),
    "gpt2_decode_step": Workload(
        "gpt2_decode_step",
        "GPT-2 117M decode-step weight set, 1 token: 12 layers x {768->2304, 768->768, "
        "768->3072, 3072->768} + lm_head 768->50257; W ~ N(0,0.02), x ~ N(0,1); seed 1",
        _GPT2_LAYER * 12 + ((768, 50257),), (1,), 1, "normal", "normal"),
    "llama3_8b_decode": Workload(
        "llama3_8b_decode",
        "Llama-3-8B-shaped projections q,k,v,o,gate,up,down,lm_head at 1 token; "
        "W ~ N(0,0.02) with 0.1% of weights x20; x ~ N(0,1) with 1% of channels x10; seed 2",
        _LLAMA_SET, (1,), 2, "normal_outliers", "normal_hot_channels"),
    "llama3_8b_batched": Workload(
        "llama3_8b_batched",
        "Llama-3-8B-shaped projections at 8, 64 and 512 tokens; W ~ N(0,0.02), x ~ N(0,1); seed 3",
        _LLAMA_SET, (8, 64, 512), 3, "normal", "normal"),
    "stress_prefill": Workload(
        "stress_prefill",
        "lm_head 4096->128256 and down 14336->4096 at 2048 tokens; W = 0.02 * Student-t(3) with "
        "5% of 32-blocks zero and 1% constant; x = Student-t(3) with 0.5% of rows zero; seed 4",
        ((4096, 128256), (14336, 4096)), (2048,), 4, "t3_blocks", "t3_zero_rows"),
}

# the order in which the workloads are usually listed (small oracle case first)
WORKLOAD_ORDER = ["gpt2_c_attn_1tok", "gpt2_decode_step", "llama3_8b_decode",
                  "llama3_8b_batched", "stress_prefill"]


def _rng(seed: int, index: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(index), int(stream)])


def gen_weights(recipe: str, ne01: int, ne00: int, seed: int, index: int) -> np.ndarray:
    """fp32 [ne01, ne00] (row i01 holds the ne00 inputs of output i01)."""
    rng = _rng(seed, index, 0)
    if recipe == "normal":
        w = rng.standard_normal((ne01, ne00), dtype=np.float32)
        w *= np.float32(0.02)
        return w
    if recipe == "normal_outliers":
        w = rng.standard_normal((ne01, ne00), dtype=np.float32)
        w *= np.float32(0.02)
        n = w.size
        k = max(1, n // 1000)
        idx = rng.integers(0, n, size=k)
        flat = w.reshape(-1)
        flat[idx] *= np.float32(20.0)
        return w
    if recipe == "t3_blocks":
        w = rng.standard_t(3, size=(ne01, ne00)).astype(np.float32)
        w *= np.float32(0.02)
        blocks = w.reshape(-1, 32)
        nb = blocks.shape[0]
        zero = rng.integers(0, nb, size=max(1, nb // 20))
        const = rng.integers(0, nb, size=max(1, nb // 100))
        blocks[zero] = 0.0
        blocks[const] = blocks[const, :1]
        return w
    raise ValueError("unknown weight recipe %r" % recipe)


def gen_acts(recipe: str, ne11: int, ne10: int, seed: int, index: int) -> np.ndarray:
    """fp32 [ne11, ne10] (row i11 is token i11)."""
    rng = _rng(seed, index, 1 + ne11)
    if recipe == "normal":
        return rng.standard_normal((ne11, ne10), dtype=np.float32)
    if recipe == "normal_hot_channels":
        x = rng.standard_normal((ne11, ne10), dtype=np.float32)
        k = max(1, ne10 // 100)
        ch = rng.choice(ne10, size=k, replace=False)
        x[:, ch] *= np.float32(10.0)
        return x
    if recipe == "t3_zero_rows":
        x = rng.standard_t(3, size=(ne11, ne10)).astype(np.float32)
        k = max(1, (ne11 * 5) // 1000)
        rows = rng.choice(ne11, size=k, replace=False)
        x[rows] = 0.0
        return x
    raise ValueError("unknown activation recipe %r" % recipe)


def problem(name: str, index: int, ne11: Optional[int] = None):
    """(W fp32 [ne01, ne00], X fp32 [ne11, ne00]) for matrix `index` of workload `name`."""
    wl = WORKLOADS[name]
    ne00, ne01 = wl.shapes[index]
    t = wl.ne11[0] if ne11 is None else int(ne11)
    w = gen_weights(wl.weights, ne01, ne00, wl.seed, index)
    x = gen_acts(wl.acts, t, ne00, wl.seed, index)
    return w, x


def random_problem(ne00: int, ne01: int, ne11: int, seed: int, wscale: float = 0.02):
    """Small ad-hoc problem for edge-case tests: W ~ N(0, wscale), X ~ N(0, 1)."""
    rng = np.random.default_rng([int(seed), ne00, ne01, ne11])
    w = rng.standard_normal((ne01, ne00), dtype=np.float32) * np.float32(wscale)
    x = rng.standard_normal((ne11, ne00), dtype=np.float32)
    return w, x


def gen_bias(ne01: int, seed: int, index: int, scale: float = 0.1) -> np.ndarray:
    """fp32 [ne01] projection bias ~ N(0, scale), for the bias epilogues (its own stream)."""
    rng = _rng(seed, index, 1 << 20)
    b = rng.standard_normal(ne01, dtype=np.float32)
    b *= np.float32(scale)
    return b
