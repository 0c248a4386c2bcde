"""The C-ABI library builds, loads and exports what include/q4q.h declares (CPU).

Also checks the host-side argument validation, which returns before any CUDA
call and therefore runs without a GPU.
"""
import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from q4_quantized_matmul_gb300 import _lib
    return _lib.load()


def test_header_declares_the_boundary():
    from q4_quantized_matmul_gb300 import _lib
    names = set(_lib.declared_entry_points())
    assert {"q4q_quantize_q4_0", "q4q_quantize_q8_0", "q4q_mul_mat", "q4q_mul_mat_ex", "q4q_mul_mat_workspace_size",
            "q4q_debug_block_isums", "q4q_debug_workspace_size", "q4q_device_status", "q4q_status_string",
            "q4q_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    from q4_quantized_matmul_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _lib.declared_entry_points():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else leaks out under the q4q_ prefix
    assert {n for n in exported if n.startswith("q4q_")} == set(_lib.declared_entry_points())


def test_header_compiles_as_c():
    src = '#include "q4q.h"\nint main(void){ return (int)sizeof(q4q_block_q4_0) + (int)sizeof(q4q_block_q8_0); }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-x", "c", "-", "-o", "/dev/null"], input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr


def test_block_struct_sizes():
    src = ('#include "q4q.h"\n#include <stdio.h>\nint main(void){ printf("%d %d", (int)sizeof(q4q_block_q4_0),'
           ' (int)sizeof(q4q_block_q8_0)); return 0; }\n')
    exe = "/tmp/q4q_sizes_%d" % os.getpid()
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-x", "c", "-", "-o", exe],
                   input=src, text=True, check=True)
    try:
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    finally:
        os.unlink(exe)
    assert out == "18 34"


def test_version_and_strings(lib):
    assert lib.q4q_version() >> 16 == 1
    assert lib.q4q_status_string(0) == b"ok"
    assert lib.q4q_status_string(3) == b"misaligned pointer"
    assert lib.q4q_status_string(99) == b"unknown status"


def test_argument_errors_need_no_gpu(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # ne00 not a multiple of 32
    assert lib.q4q_mul_mat(fake, 33, 4, fake, 33, 1, fake, None, 0, None) == 2
    # ne10 != ne00
    assert lib.q4q_mul_mat(fake, 64, 4, fake, 96, 1, fake, None, 0, None) == 2
    # negative sizes
    assert lib.q4q_mul_mat(fake, 64, -1, fake, 64, 1, fake, None, 0, None) == 2
    assert lib.q4q_mul_mat(fake, 64, 4, fake, 64, -1, fake, None, 0, None) == 2
    # empty problems are valid and launch nothing
    assert lib.q4q_mul_mat(None, 64, 0, None, 64, 3, None, None, 0, None) == 0
    assert lib.q4q_mul_mat(None, 64, 5, None, 64, 0, None, None, 0, None) == 0
    # null pointers
    assert lib.q4q_mul_mat(None, 64, 4, fake, 64, 1, fake, None, 0, None) == 1
    assert lib.q4q_mul_mat(fake, 64, 4, fake, 64, 1, None, None, 0, None) == 1
    # misaligned pointers
    assert lib.q4q_mul_mat(P(0x1001), 64, 4, fake, 64, 1, fake, None, 0, None) == 3
    assert lib.q4q_mul_mat(fake, 64, 4, P(0x1002), 64, 1, fake, None, 0, None) == 3
    # quantizers
    assert lib.q4q_quantize_q4_0(fake, fake, 31, 2, None) == 2
    assert lib.q4q_quantize_q8_0(fake, fake, 0, 2, None) == 2
    assert lib.q4q_quantize_q4_0(fake, fake, 32, 0, None) == 0
    assert lib.q4q_quantize_q4_0(None, fake, 32, 1, None) == 1
    assert lib.q4q_quantize_q8_0(P(0x1002), fake, 32, 1, None) == 3
    # debug entry
    assert lib.q4q_debug_block_isums(fake, fake, 64, 2, 1, 5, fake, None, 0, None) == 7
    assert lib.q4q_debug_block_isums(fake, fake, 64, 0, 1, 0, fake, None, 0, None) == 0
    assert lib.q4q_debug_workspace_size(64, 1, 0, ctypes.byref(ctypes.c_size_t())) == 0
    assert lib.q4q_debug_workspace_size(64, 1, 2, ctypes.byref(ctypes.c_size_t())) == 7
    # unknown launch flags
    assert lib.q4q_mul_mat_ex(fake, 64, 4, fake, 64, 1, fake, None, 0, 2, None) == 7
    # workspace query
    n = ctypes.c_size_t(123)
    assert lib.q4q_mul_mat_workspace_size(64, 4, 1, None) == 1
    assert lib.q4q_mul_mat_workspace_size(48, 4, 1, ctypes.byref(n)) == 2
    assert lib.q4q_mul_mat_workspace_size(64, 4, 3, ctypes.byref(n)) == 0
    assert n.value == 3 * 2 * 34


def test_binding_fails_loudly_without_cuda_tensors(lib):
    import torch
    import q4_quantized_matmul_gb300 as q4q
    with pytest.raises(TypeError):
        q4q.q4q_quantize_q4_0(torch.zeros(2, 32))


def test_argument_errors_of_the_entry_points_next_to_the_matmul(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    n = ctypes.c_size_t(0)
    # bias / activation
    assert lib.q4q_mul_mat_bias_act(fake, 33, 4, fake, 33, 1, fake, 0, fake, None, 0, 0, None) == 2
    assert lib.q4q_mul_mat_bias_act(fake, 64, 4, fake, 64, 1, fake, 2, fake, None, 0, 0, None) == 7
    assert lib.q4q_mul_mat_bias_act(fake, 64, 4, fake, 64, 1, fake, 0, fake, None, 0, 4, None) == 7
    assert lib.q4q_mul_mat_bias_act(fake, 64, 4, fake, 64, 1, P(0x1002), 1, fake, None, 0, 0, None) == 3
    assert lib.q4q_mul_mat_bias_act(fake, 64, 4, fake, 64, 1, None, 0, None, None, 0, 0, None) == 1
    assert lib.q4q_mul_mat_bias_act(None, 64, 0, None, 64, 1, None, 1, None, None, 0, 0, None) == 0
    # SwiGLU
    assert lib.q4q_mul_mat_swiglu(fake, fake, 64, 4, fake, 96, 1, fake, None, 0, 0, None) == 2
    assert lib.q4q_mul_mat_swiglu(fake, None, 64, 4, fake, 64, 1, fake, None, 0, 0, None) == 1
    assert lib.q4q_mul_mat_swiglu(fake, P(0x1001), 64, 4, fake, 64, 1, fake, None, 0, 0, None) == 3
    assert lib.q4q_mul_mat_swiglu(fake, fake, 64, 4, fake, 64, 1, fake, None, 0, 8, None) == 7
    assert lib.q4q_mul_mat_swiglu(None, None, 64, 4, None, 64, 0, None, None, 0, 0, None) == 0
    assert lib.q4q_mul_mat_swiglu_workspace_size(64, 4, 3, None) == 1
    # get_rows
    for fn in (lib.q4q_get_rows_q4_0, lib.q4q_get_rows_q8_0):
        assert fn(fake, 48, 10, fake, 3, fake, None) == 2
        assert fn(fake, 64, 10, None, 11, fake, None) == 2      # whole-table decode past the end
        assert fn(fake, 64, 10, fake, -1, fake, None) == 2
        assert fn(fake, 64, 10, fake, 0, fake, None) == 0
        assert fn(None, 64, 10, fake, 3, fake, None) == 1
        assert fn(fake, 64, 10, fake, 3, P(0x1004), None) == 3   # dst not 16-byte aligned
        assert fn(fake, 64, 10, P(0x1002), 3, fake, None) == 3
    # Q8_0 weights
    assert lib.q4q_mul_mat_q8_0(fake, 33, 4, fake, 33, 1, fake, None, 0, 0, None) == 2
    assert lib.q4q_mul_mat_q8_0(P(0x1001), 64, 4, fake, 64, 1, fake, None, 0, 0, None) == 3
    assert lib.q4q_mul_mat_q8_0(fake, 64, 4, fake, 64, 1, fake, None, 0, 2, None) == 7
    assert lib.q4q_mul_mat_q8_0(None, 64, 0, None, 64, 1, None, None, 0, 0, None) == 0
    assert lib.q4q_mul_mat_q8_0_workspace_size(64, 4, 3, ctypes.byref(n)) == 0
    assert n.value == 3 * 2 * 34
    assert lib.q4q_debug_block_isums_q8_0(fake, fake, 48, 2, 1, 0, fake, None, 0, None) == 2
    assert lib.q4q_debug_block_isums_q8_0(fake, None, 64, 2, 1, 0, fake, None, 0, None) == 1
    assert lib.q4q_debug_block_isums_q8_0(fake, fake, 64, 2, 1, 3, fake, None, 0, None) == 7


def test_new_bindings_fail_loudly_without_cuda_tensors(lib):
    import torch
    import q4_quantized_matmul_gb300 as q4q
    w = torch.zeros(4 * 18 * 2, dtype=torch.uint8)
    with pytest.raises(TypeError):
        q4q.q4q_get_rows_q4_0(w, 64, 4, ids=torch.zeros(2, dtype=torch.int32))


def test_argument_errors_of_the_group_entry(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    fake = 0x1000
    ptrs = (P * 4)(fake, fake, fake, fake)
    rows = (I64 * 4)(4, 4, 4, 4)
    n = ctypes.c_size_t(0)
    assert lib.q4q_mul_mat_group(0, ptrs, rows, 64, P(fake), 64, 1, ptrs, None, 0, 0, None) == 7
    assert lib.q4q_mul_mat_group(5, ptrs, rows, 64, P(fake), 64, 1, ptrs, None, 0, 0, None) == 7
    assert lib.q4q_mul_mat_group(2, None, rows, 64, P(fake), 64, 1, ptrs, None, 0, 0, None) == 1
    assert lib.q4q_mul_mat_group(2, ptrs, rows, 48, P(fake), 48, 1, ptrs, None, 0, 0, None) == 2
    assert lib.q4q_mul_mat_group(2, ptrs, rows, 64, P(fake), 64, 1, ptrs, None, 0, 2, None) == 7
    bad = (P * 2)(fake, fake + 1)
    assert lib.q4q_mul_mat_group(2, bad, rows, 64, P(fake), 64, 1, ptrs, None, 0, 0, None) == 3
    zero = (I64 * 2)(0, 0)
    assert lib.q4q_mul_mat_group(2, ptrs, zero, 64, None, 64, 1, ptrs, None, 0, 0, None) == 0
    assert lib.q4q_mul_mat_group_workspace_size(2, rows, 64, 3, None) == 1
    assert lib.q4q_mul_mat_group_workspace_size(9, rows, 64, 3, ctypes.byref(n)) == 7


def test_wait_timeout_argument_errors(lib):
    assert lib.q4q_debug_wait_timeout(0, None) == 7
    assert lib.q4q_debug_wait_timeout(2 * 10 ** 9, None) == 7


def test_path_entry_argument_errors(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    f = lib.q4q_debug_mul_mat_path
    assert f(fake, 256, 4, fake, 1, fake, None, 0, 2, None) == 7                   # the chain is no path here
    assert f(fake, 256, 4, fake, 1, fake, None, 0, 4, None) == 7                   # unknown path
    assert f(fake, 48, 4, fake, 1, fake, None, 0, 0, None) == 2                    # ne00 % 32
    assert f(fake, 256, 0, fake, 1, fake, None, 0, 3, None) == 2                   # nothing to run
    assert f(None, 256, 4, fake, 1, fake, None, 0, 3, None) == 1
    assert f(P(0x1008), 256, 4, fake, 1, fake, None, 0, 3, None) == 3              # src0 not 16-byte aligned
    n = ctypes.c_size_t(7)
    g = lib.q4q_debug_mul_mat_path_workspace_size
    assert g(256, 4, 1, 0, ctypes.byref(n)) == 0 and n.value == 0                  # the GEMV needs none
    assert g(256, 4, 1, 5, ctypes.byref(n)) == 7
    assert g(256, 4, 1, 3, None) == 1


def test_kernel_timeout_entry_argument_errors(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    f = lib.q4q_debug_mul_mat_timeout
    assert f(fake, 256, 4, fake, 1, fake, None, 0, 4, 10 ** 6, None) == 7          # unknown path
    assert f(fake, 256, 4, fake, 1, fake, None, 0, 0, 0, None) == 7                # limit 0
    assert f(fake, 256, 4, fake, 1, fake, None, 0, 0, 2 * 10 ** 9, None) == 7      # limit above 1 s
    assert f(fake, 48, 4, fake, 1, fake, None, 0, 0, 10 ** 6, None) == 2           # ne00 % 32
    assert f(fake, 256, 0, fake, 1, fake, None, 0, 0, 10 ** 6, None) == 2          # nothing to run
    assert f(None, 256, 4, fake, 1, fake, None, 0, 0, 10 ** 6, None) == 1


def test_c_program_links_and_calls_the_library(lib):
    """A plain C99 caller: includes q4q.h, links libq4q.so and makes the calls that
    need no GPU (version, status strings, argument errors, host-only planning)."""
    from q4_quantized_matmul_gb300 import _lib
    src = r"""
#include <stdio.h>
#include <string.h>
#include "q4q.h"
int main(void) {
    int64_t plan[Q4Q_DEBUG_GEMV_PLAN_FIELDS];
    int splits = 0;
    size_t ws = 0;
    if ((q4q_version() >> 16) != 1) return 1;
    if (strcmp(q4q_status_string(Q4Q_ERR_SHAPE), "invalid shape") != 0) return 2;
    if (q4q_mul_mat((const void*)0x1000, 33, 4, (const float*)0x1000, 33, 1, (float*)0x1000, NULL, 0, NULL)
        != Q4Q_ERR_SHAPE) return 3;
    if (q4q_mul_mat_workspace_size(64, 4, 3, &ws) != Q4Q_OK || ws != 3 * 2 * 34) return 4;
    if (q4q_debug_gemv_plan(4096, 128256, 1, Q4Q_BLOCK_Q4_0_BYTES, 1, 152, 232448, plan) != Q4Q_OK) return 5;
    if (plan[0] != 8 || plan[4] != 304) return 6;
    if (q4q_debug_mma_splits(4096, 1024, 8, 152, &splits) != Q4Q_OK || splits != 8) return 7;
    if (q4q_get_rows_q4_0((const void*)0x1000, 48, 10, NULL, 3, (float*)0x1000, NULL) != Q4Q_ERR_SHAPE) return 8;
    printf("ok\n");
    return 0;
}
"""
    exe = "/tmp/q4q_c_caller_%d" % os.getpid()
    build_dir = os.path.dirname(_lib.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-x", "c", "-",
                        "-L", build_dir, "-lq4q", "-Wl,-rpath," + build_dir, "-o", exe],
                       input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr
    try:
        out = subprocess.run([exe], capture_output=True, text=True)
    finally:
        os.unlink(exe)
    assert out.returncode == 0 and out.stdout == "ok\n", (out.returncode, out.stdout, out.stderr)


def test_chain_argument_errors(lib):
    import q4_quantized_matmul_gb300 as q4q
    P = ctypes.c_void_p
    fake = 0x1000
    links = (q4q.ChainLink * 3)(*[q4q.ChainLink(fake, 256, 4, fake, fake) for _ in range(3)])
    n = ctypes.c_size_t(0)
    assert lib.q4q_mul_mat_chain_workspace_size(3, ctypes.byref(n)) == 0 and n.value == 256
    assert lib.q4q_mul_mat_chain_workspace_size(0, ctypes.byref(n)) == 7
    assert lib.q4q_mul_mat_chain_workspace_size(65, ctypes.byref(n)) == 7
    assert lib.q4q_mul_mat_chain_workspace_size(3, None) == 1
    ws = P(fake)
    assert lib.q4q_mul_mat_chain(links, 0, 1, ws, 256, 0, None) == 7          # no links
    assert lib.q4q_mul_mat_chain(links, 65, 1, ws, 256, 0, None) == 7         # above Q4Q_CHAIN_MAX
    assert lib.q4q_mul_mat_chain(links, 3, 1, ws, 256, 1, None) == 7          # flags must be 0
    assert lib.q4q_mul_mat_chain(None, 3, 1, ws, 256, 0, None) == 1
    assert lib.q4q_mul_mat_chain(links, 3, 2, ws, 256, 0, None) == 2          # one token only
    assert lib.q4q_mul_mat_chain(links, 3, 1, ws, 16, 0, None) == 4           # workspace too small
    assert lib.q4q_mul_mat_chain(links, 3, 1, None, 256, 0, None) == 1
    links[1].ne00 = 288                                                        # ne00 % 256 != 0
    assert lib.q4q_mul_mat_chain(links, 3, 1, ws, 256, 0, None) == 2
    links[1].ne00 = 256
    links[2].ne01 = 0
    assert lib.q4q_mul_mat_chain(links, 3, 1, ws, 256, 0, None) == 2
    links[2].ne01 = 4
    links[0].src1 = fake + 4                                                   # src1 not 16-byte aligned
    assert lib.q4q_mul_mat_chain(links, 3, 1, ws, 256, 0, None) == 3
    links[0].src1 = fake
    links[2].dst = None
    assert lib.q4q_mul_mat_chain(links, 3, 1, ws, 256, 0, None) == 1
