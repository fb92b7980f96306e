"""C-ABI checks that need no GPU: the library loads, exports every function
that include/poetx.h declares, and its host-side logic (permutation
generator, generator lengths, argument checks) behaves as documented.

No call here launches a kernel: argument errors are returned before any
launch, and the permutation generator runs on the host.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle as O
import orthogonal_equivalence_reparameterized_poetx_b300 as px

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "poetx.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(poetx_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported():
    declared = _declared_functions()
    assert len(declared) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", px.lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (poetx_[a-z0-9_]+)$", out, flags=re.M))
    missing = [f for f in declared if f not in exported]
    assert not missing, missing
    assert sorted(px.EXPORTED_SYMBOLS) == declared


def test_library_is_sm103a_only_build():
    # the binding loaded the in-tree library built for sm_103a
    assert os.path.dirname(px.lib_path).endswith("orthogonal_equivalence_reparameterized_poetx_b300")
    assert px.poetx_version() == 1000


def test_desc_struct_layout_matches_header():
    assert ctypes.sizeof(px.poetx_layer_desc) == 48
    assert px.poetx_layer_desc.seed_R.offset == 16
    assert px.poetx_layer_desc.mode.offset == 32


@pytest.mark.parametrize("seed,d", [(0, 4), (0, 5), (1, 1), (7, 2), (6000, 256), (6003, 1376),
                                    (7001, 5632), (6000, 11008), (2**64 - 1, 33)])
def test_host_permutation_bit_exact_with_oracle(seed, d):
    got = px.poetx_perm_generate(seed, d)
    want = O.permutation(seed, d)
    assert got.dtype == np.int32
    assert np.array_equal(got.astype(np.int64), want)


@pytest.mark.parametrize("d,b", [(256, 32), (1376, 32), (11008, 512), (7, 4), (9, 9), (5, 1)])
def test_gen_length_matches_oracle(d, b):
    assert px.poetx_gen_length(d, b) == O.packed_length(d, b)


def test_gen_length_rejects_bad_sizes():
    assert px.poetx_gen_length(0, 1) == -1
    assert px.poetx_gen_length(8, 9) == -1
    assert px.poetx_gen_length(8, 0) == -1


def test_params_size_validation():
    good = px.make_desc(512, 1376, 32, 32, 1, 2, dtype="bf16")
    assert px.poetx_params_size(good) > 0
    bad = [
        px.make_desc(512, 1376, 48, 32, 1, 2, dtype="bf16"),     # b not in the bf16 set
        px.make_desc(512, 1372, 32, 32, 1, 2, dtype="bf16"),     # n % 8 != 0
        px.make_desc(0, 16, 1, 1, 1, 2, dtype="fp32"),           # m < 1
        px.make_desc(16, 16, 32, 4, 1, 2, dtype="fp32"),         # b > d
        px.make_desc(512, 512, 200, 32, 1, 2, dtype="fp32"),     # fp32 b > 128 not a multiple of 128
    ]
    for d in bad:
        assert px.poetx_params_size(d) == 0
    d = px.make_desc(64, 64, 8, 8, 1, 2, dtype="fp32")
    d.weight_format = 7
    assert px.poetx_params_size(d) == 0
    # POET-XQ int8 storage is for bf16 layers only
    assert px.poetx_params_size(px.make_desc(64, 64, 8, 8, 1, 2, dtype="fp32", weight="int8")) == 0
    q = px.make_desc(96, 64, 32, 32, 1, 2, dtype="bf16", weight="int8")
    assert px.poetx_params_size(q) > 0
    # codes padded to 256 bytes, then one float scale per row
    assert px.poetx_weight_size(q) == 96 * 64 + 512
    assert px.poetx_weight_size(px.make_desc(96, 64, 32, 32, 1, 2, dtype="bf16")) == 96 * 64 * 2
    assert px.poetx_workspace_size(q, 10) > px.poetx_workspace_size(
        px.make_desc(96, 64, 32, 32, 1, 2, dtype="bf16"), 10)
    d = px.make_desc(64, 64, 8, 8, 1, 2, dtype="fp32", mode="neumann", neumann_k=0)
    assert px.poetx_params_size(d) == 0


def test_argument_errors_return_before_launch():
    d = px.make_desc(64, 64, 8, 8, 1, 2, dtype="fp32")
    L = px.LIB
    D = ctypes.byref(d)
    # null params / workspace
    assert L.poetx_linear_fwd(D, None, 256, 256, 4, 256, None, None, 256, None) == px.POETX_ERR_INVALID_ARG
    # misaligned tensor pointer (not 16-byte aligned)
    assert L.poetx_linear_fwd(D, 256, 264 + 2, 256, 4, 256, None, None, 256, None) == px.POETX_ERR_MISALIGNED
    # misaligned params buffer (not 256-byte aligned)
    assert L.poetx_linear_fwd(D, 272, 256, 256, 4, 256, None, None, 256, None) == px.POETX_ERR_MISALIGNED
    # negative token count
    assert L.poetx_linear_fwd(D, 256, 256, 256, -1, 256, None, None, 256, None) == px.POETX_ERR_INVALID_ARG
    # T == 0 is a no-op
    assert L.poetx_linear_fwd(D, 256, 256, 256, 0, 256, None, None, 256, None) == px.POETX_OK
    # backward needs generator-gradient outputs
    assert L.poetx_linear_bwd(D, 256, 256, 256, 256, None, None, 4, None, None, None, 0, 256,
                              None) == px.POETX_ERR_INVALID_ARG
    # a saved u must not alias the input or the output
    assert L.poetx_linear_fwd(D, 256, 256, 512, 4, 768, None, 512, 256, None) == px.POETX_ERR_INVALID_ARG
    assert L.poetx_linear_fwd(D, 256, 256, 512, 4, 768, None, 768, 256, None) == px.POETX_ERR_INVALID_ARG
    # the backward needs X or a saved u
    assert L.poetx_linear_bwd(D, 256, 256, None, 256, None, None, 4, None, 256, 256, 0, 256,
                              None) == px.POETX_ERR_INVALID_ARG
    # the host step needs both host inputs, both device input buffers and
    # both host gradient outputs (checked before any copy)
    for missing in range(6):
        ptrs = [256] * 6
        ptrs[missing] = None
        xh, dyh, xd, dyd, gh_r, gh_p = ptrs
        assert L.poetx_linear_step_host(D, 256, 256, xh, dyh, 4, xd, dyd, 256, None, None, None,
                                        256, 256, gh_r, gh_p, 256, None) == px.POETX_ERR_INVALID_ARG
    assert L.poetx_linear_step_host(D, 256, 256, 256, 256, -1, 256, 256, 256, None, None, None,
                                    256, 256, 256, 256, 256, None) == px.POETX_ERR_INVALID_ARG
    assert L.poetx_linear_step_host_async(D, 256, 256, None, 256, 4, 256, 256, 256, None, None,
                                          None, 256, 256, 256, 256, 256,
                                          None) == px.POETX_ERR_INVALID_ARG
    # token counts the kernels cannot index are refused before any copy
    assert L.poetx_linear_step_host(D, 256, 256, 256, 256, 1 << 31, 256, 256, 256, None, None, None,
                                    256, 256, 256, 256, 256, None) == px.POETX_ERR_UNSUPPORTED
    # invalid descriptor
    bad = px.make_desc(64, 64, 8, 8, 1, 2, dtype="fp32")
    bad.mode = 7
    assert L.poetx_params_build(ctypes.byref(bad), 256, 256, 256, None) == px.POETX_ERR_INVALID_ARG
    assert L.poetx_perm_generate(1, 0, None) == px.POETX_ERR_INVALID_ARG
    assert px.poetx_status_string(px.POETX_ERR_TIMEOUT) == "POETX_ERR_TIMEOUT"


def test_workspace_size_scales_with_tokens():
    d = px.make_desc(2048, 2048, 128, 128, 1, 2, dtype="bf16")
    a = px.poetx_workspace_size(d, 1024)
    b = px.poetx_workspace_size(d, 65536)
    assert 0 < a < b
    # five activation-sized bf16 buffers at least
    assert b >= 5 * 65536 * 2048 * 2
