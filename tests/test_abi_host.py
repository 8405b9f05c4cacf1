"""Host-side checks of the C ABI (no GPU): the library loads, exports every function the header
declares, the ctypes mirror of dsa_args matches the C layout, and argument validation rejects bad
calls before touching CUDA."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def native():
    from top_sparse_attention_gb300 import build

    build.build()
    from top_sparse_attention_gb300 import _native

    return _native


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(dsa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_expected_entry_points(native):
    decl = _declared_functions()
    assert set(decl) == set(native.EXPORTS), decl


def test_library_exports_every_declared_symbol(native):
    out = subprocess.run(["nm", "-D", "--defined-only", native.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(dsa_\w+)", out))
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(native.lib, name) is not None


def test_args_struct_layout_matches_c(tmp_path, native):
    fields = [f for f, _ in native.DsaArgs._fields_]
    src = tmp_path / "layout.c"
    body = "\n".join(f'  printf("{f} %zu\\n", offsetof(dsa_args, {f}));' for f in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dsa.h"\nint main(void){\n'
                   f'  printf("sizeof %zu\\n", sizeof(dsa_args));\n{body}\n  return 0;\n}}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.split("\n") if line)
    assert int(got["sizeof"]) == ctypes.sizeof(native.DsaArgs)
    for f in fields:
        assert int(got[f]) == getattr(native.DsaArgs, f).offset, f


def test_header_compiles_as_cxx(tmp_path):
    src = tmp_path / "x.cc"
    src.write_text('#include "dsa.h"\nint main(){ dsa_args a = {}; (void)a; return DSA_ABI_VERSION - 1; }\n')
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(tmp_path / "x")], check=True)


def test_status_strings_and_version(native):
    assert native.lib.dsa_abi_version() == 3
    for s in range(6):
        assert native.status_string(s).startswith("DSA_")
    assert "unknown" in native.status_string(99)


F = 16  # a fake, 16-byte aligned device address; validation rejects before it is ever used


def test_attention_kernel_switch(native):
    # host-only: the switch accepts the two documented kernels and rejects anything else
    assert native.lib.dsa_set_attn_kernel(7) == 1
    assert native.lib.dsa_set_attn_kernel(-1) == 1
    assert native.lib.dsa_set_attn_kernel(native.DSA_ATTN_TCGEN05) == 0
    # the workspace query covers the selected kernel: 128-row splits for the tensor-memory one
    tc = native.lib.dsa_sparse_attn_workspace_size(64, 16, 2048, 512)
    assert native.lib.dsa_set_attn_kernel(native.DSA_ATTN_AUTO) == 0
    auto = native.lib.dsa_sparse_attn_workspace_size(64, 16, 2048, 512)
    assert tc >= 64 * 16 * 16 * 512 * 4 and auto <= tc


def test_validation_rejects_before_any_launch(native):
    lib = native.lib
    # Top-K: K out of range, non-divisible grouping, null output
    assert lib.dsa_topk(F, 64, 2, 1, -1, None, 64, 0, F, None, 0, None) == 1
    assert lib.dsa_topk(F, 64, 2, 1, -1, None, 64, 5000, F, None, 0, None) == 2
    assert lib.dsa_topk(F, 64, 3, 2, -1, None, 64, 8, F, None, 0, None) == 1
    assert lib.dsa_topk(F, 64, 2, 1, -1, None, 64, 8, None, None, 0, None) == 1
    assert lib.dsa_topk(F, 32, 2, 1, -1, None, 64, 8, F, None, 0, None) == 1  # ld < L
    # index score: unsupported d_idx / dtype / heads; misaligned pointer; MXFP8 without scales
    # a base call that passes validation is never made here: it would launch on fake pointers
    base = [F, None, F, F, None, 8192, 0, 2, 1, -1, None, 32, 8, 128, 0, F, 32, None]
    bad = list(base); bad[13] = 96
    assert lib.dsa_index_score(*bad) == 2
    bad = list(base); bad[12] = 65
    assert lib.dsa_index_score(*bad) == 2
    bad = list(base); bad[14] = 7
    assert lib.dsa_index_score(*bad) == 2
    bad = list(base); bad[0] = F + 4
    assert lib.dsa_index_score(*bad) == 1
    bad = list(base); bad[14] = 2  # MXFP8 without scale pointers
    assert lib.dsa_index_score(*bad) == 1
    bad = list(base); bad[5] = 100  # sequence stride not a multiple of 16
    assert lib.dsa_index_score(*bad) == 1
    bad = list(base); bad[16] = 30  # ld_scores < L
    assert lib.dsa_index_score(*bad) == 1
    # sparse attention: unsupported dims, FP8 without scales, bad stride, too many heads
    sa = [F, F, None, None, 1152, 1152 * 64, 0, 0, F, 2, 1, 64, 16, 16, 576, 512, 0.04, 0, F, None,
          None, 0, None]
    bad = list(sa); bad[14] = 128
    assert lib.dsa_sparse_attn(*bad) == 2
    bad = list(sa); bad[17] = 1
    assert lib.dsa_sparse_attn(*bad) == 1
    bad = list(sa); bad[4] = 1000
    assert lib.dsa_sparse_attn(*bad) == 1
    bad = list(sa); bad[13] = 129
    assert lib.dsa_sparse_attn(*bad) == 2
    bad = list(sa); bad[12] = 0
    assert lib.dsa_sparse_attn(*bad) == 1


def test_quantiser_and_tiled_kv_validation(native):
    # every case returns from the host checks, which run before the device query (without a
    # device that query would answer DSA_ERR_CUDA = 4)
    lib = native.lib
    mx = lib.dsa_quantize_mxfp8  # (x, x_row_stride, rows, d, codes, sf, dst_rows, stream)
    assert mx(F, 100, 4, 100, F, F, None, None) == 1    # d not a multiple of 32
    assert mx(F, 64, 4, 128, F, F, None, None) == 1     # row pitch below d
    assert mx(F, 128, -1, 128, F, F, None, None) == 1   # negative row count
    assert mx(None, 128, 4, 128, F, F, None, None) == 1
    assert mx(F + 1, 128, 4, 128, F, F, None, None) == 1  # bf16 source not 2-byte aligned
    assert mx(F, 128, 0, 128, None, None, None, None) == 0  # no rows: nothing to do
    rows = lib.dsa_quantize_fp8_rows  # (x, x_row_stride, rows, width, codes, code_stride, scales, dst, stream)
    assert rows(F, 576, 4, 576, F, 500, F, None, None) == 1  # code pitch below the width
    assert rows(F, 576, 4, 576, F, 576, None, None, None) == 1  # no scale buffer
    tiles = lib.dsa_quantize_fp8_tiles  # (x, x_row_stride, rows, width, tile, codes, stride, scales, dst, stream)
    assert tiles(F, 576, 4, 576, 0, F, 576, F, None, None) == 1
    assert tiles(F, 576, 4, 576, 2048, F, 576, F, None, None) == 1  # tile above 1024
    # 128-element KV scale tiles: the 576 / 512 latent row only; a valid call passes validation and
    # stops at the missing workspace (3)
    sa = [F, F, None, F, 64, 64 * 64, 0, 0, F, 2, 1, 64, 16, 16, 64, 64, 0.125, 3, F, None, None, 0, None]
    assert lib.dsa_sparse_attn(*sa) == 2
    sa = [F, F, None, F, 576, 576 * 64, 0, 0, F, 2, 1, 64, 2048, 16, 576, 512, 0.04, 3, F, None, None, 0,
          None]
    assert lib.dsa_sparse_attn(*sa) == 3
    sa[3] = None  # tiled scales missing
    assert lib.dsa_sparse_attn(*sa) == 1


def test_fused_validation(native):
    a = native.DsaArgs()
    a.T, a.q_per_seq, a.q_pos0, a.L, a.K = 2, 1, -1, 64, 8
    a.H_idx, a.d_idx, a.H, a.D_qk, a.D_v = 4, 64, 1, 64, 64
    a.sm_scale = 0.125
    a.q_idx = a.w = a.k_idx = a.q = a.kv = a.out = F
    a.k_seq_stride = 64 * 128
    a.kv_row_stride, a.kv_seq_stride = 128, 128 * 64
    n = ctypes.c_size_t(0)
    assert native.lib.dsa_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value >= 2 * 64 * 4
    # launches per call: index score, Top-K, attention (+ combine when K is split over CTAs)
    c = ctypes.c_int(-1)
    assert native.lib.dsa_launch_count(ctypes.byref(a), 0, ctypes.byref(c)) == 0
    assert c.value in (3, 4)
    assert native.lib.dsa_launch_count(ctypes.byref(a), 0, None) == 1
    # a row long enough for the row-split Top-K (three kernels after the fused histogram)
    a.L, a.K = 300000, 2048
    a.k_seq_stride = 300000 * 128
    a.kv_seq_stride = 128 * 300000
    assert native.lib.dsa_launch_count(ctypes.byref(a), 0, ctypes.byref(c)) == 0
    assert c.value in (5, 6)
    a.L, a.K, a.k_seq_stride, a.kv_seq_stride = 64, 8, 64 * 128, 128 * 64
    # decode entry with a causal q_pos0, prefill entry without one, and a block table
    assert native.lib.dsa_workspace_size(ctypes.byref(a), 1, ctypes.byref(n)) == 1
    # a block table with a block size that is not a multiple of 64, or too few entries per sequence
    a.block_table = F
    a.block_size, a.max_blocks, a.num_blocks = 48, 2, 4
    assert native.lib.dsa_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 1
    a.block_size, a.max_blocks = 64, 0
    assert native.lib.dsa_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 1
    a.max_blocks = 1
    assert native.lib.dsa_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    a.block_table = None
    a.block_size = a.max_blocks = a.num_blocks = 0
    # too-small workspace is reported before any launch
    assert native.lib.dsa_decode(ctypes.byref(a), F, 16, None) == 3
    assert native.lib.dsa_decode(None, F, 16, None) == 1


def test_product_package_does_not_import_the_oracle():
    code = ("import sys; sys.path.insert(0, %r); import top_sparse_attention_gb300; "
            "assert 'oracle' not in sys.modules and 'synth' not in sys.modules" % ROOT)
    subprocess.run([sys.executable, "-c", code], check=True)
