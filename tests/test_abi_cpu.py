"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import gemm_affine_int4_gb300 as g4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gai4.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gai4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(g4.LIB_PATH):
        from gemm_affine_int4_gb300 import build
        build.build()
    return g4.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("gai4_qmv", "gai4_qmm_t", "gai4_quantize", "gai4_q8_0_gemv", "gai4_q4_k_gemv"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    # and the Python binding knows the signature of each
    assert sorted(g4.SIGNATURES) == _declared()


def test_status_strings(lib):
    for st in range(7):
        s = g4.gai4_status_string(st)
        assert s and s != "unknown status"
    assert g4.gai4_status_string(99) == "unknown status"
    assert g4.gai4_version() >= 100


P = ctypes.c_void_p


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_rejects_bad_arguments_without_launching(lib):
    A = _fake()
    # null pointers
    assert lib.gai4_qmv(None, A, A, A, A, 2, 4, 64, 16, 64, None) == g4.GAI4_ERR_INVALID_ARG
    # K not a multiple of the group size
    assert lib.gai4_qmv(A, A, A, A, A, 2, 4, 64, 16, 96, None) == g4.GAI4_ERR_INVALID_ARG
    # unsupported width / group size / dtype
    assert lib.gai4_qmv(A, A, A, A, A, 2, 5, 64, 16, 64, None) == g4.GAI4_ERR_UNSUPPORTED
    assert lib.gai4_qmv(A, A, A, A, A, 2, 4, 48, 16, 96, None) == g4.GAI4_ERR_UNSUPPORTED
    assert lib.gai4_qmv(A, A, A, A, A, 7, 4, 64, 16, 64, None) == g4.GAI4_ERR_UNSUPPORTED
    # non-positive sizes
    assert lib.gai4_qmv(A, A, A, A, A, 2, 4, 64, 0, 64, None) == g4.GAI4_ERR_INVALID_ARG
    # misaligned weights / activations
    assert lib.gai4_qmv(_fake(0x10004), A, A, A, A, 2, 4, 64, 16, 64, None) == g4.GAI4_ERR_MISALIGNED
    assert lib.gai4_qmv(A, A, A, _fake(0x10002), A, 2, 4, 64, 16, 64, None) == g4.GAI4_ERR_MISALIGNED
    # block formats
    assert lib.gai4_q8_0_gemv(A, A, A, 4, 48, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q4_k_gemv(A, A, A, 4, 300, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q4_k_gemv(_fake(0x10008), A, A, 4, 256, None) == g4.GAI4_ERR_MISALIGNED
    assert lib.gai4_quantize(A, None, A, A, 2, 4, 64, 4, 64, None) == g4.GAI4_ERR_INVALID_ARG
    # qmm_t: forced illegal split, too-small workspace
    assert lib.gai4_qmm_t(A, A, A, A, A, 2, 4, 64, 32, 256, 256, 2, A, 1 << 30, None) == g4.GAI4_ERR_UNSUPPORTED
    assert lib.gai4_qmm_t(A, A, A, A, A, 2, 4, 64, 0, 256, 256, 0, None, 0, None) == g4.GAI4_ERR_INVALID_ARG


def test_split_rules(lib):
    plan = g4.gai4_qmm_t_plan
    import torch
    bf = torch.bfloat16
    # K < 512 is never split
    with pytest.raises(g4.Gai4Error):
        plan(40, 4096, 256, 4, 64, bf, split_k=2, workspace_bytes=1 << 30)
    # a forced split must give ranges that are multiples of 64 and >= 256 long
    with pytest.raises(g4.Gai4Error):
        plan(40, 4096, 640, 4, 64, bf, split_k=4, workspace_bytes=1 << 30)   # 160-long ranges
    with pytest.raises(g4.Gai4Error):
        plan(40, 4096, 5 * 64 * 3, 4, 64, bf, split_k=2, workspace_bytes=1 << 30)  # 480: not a multiple of 128
    # other code widths take the tensor-core path in whole 256-column stages
    assert plan(64, 4096, 4096, 6, 64, bf)[0] == 1
    assert plan(64, 4096, 4096 + 64, 3, 64, bf)[0] == 0
    assert plan(33, 4096, 3072, 8, 64, bf, split_k=3, workspace_bytes=1 << 30) == (1, 3)
    assert plan(33, 4096, 2560, 2, 64, bf, split_k=2, workspace_bytes=1 << 30) == (1, 2)
    with pytest.raises(g4.Gai4Error):
        plan(33, 4096, 2560, 2, 64, bf, split_k=4, workspace_bytes=1 << 30)   # 640-column pieces
    # f32 never takes the tensor-core path and never splits
    assert plan(64, 4096, 4096, 4, 64, torch.float32) == (0, 1)
    # no workspace, automatic: no split
    assert plan(64, 4096, 4096, 4, 64, bf, 0, 0)[1] == 1
    # workspace bytes match the split
    assert g4.gai4_qmm_t_workspace_bytes(8, 100, 4096, 4, 64, torch.float32, 1) == 0


def test_binding_requires_cuda_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        g4.gai4_qmv(torch.zeros(4, 8, dtype=torch.int32), torch.zeros(4, 1), torch.zeros(4, 1), torch.zeros(64),
                    bits=4, group_size=64)


def test_batched_rejects_bad_arguments_without_launching(lib):
    A = _fake()
    f = lib.gai4_qmm_t_batched
    # (w, s, b, w_batched, x, x_batch_stride, x_row_stride, out, dtype, bits, gs, batch, M, N, K, split_k, ws, bytes, stream)
    assert f(A, A, A, 1, A, 256 * 8, 256, A, 2, 4, 64, 0, 8, 128, 256, 0, None, 0, None) == g4.GAI4_ERR_INVALID_ARG
    assert f(A, A, A, 1, None, 256 * 8, 256, A, 2, 4, 64, 2, 8, 128, 256, 0, None, 0, None) == g4.GAI4_ERR_INVALID_ARG
    # a row stride shorter than a row
    assert f(A, A, A, 1, A, 256 * 8, 255, A, 2, 4, 64, 2, 8, 128, 256, 0, None, 0, None) == g4.GAI4_ERR_INVALID_ARG
    # activations not aligned to their element size
    assert f(A, A, A, 1, _fake(0x10001), 256 * 8, 256, A, 2, 4, 64, 2, 8, 128, 256, 0, None, 0,
             None) == g4.GAI4_ERR_MISALIGNED
    # strided (or odd-offset) activations need the gather buffer in the workspace
    assert f(A, A, A, 1, A, 264 * 8, 264, A, 2, 4, 64, 2, 8, 128, 256, 0, None, 0, None) == g4.GAI4_ERR_WORKSPACE
    assert f(A, A, A, 1, _fake(0x10002), 256 * 8, 256, A, 2, 4, 64, 2, 8, 128, 256, 0, A, 1024,
             None) == g4.GAI4_ERR_WORKSPACE


def test_batched_workspace_bytes(lib):
    import torch
    # tensor-core path (one launch over the batches): gather buffer (rounded
    # up to 256 bytes) + split-K partials [S, batch * M, N] for S in 1..4
    B, M, N, K = 3, 33, 4096, 14336
    got = g4.gai4_qmm_t_batched_workspace_bytes(B, M, N, K, 4, 64, torch.bfloat16, 0)
    gather = (B * M * K * 2 + 255) // 256 * 256
    parts = got - gather
    assert parts == 0 or (parts % (B * M * N * 4) == 0 and 2 <= parts // (B * M * N * 4) <= 4)
    # a forced split: exactly S slots
    assert g4.gai4_qmm_t_batched_workspace_bytes(B, M, N, K, 4, 64, torch.bfloat16, 2) == gather + 2 * B * M * N * 4
    # CUDA-core path (f32): gather + one call's workspace (none)
    assert g4.gai4_qmm_t_batched_workspace_bytes(B, M, N, K, 4, 64, torch.float32, 0) == (B * M * K * 4 + 255) // 256 * 256
    assert g4.gai4_qmm_t_batched_workspace_bytes(0, 33, 4096, 14336, 4, 64, torch.bfloat16, 0) == 0


def test_int8_activation_entry_points_reject_bad_arguments(lib):
    A = _fake()
    assert lib.gai4_quantize_x_q8(A, A, A, 48, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_quantize_x_q8(None, A, A, 64, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_quantize_x_q8(A, _fake(0x10008), A, 64, None) == g4.GAI4_ERR_MISALIGNED
    assert lib.gai4_q8_0_gemv_i8(A, A, A, A, 4, 40, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q8_0_gemv_i8(A, A, _fake(0x10002), A, 4, 64, None) == g4.GAI4_ERR_MISALIGNED
    assert lib.gai4_q8_0_gemv_i8(A, _fake(0x10004), A, A, 4, 64, None) == g4.GAI4_ERR_MISALIGNED


def test_bounded_wait_check_rejects_bad_arguments(lib):
    A = _fake()
    assert lib.gai4_check_bounded_wait(0, 1000, None, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_check_bounded_wait(0, 0, A, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_check_bounded_wait(0, 4000000001, A, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_check_bounded_wait(1, 1000, _fake(0x10002), None) == g4.GAI4_ERR_MISALIGNED


def test_gguf_block_gemvs_reject_bad_arguments(lib):
    A = _fake()
    assert lib.gai4_q8_0_34b_gemv(None, A, A, 4, 64, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q8_0_34b_gemv(A, A, A, 4, 48, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q8_0_34b_gemv(A, A, A, 0, 64, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q8_0_34b_gemv(_fake(0x10002), A, A, 4, 64, None) == g4.GAI4_ERR_MISALIGNED
    assert lib.gai4_q6_k_gemv(A, A, None, 4, 256, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q6_k_gemv(A, A, A, 4, 300, None) == g4.GAI4_ERR_INVALID_ARG
    assert lib.gai4_q6_k_gemv(A, _fake(0x10004), A, 4, 256, None) == g4.GAI4_ERR_MISALIGNED


def test_planner_properties_sweep(lib):
    """The split planner over a grid of shapes (host logic through the C ABI):
    automatic splits stay within 1..4, never split K < 512, fit the workspace
    they are given and report matching workspace bytes; a forced split S is
    accepted exactly when K cuts into S equal ranges that are multiples of
    max(64, group_size) and at least 256 long; the tensor-core path is taken
    exactly for 16-bit activations, 4-bit codes and M >= 3."""
    import torch
    bf = torch.bfloat16
    for M in (1, 2, 3, 16, 85, 300, 2048):
        for N in (131, 4096, 14336):
            for K in (256, 512, 1088, 4096, 17408):
                for gs in (32, 64, 128):
                    if K % gs:
                        continue
                    path, S = g4.gai4_qmm_t_plan(M, N, K, 4, gs, bf, 0, 1 << 40)
                    assert path == (1 if M >= 3 else 0)
                    assert 1 <= S <= 4 and (S == 1 or (K >= 512 and path == 1))
                    want_ws = S * M * N * 4 if S > 1 else 0
                    assert g4.gai4_qmm_t_workspace_bytes(M, N, K, 4, gs, bf, 0) == want_ws
                    # a workspace of one slot less than the automatic plan: fewer pieces
                    if S > 1:
                        _, S2 = g4.gai4_qmm_t_plan(M, N, K, 4, gs, bf, 0, (S - 1) * M * N * 4)
                        assert S2 <= S - 1 or S2 == 1
                    unit = max(64, gs)
                    for F in (1, 2, 3, 4):
                        legal = F == 1 or (K >= 512 and K % (F * unit) == 0 and K // F >= 256)
                        if legal and (F == 1 or path == 1):
                            assert g4.gai4_qmm_t_plan(M, N, K, 4, gs, bf, F, 1 << 40) == (path, F)
                        else:
                            with pytest.raises(g4.Gai4Error):
                                g4.gai4_qmm_t_plan(M, N, K, 4, gs, bf, F, 1 << 40)


def test_plain_c_program_uses_the_library(lib, tmp_path):
    """The boundary is a C ABI: a C99 program includes the header, links
    libgai4.so and calls host-only entry points (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_gai4.c"
    src.write_text(r'''
#include <stdio.h>
#include "gai4.h"
int main(void) {
    int path = -1, splits = -1;
    gai4_status st = gai4_qmm_t_plan(33, 4096, 14336, 4, 64, GAI4_BF16, 2, (size_t)1 << 30, &path, &splits);
    gai4_status bad = gai4_qmv(NULL, NULL, NULL, NULL, NULL, GAI4_BF16, 4, 64, 16, 64, NULL);
    printf("%d %d %d %d %d %s\n", gai4_version(), (int)st, path, splits, (int)bad, gai4_status_string(bad));
    return 0;
}
''')
    exe = tmp_path / "use_gai4"
    libdir = os.path.dirname(g4.LIB_PATH)
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe), "-L", libdir, "-lgai4", "-Wl,-rpath," + libdir])
    out = subprocess.check_output([str(exe)], text=True).split()
    assert out[:5] == [str(g4.gai4_version()), "0", "1", "2", str(g4.GAI4_ERR_INVALID_ARG)]


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without libgai4.so every call raises instead of computing
    anything on the host."""
    import torch
    monkeypatch.setattr(g4, "_lib", None)
    monkeypatch.setattr(g4, "LIB_PATH", str(tmp_path / "absent" / "libgai4.so"))
    with pytest.raises(RuntimeError):
        g4.lib()
    with pytest.raises(RuntimeError):
        g4.gai4_qmm_t_plan(8, 128, 256, 4, 64, torch.bfloat16)
