"""The C-ABI library loads and exports every symbol include/qgemv.h declares;
host-only calls (sizes, status strings, argument validation that rejects
before any CUDA call) behave as documented.  No GPU needed."""
import ctypes
import os
import re

import pytest

from block_quantized_gemv_quantize_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("quantize_q8_1", "qgemv_q4_0", "qgemv_q6_k", "lmhead_q6_k_top1", "qpack_q4_0", "qpack_q6_k",
                     "argmax_f32_rows", "q8_1_bytes", "q4_0_pack_bytes", "q6_k_pack_bytes",
                     "lmhead_q6_k_top1_workspace_bytes", "qgemv_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_the_header():
    from block_quantized_gemv_quantize_gb300 import _lib

    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_sizes(lib):
    lib.q8_1_bytes.restype = ctypes.c_size_t
    lib.q4_0_pack_bytes.restype = ctypes.c_size_t
    lib.q6_k_pack_bytes.restype = ctypes.c_size_t
    assert lib.q8_1_bytes(6, 5120) == 6 * 160 * 36 == 34560
    assert lib.q8_1_bytes(6, 17408) == 117504
    assert lib.q8_1_bytes(5, 5120) == 28800
    assert lib.q4_0_pack_bytes(17408, 5120) == 50135040
    assert lib.q4_0_pack_bytes(1, 96) == 3 * 16 + 16  # a 3-block tile pads its 6 scale bytes to 16
    assert lib.q6_k_pack_bytes(1, 256) == 8 * 26 + 16  # one row's 2 scale bytes pad to 16
    assert lib.q4_0_pack_bytes(5120, 17408) == 50135040
    assert lib.q4_0_pack_bytes(248320, 5120) == 715161600
    assert lib.q6_k_pack_bytes(248320, 5120) == 1042944000
    assert lib.q6_k_pack_bytes(5120, 5120) == 21504000
    lib.q8_0_pack_bytes.restype = ctypes.c_size_t
    assert lib.q8_0_pack_bytes(17408, 5120) == 17408 * 160 * 34  # the canonical size when N % 16 == 0
    assert lib.q8_0_pack_bytes(17, 256) == 2 * 1 * 4352  # two tiles, rows padded to 32
    assert lib.q8_0_pack_bytes(16, 96) == 0  # K % 256
    lib.q4_k_pack_bytes.restype = ctypes.c_size_t
    assert lib.q4_k_pack_bytes(16, 5120) == 20 * 2368  # 148 B per row and superblock
    assert lib.q4_k_pack_bytes(17, 256) == 2 * 2368  # rows padded to 32
    assert lib.q4_k_pack_bytes(16, 384) == 0  # K % 256
    lib.q5_k_pack_bytes.restype = ctypes.c_size_t
    assert lib.q5_k_pack_bytes(16, 5120) == 20 * 2880  # 180 B per row and superblock
    assert lib.q5_k_pack_bytes(16, 384) == 0  # K % 256
    # top-k: the top-1 workspace rounded to 256 bytes, then k 8-byte keys per
    # row for each CTA, at most min(ceil(N / 4), 256) CTAs
    lib.lmhead_q6_k_topk_workspace_bytes.restype = ctypes.c_size_t
    lib.lmhead_q6_k_topk_workspace_bytes.argtypes = [ctypes.c_int] * 4
    assert lib.lmhead_q6_k_topk_workspace_bytes(5, 5120, 248320, 8) == 29184 + 256 * 5 * 8 * 8
    assert lib.lmhead_q6_k_topk_workspace_bytes(1, 256, 7, 7) == 768 + 2 * 1 * 7 * 8


def test_status_strings(lib):
    lib.qgemv_status_string.restype = ctypes.c_char_p
    for s in (0, -1, -2, -3, -4, -5):
        assert lib.qgemv_status_string(s).decode() != "unknown status"
    assert lib.qgemv_status_string(7).decode() == "unknown status"


def test_validation_rejects_before_any_cuda_call(lib):
    P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.qgemv_q4_0.argtypes = [P, P, P, L, I, I, I, P]
    lib.quantize_q8_1.argtypes = [P, L, P, I, I, P]
    lib.lmhead_q6_k_top1.argtypes = [P, P, L, P, P, ctypes.c_size_t, I, I, I, P]
    fake = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
    odd = 0x10008
    assert lib.qgemv_q4_0(None, fake, fake, 10, 6, 64, 10, None) == -1
    assert lib.qgemv_q4_0(fake, fake, fake, 10, 0, 64, 10, None) == -1
    assert lib.qgemv_q4_0(fake, fake, fake, 10, 18, 64, 10, None) == -2
    assert lib.qgemv_q4_0(fake, fake, fake, 10, 6, 48, 10, None) == -2
    assert lib.qgemv_q4_0(fake, fake, fake, 9, 6, 64, 10, None) == -1
    assert lib.qgemv_q4_0(fake, fake, fake, 10, 6, 64, 0, None) == -1
    assert lib.qgemv_q4_0(odd, fake, fake, 10, 6, 64, 10, None) == -3
    assert lib.quantize_q8_1(fake, 31, fake, 1, 32, None) == -1
    assert lib.quantize_q8_1(fake, 32, odd, 1, 32, None) == -3
    assert lib.lmhead_q6_k_top1(fake, fake, 512, fake, fake, 8, 5, 512, 100, None) == -4
    assert lib.lmhead_q6_k_top1(fake, fake, 512, fake, fake, 4096, 5, 320, 100, None) == -2
    topk = lib.lmhead_q6_k_topk
    topk.argtypes = [P, P, L, I, P, P, P, P, P, ctypes.c_size_t, I, I, I, P]
    big = 1 << 20
    assert topk(fake, fake, 512, 0, None, fake, fake, None, fake, big, 5, 512, 100, None) == -1  # k = 0
    assert topk(fake, fake, 512, 9, None, fake, fake, None, fake, big, 5, 512, 100, None) == -1  # k > 8
    assert topk(fake, fake, 512, 8, None, fake, fake, None, fake, big, 5, 512, 7, None) == -1  # k > N
    assert topk(fake, fake, 512, 8, fake, fake, fake, None, fake, big, 5, 512, 100, None) == -1  # cand alone
    assert topk(fake, fake, 512, 8, None, fake, fake, None, fake, 4096, 5, 512, 100, None) == -4
    assert topk(fake, fake, 512, 8, None, fake, odd, None, fake, big, 5, 512, 100, None) == -3
    assert topk(fake, fake, 512, 8, None, fake, None, None, fake, big, 18, 512, 100, None) == -2


def test_fused_failure_hook_refuses_before_any_cuda_call(lib):
    # the test-only hook makes the next validated fused LM-head call return
    # QGEMV_CUDA_ERROR before anything is enqueued: on a machine without a
    # GPU the call returns at once, touching none of the (fake) buffers
    lib.qgemv_debug_fail_fused.argtypes = [ctypes.c_int]
    fn = lib.lmhead_q6_k_top1
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fake = 0x10000  # 16-byte aligned, never dereferenced
    assert lib.qgemv_debug_fail_fused(1) == 0
    assert fn(fake, fake, 5120, fake, fake, 1 << 20, 5, 5120, 248320, None) == -5
    assert lib.qgemv_debug_fail_fused(0) == 0  # the one request was taken
    # validation still comes first: a bad argument is reported as such
    assert lib.qgemv_debug_fail_fused(1) == 0
    assert fn(None, fake, 5120, fake, fake, 1 << 20, 5, 5120, 248320, None) == -1
    assert lib.qgemv_debug_fail_fused(0) == 1


def test_fused_failure_hook_from_the_environment():
    # QGEMV_FAIL_FUSED=2 in a fresh process: its first two validated fused
    # calls are refused before any CUDA call, the third is not refused by the
    # hook (without a GPU it then fails later, with another status)
    code = (
        "import ctypes, sys\n"
        "lib = ctypes.CDLL(sys.argv[1])\n"
        "fn = lib.lmhead_q6_k_top1\n"
        "fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,\n"
        "               ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]\n"
        "fake = 0x10000\n"
        "print(fn(fake, fake, 5120, fake, fake, 1 << 20, 5, 5120, 248320, None),\n"
        "      fn(fake, fake, 5120, fake, fake, 1 << 20, 5, 5120, 248320, None),\n"
        "      lib.qgemv_debug_fail_fused(0))\n"
    )
    import subprocess
    import sys

    from block_quantized_gemv_quantize_gb300 import build

    env = dict(os.environ, QGEMV_FAIL_FUSED="2")
    out = subprocess.run([sys.executable, "-c", code, build.LIB], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["-5", "-5", "0"]
