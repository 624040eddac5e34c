"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument validation returns the documented status codes (no GPU needed: no
call here reaches a CUDA launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4k.h")


@pytest.fixture(scope="module")
def lib():
    from q4_weight_matmul_gb300.build import build
    path = build()
    handle = ctypes.CDLL(path)
    import q4_weight_matmul_gb300 as q4k
    for name, (res, args) in q4k.SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype, fn.argtypes = res, args
    return handle


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return sorted(set(re.findall(r"\b((?:q4k|q6k|q8|x_split)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("q4k_pack", "q8_quantize", "q4k_gemv", "q4k_gemm", "q6k_pack", "q6k_gemv"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    import q4_weight_matmul_gb300 as q4k
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in q4k.SIGNATURES, f"binding lacks {name}"


def test_packed_bytes(lib):
    assert lib.q4k_packed_bytes(9728, 2560, 0) == 9728 * 10 * 144
    assert lib.q4k_packed_bytes(1, 256, 0) == 144
    assert lib.q4k_packed_bytes(0, 256, 0) == 0
    assert lib.q4k_packed_bytes(4, 100, 0) == 0        # cols not a multiple of 256
    assert lib.q4k_packed_bytes(4, 256, 7) == 0        # unknown layout
    assert lib.q4k_packed_bytes(-1, 256, 0) == 0


def test_gpu_layout_is_declared_and_refused(lib):
    assert lib.q4k_packed_bytes(8, 256, 1) == 0                     # Q4K_LAYOUT_GPU
    fake = ctypes.c_void_p(0x10000)
    assert lib.q4k_pack(fake, fake, fake, fake, fake, 8, 256, 1, fake, None) == 3
    assert lib.q4k_unpack(fake, 1, 8, 256, fake, fake, fake, fake, fake, None) == 3
    assert lib.q4k_gemv(fake, 1, 8, 256, fake, 1, None, fake, None) == 3
    assert lib.q4k_gemm(fake, 1, 8, 256, fake, fake, fake, 16, fake, None) == 3


def test_q6k_packed_bytes(lib):
    # GGUF: 210 bytes a superblock; GPU layout: a row's 210*nb bytes padded to 16
    assert lib.q6k_packed_bytes(151936, 2560, 0) == 151936 * 10 * 210
    assert lib.q6k_packed_bytes(151936, 2560, 1) == 151936 * 2112
    assert lib.q6k_packed_bytes(2560, 9728, 1) == 2560 * 7984
    assert lib.q6k_packed_bytes(3, 2048, 1) == 3 * 1680                # 8 * 210, already a multiple of 16
    assert lib.q6k_packed_bytes(0, 256, 1) == 0
    assert lib.q6k_packed_bytes(4, 100, 1) == 0
    assert lib.q6k_packed_bytes(4, 256, 2) == 0


def test_q6k_validation_before_any_launch(lib):
    fake, odd16, odd2 = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10002), ctypes.c_void_p(0x10001)
    # the GEMV reads the GPU layout only
    assert lib.q6k_gemv(fake, 0, 8, 256, fake, 1, None, fake, None) == 3
    assert lib.q6k_gemv(fake, 1, 8, 256, fake, 9, None, fake, None) == 3
    assert lib.q6k_gemv(fake, 1, 8, 256, fake, -1, None, fake, None) == 1
    assert lib.q6k_gemv(fake, 1, 8, 300, fake, 1, None, fake, None) == 1
    assert lib.q6k_gemv(None, 1, 8, 256, fake, 1, None, fake, None) == 1
    assert lib.q6k_gemv(odd16, 1, 8, 256, fake, 1, None, fake, None) == 2
    assert lib.q6k_gemv(None, 1, 0, 256, None, 1, None, None, None) == 0
    assert lib.q6k_pack(fake, fake, fake, 2, 256, 5, fake, None) == 3
    assert lib.q6k_pack(fake, fake, None, 2, 256, 1, fake, None) == 1
    assert lib.q6k_pack(fake, fake, fake, 2, 256, 1, odd16, None) == 2
    # a GGUF buffer needs 2-byte alignment only; the GPU layout 16
    big = ctypes.c_void_p(0x100000)
    assert lib.q6k_repack(odd2, 0, 2, 256, big, 1, None) == 2
    assert lib.q6k_repack(fake, 0, 2, 256, odd16, 1, None) == 2
    # overlapping source and destination
    assert lib.q6k_repack(fake, 0, 2, 256, fake, 1, None) == 1
    assert lib.q6k_unpack(fake, 3, 2, 256, fake, fake, fake, None) == 3
    assert lib.q6k_unpack(fake, 1, 2, 256, fake, fake, odd16, None) == 2
    assert lib.q6k_unpack(None, 1, 0, 256, None, None, None, None) == 0
    # the MMQ products read the GPU layout only; block sums may be NULL
    assert lib.q6k_gemv_q8(fake, 0, 8, 256, fake, fake, None, 1, None, fake, None) == 3
    assert lib.q6k_gemv_q8(fake, 1, 8, 256, fake, fake, None, 9, None, fake, None) == 3
    assert lib.q6k_gemv_q8(fake, 1, 8, 256, None, fake, None, 1, None, fake, None) == 1
    assert lib.q6k_gemv_q8(fake, 1, 8, 256, fake, fake, None, 1, None, odd16, None) == 2
    assert lib.q6k_gemm(fake, 1, 8, 300, fake, fake, None, 4, fake, None) == 1
    assert lib.q6k_gemm(fake, 1, 8, 256, fake, None, None, 4, fake, None) == 1
    assert lib.q6k_gemm(None, 1, 0, 256, None, None, None, 4, None, None) == 0
    assert lib.q6k_gemm_blockdots(fake, 1, 8, 256, fake, 4, None, None) == 1
    assert lib.q6k_gemm_f16(fake, 0, 8, 256, fake, fake, None, fake, 4, fake, None) == 3
    assert lib.q6k_gemm_f16(fake, 1, 8, 256, fake, None, None, fake, 4, fake, None) == 1
    assert lib.q6k_gemm_f16(fake, 1, 8, 256, fake, fake, None, fake, 4, odd16, None) == 2
    assert lib.q6k_gemm_f16(None, 1, 0, 256, None, None, None, None, 4, None, None) == 0


def test_f16_split_bytes_and_validation(lib):
    # hi and lo: 2 bytes each per element; 16 binary16 block sums per superblock; 1/s per token
    assert lib.x_split_f16_bytes(512, 2560) == 512 * (2560 * 4 + 10 * 32 + 4)
    assert lib.x_split_f16_bytes(4, 100) == 0
    fake, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
    assert lib.x_split_f16(fake, 2, 300, fake, fake, fake, fake, None) == 1
    assert lib.x_split_f16(fake, 2, 256, fake, fake, None, fake, None) == 1
    assert lib.x_split_f16(fake, 2, 256, fake, odd, fake, fake, None) == 2
    assert lib.x_split_f16(None, 0, 256, None, None, None, None, None) == 0
    assert lib.q4k_gemm_f16(fake, 1, 8, 256, fake, fake, fake, fake, 4, fake, None) == 3   # GPU layout
    assert lib.q4k_gemm_f16(fake, 0, 8, 256, fake, fake, None, fake, 4, fake, None) == 1
    assert lib.q4k_gemm_f16(fake, 0, 8, 256, fake, fake, fake, fake, 4, odd, None) == 2
    assert lib.q4k_gemm_f16(None, 0, 0, 256, None, None, None, None, 4, None, None) == 0


def test_q8_1_bytes(lib):
    # q: one byte per element; d8 and sum: four bytes each per 32 elements
    assert lib.q8_1_bytes(512, 2560) == 512 * 2560 + 2 * 4 * 512 * 80
    assert lib.q8_1_bytes(1, 256) == 256 + 64
    assert lib.q8_1_bytes(0, 256) == 0
    assert lib.q8_1_bytes(4, 100) == 0
    assert lib.q8_1_bytes(-1, 256) == 0


def test_unpack_validates_before_any_launch(lib):
    fake, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10004)
    assert lib.q4k_unpack(fake, 0, 8, 300, fake, fake, fake, fake, fake, None) == 1
    assert lib.q4k_unpack(fake, 0, -1, 256, fake, fake, fake, fake, fake, None) == 1
    assert lib.q4k_unpack(None, 0, 8, 256, fake, fake, fake, fake, fake, None) == 1
    assert lib.q4k_unpack(fake, 0, 8, 256, fake, fake, fake, fake, None, None) == 1
    assert lib.q4k_unpack(odd, 0, 8, 256, fake, fake, fake, fake, fake, None) == 2
    assert lib.q4k_unpack(fake, 0, 0, 256, None, None, None, None, None, None) == 0


def test_gemv_seq_plan_validates_like_the_one_shot_call(lib):
    import q4_weight_matmul_gb300 as q4k
    fake, odd = 0x10000, 0x10004

    def jobs(*specs):
        arr = (q4k.GemvJob * len(specs))()
        for i, (rows, cols, x) in enumerate(specs):
            arr[i].w, arr[i].rows, arr[i].cols, arr[i].x, arr[i].y = fake, rows, cols, x, fake
        return arr

    n1 = lib.q4k_gemv_seq_plan_bytes(1)
    # room for one launch per 48 jobs: a list may hold up to 48 Q6_K jobs a launch
    assert n1 > 0 and lib.q4k_gemv_seq_plan_bytes(48) == n1
    assert lib.q4k_gemv_seq_plan_bytes(49) > n1
    assert lib.q4k_gemv_seq_plan_bytes(256) > lib.q4k_gemv_seq_plan_bytes(97)
    assert lib.q4k_gemv_seq_plan_bytes(257) == 0 and lib.q4k_gemv_seq_plan_bytes(-1) == 0
    raw = ctypes.create_string_buffer(n1 + 128)
    base = ctypes.addressof(raw)
    plan = base + (-base) % 64
    ws = ctypes.c_void_p(fake)
    ok1 = jobs((8, 256, fake))
    assert lib.q4k_gemv_seq_plan(None, 1, 0, 1, ws, 1 << 20, plan, n1) == 1          # null list
    assert lib.q4k_gemv_seq_plan(ok1, 1, 5, 1, ws, 1 << 20, plan, n1) == 3            # unknown layout
    assert lib.q4k_gemv_seq_plan(ok1, 1, 0, 9, ws, 1 << 20, plan, n1) == 3            # batch above 8
    assert lib.q4k_gemv_seq_plan(jobs((8, 300, fake)), 1, 0, 1, ws, 1 << 20, plan, n1) == 1
    assert lib.q4k_gemv_seq_plan(jobs((8, 256, odd)), 1, 0, 1, ws, 1 << 20, plan, n1) == 2
    assert lib.q4k_gemv_seq_plan(ok1, 1, 0, 1, None, 1 << 20, plan, n1) == 1          # no workspace
    assert lib.q4k_gemv_seq_plan(ok1, 1, 0, 1, ws, 1 << 20, None, n1) == 1            # no plan
    assert lib.q4k_gemv_seq_launch(None, None) == 1
    # the host-buffer step checks its pointers and the plan before any copy
    zeroed = ctypes.create_string_buffer(n1 + 128)
    zplan = ctypes.addressof(zeroed) + (-ctypes.addressof(zeroed)) % 64
    assert lib.q4k_gemv_seq_launch_host(None, fake, fake, 16, fake, fake, 16, None) == 1
    assert lib.q4k_gemv_seq_launch_host(zplan, None, fake, 16, fake, fake, 16, None) == 1
    assert lib.q4k_gemv_seq_launch_host(zplan, fake, None, 16, fake, fake, 16, None) == 1
    assert lib.q4k_gemv_seq_launch_host(zplan, fake, fake, 16, None, fake, 16, None) == 1
    assert lib.q4k_gemv_seq_launch_host(zplan, fake, fake, 16, fake, None, 16, None) == 1
    assert lib.q4k_gemv_seq_launch_host(zplan, None, None, 0, None, None, 0, None) == 1   # not a plan


def test_status_strings_and_version(lib):
    assert lib.q4k_status_string(0) == b"Q4K_OK"
    assert lib.q4k_status_string(5) == b"Q4K_ERR_DEVICE_TIMEOUT"
    assert lib.q4k_status_string(99) == b"Q4K_ERR_UNKNOWN"
    assert b"sm_103a" in lib.q4k_version()


def test_validation_before_any_launch(lib):
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x10008)
    # cols must be a positive multiple of 256
    assert lib.q4k_gemv(fake, 0, 8, 300, fake, 1, None, fake, None) == 1
    assert lib.q4k_gemm(fake, 0, 8, 0, fake, fake, fake, 4, fake, None) == 1
    assert lib.q8_quantize(fake, 2, 100, fake, fake, fake, None) == 1
    # unknown layout
    assert lib.q4k_gemv(fake, 9, 8, 256, fake, 1, None, fake, None) == 3
    # batch out of range
    assert lib.q4k_gemv(fake, 0, 8, 256, fake, 9, None, fake, None) == 3
    assert lib.q4k_gemv(fake, 0, 8, 256, fake, -1, None, fake, None) == 1
    # null pointers
    assert lib.q4k_gemv(None, 0, 8, 256, fake, 1, None, fake, None) == 1
    assert lib.q4k_gemm(fake, 0, 8, 256, fake, None, fake, 4, fake, None) == 1
    assert lib.q4k_pack(fake, fake, fake, None, fake, 2, 256, 0, fake, None) == 1
    # misaligned pointers
    assert lib.q4k_pack(fake, fake, fake, fake, odd, 2, 256, 0, fake, None) == 2
    assert lib.q8_quantize(odd, 2, 256, fake, fake, fake, None) == 2
    assert lib.q4k_gemm(fake, 0, 8, 256, fake, fake, fake, 4, odd, None) == 2
    # empty problems enqueue nothing and succeed
    assert lib.q4k_gemv(None, 0, 0, 256, None, 1, None, None, None) == 0
    assert lib.q4k_gemm(None, 0, 8, 256, None, None, None, 0, None, None) == 0
    assert lib.q8_quantize(None, 0, 256, None, None, None, None) == 0
    assert lib.q4k_pack(None, None, None, None, None, 0, 256, 0, None, None) == 0


def test_gemv_seq_validation_before_any_launch(lib):
    import q4_weight_matmul_gb300 as q4k
    fake, odd = 0x10000, 0x10008

    def jobs(*specs):
        arr = (q4k.GemvJob * max(1, len(specs)))()
        for i, (rows, cols, x) in enumerate(specs):
            arr[i].w, arr[i].rows, arr[i].cols, arr[i].x, arr[i].y = fake, rows, cols, x, fake
        return arr

    ws = ctypes.c_void_p(fake)
    ok2 = jobs((8, 256, fake), (16, 512, fake))
    assert lib.q4k_gemv_seq(None, 1, 0, 1, ws, 1 << 20, None) == 1          # null list
    assert lib.q4k_gemv_seq(ok2, -1, 0, 1, ws, 1 << 20, None) == 1
    assert lib.q4k_gemv_seq(jobs(*[(8, 256, fake)] * 257), 257, 0, 1, ws, 1 << 20, None) == 3
    assert lib.q4k_gemv_seq(ok2, 2, 5, 1, ws, 1 << 20, None) == 3            # unknown layout
    bad_fmt = jobs((8, 256, fake))
    bad_fmt[0].format = 2                                                     # neither Q4_K nor Q6_K
    assert lib.q4k_gemv_seq(bad_fmt, 1, 0, 1, ws, 1 << 20, None) == 1
    assert lib.q4k_gemv_seq(ok2, 2, 0, 9, ws, 1 << 20, None) == 3            # batch above 8
    assert lib.q4k_gemv_seq(ok2, 2, 0, -1, ws, 1 << 20, None) == 1
    assert lib.q4k_gemv_seq(jobs((8, 300, fake)), 1, 0, 1, ws, 1 << 20, None) == 1
    assert lib.q4k_gemv_seq(jobs((8, 256, odd)), 1, 0, 1, ws, 1 << 20, None) == 2
    assert lib.q4k_gemv_seq(ok2, 2, 0, 1, None, 1 << 20, None) == 1          # no workspace
    assert lib.q4k_gemv_seq(ok2, 2, 0, 1, ctypes.c_void_p(odd), 1 << 20, None) == 2
    # nothing to do: zero rows everywhere, or batch 0
    assert lib.q4k_gemv_seq(jobs((0, 256, None)), 1, 0, 1, None, 0, None) == 0
    assert lib.q4k_gemv_seq(ok2, 2, 0, 0, None, 0, None) == 0
    assert lib.q4k_gemv_seq(None, 0, 0, 1, None, 0, None) == 0
    assert lib.q4k_gemv_seq_workspace_bytes(jobs((8, 300, fake)), 1, 1) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    import q4_weight_matmul_gb300 as q4k
    x = torch.zeros(1, 256)
    with pytest.raises(TypeError):
        q4k.q8_quantize(x)


def test_rate_probe_library_loads_and_exports_its_probes(lib):
    from q4_weight_matmul_gb300.build import PEAKS_LIB
    probe = ctypes.CDLL(PEAKS_LIB)
    for name in ("q4kp_mma_s8_tops", "q4kp_tc_f16_tflops"):
        assert hasattr(probe, name), name
