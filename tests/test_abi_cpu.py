"""CPU checks of the boundary: the library builds and loads, exports every
symbol include/mc_max.h declares, and rejects bad arguments on the host
before touching the GPU.  No compute call is made here."""
import ctypes

import pytest

from muonclip_mc_max_gb300 import api, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def test_header_symbols_exported(lib):
    names = api.header_symbols()
    assert len(names) >= 14
    for n in ["mc_max_logits_mha", "mc_max_logits_mla", "mc_qk_clip_mha", "mc_qk_clip_mla",
              "mc_newton_schulz", "mc_muon_step"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n
        assert hasattr(api, n), f"python binding lacks {n}"


def test_status_strings(lib):
    assert api.mc_status_string(0) == "ok"
    assert "workspace" in api.mc_status_string(4)
    assert api.mc_status_string(99) == "unknown status"


def test_invalid_arguments_rejected_on_host(lib):
    nil = None
    ws = ctypes.c_void_p(256)
    # null inputs
    assert lib.mc_max_logits_mha(nil, nil, nil, 1, 2, 8, 64, 1, 64, 0, 0, nil, nil, ws, 1 << 30,
                                 nil) == 1
    fake = ctypes.c_void_p(4096)
    # non-positive sizes
    assert lib.mc_max_logits_mha(fake, fake, fake, 1, 0, 8, 64, 1, 64, 0, 0, fake, nil, ws,
                                 1 << 30, nil) == 1
    # workspace too small / misaligned
    assert lib.mc_max_logits_mha(fake, fake, fake, 1, 2, 8, 64, 1, 64, 0, 0, fake, nil, ws, 16,
                                 nil) == 4
    assert lib.mc_max_logits_mha(fake, fake, fake, 1, 2, 8, 64, 1, 64, 0, 0, fake, nil,
                                 ctypes.c_void_p(4097), 1 << 30, nil) == 4
    # bad dtype
    assert lib.mc_max_logits_mha(fake, fake, fake, 7, 2, 8, 64, 1, 64, 0, 0, fake, nil, ws,
                                 1 << 30, nil) == 1
    # S_max outputs not 4-byte aligned (the kernels merge into them with 32-bit atomics)
    assert lib.mc_max_logits_mha(fake, fake, fake, 1, 2, 8, 64, 1, 64, 0, 0, ctypes.c_void_p(4098), nil,
                                 ws, 1 << 30, nil) == 1
    assert lib.mc_max_logits_mha(fake, fake, fake, 1, 2, 8, 64, 1, 64, 0, 0, fake, ctypes.c_void_p(4098),
                                 ws, 1 << 30, nil) == 1
    # Muon: a zero-size matrix, a pointer that is not float-aligned, an empty batch
    rows = (ctypes.c_int * 1)(8)
    cols = (ctypes.c_int * 1)(0)
    ptrs = (ctypes.c_void_p * 1)(4096)
    assert lib.mc_muon_step(ptrs, ptrs, ptrs, rows, cols, 1, 1e-3, 0.95, 0.1, 0.2, 5, 3.4, -4.7,
                            2.0, 1e-7, 0, ws, 1 << 30, nil) == 1
    cols = (ctypes.c_int * 1)(6)
    odd = (ctypes.c_void_p * 1)(4098)
    assert lib.mc_muon_step(odd, odd, odd, rows, cols, 1, 1e-3, 0.95, 0.1, 0.2, 5, 3.4, -4.7,
                            2.0, 1e-7, 0, ws, 1 << 30, nil) == 1
    assert lib.mc_newton_schulz(ptrs, ptrs, rows, cols, 0, 5, 3.4, -4.7, 2.0, 1e-7, ws, 1 << 30,
                                nil) == 1
    # MLA: unsupported rope width for the scan
    L = api.MlaLayer(D=64, q_lora=64, kv_lora=64, H=1, nope=64, rope=32, rope_base=1e4, wtype=1,
                     w_qa=4096, w_qb=4096, w_kva=4096, w_kb=4096)
    s = lib.mc_max_logits_mla(ctypes.byref(L), fake, 1, 8, 1, 0, fake, nil, ws, 1 << 30, nil)
    assert s == 2
    # GEMM: K not a multiple of 8
    assert lib.mc_gemm_bf16(fake, fake, fake, 0, 8, 8, 12, 1, 1, nil) == 2
    # attention: null input, unsupported head width, misaligned pointer, output
    # aliasing an input (it takes no workspace)
    q, k, v, o = (ctypes.c_void_p(4096 * (i + 1)) for i in range(4))
    big = 1 << 20
    assert lib.mc_attention_mha(nil, k, v, 1, 8, 2, 64, 0, 0, o, fake, nil, ws, big, nil) == 1
    assert lib.mc_attention_mha(q, k, v, 1, 8, 2, 96, 0, 0, o, fake, nil, ws, big, nil) == 2
    assert lib.mc_attention_mha(q, k, v, 1, 0, 2, 64, 0, 0, o, fake, nil, ws, big, nil) == 1
    assert lib.mc_attention_mha(ctypes.c_void_p(4104), k, v, 1, 8, 2, 64, 0, 0, o, fake, nil, ws, big,
                                nil) == 1
    assert lib.mc_attention_mha(q, k, v, 1, 8, 2, 64, 0, 0, q, fake, nil, ws, big, nil) == 1
    assert lib.mc_attention_mha(q, k, v, 1, 8, 2, 64, 0, 0, o, ctypes.c_void_p(4098), nil, ws, big, nil) == 1
    # QK-Clip: a bf16 weight at an odd address, an f32 weight or S_max not 4-byte aligned
    assert lib.mc_qk_clip_mha(ctypes.c_void_p(4097), fake, 1, 8, 2, 64, fake, ctypes.c_float(100.0), nil,
                              nil) == 1
    assert lib.mc_qk_clip_mha(ctypes.c_void_p(4098), fake, 0, 8, 2, 64, fake, ctypes.c_float(100.0), nil,
                              nil) == 1
    assert lib.mc_qk_clip_mha(fake, fake, 1, 8, 2, 64, ctypes.c_void_p(4098), ctypes.c_float(100.0), nil,
                              nil) == 1
    assert lib.mc_qk_clip_global(ctypes.c_void_p(4097), fake, 1, 8, 8, fake, 2, ctypes.c_float(100.0),
                                 ctypes.c_float(0.5), nil, nil) == 1
    # bounded-wait self-test: limit out of range, null or misaligned result
    assert lib.mc_selftest_wait_timeout(0, fake, nil) == 1
    assert lib.mc_selftest_wait_timeout(1000001, fake, nil) == 1
    assert lib.mc_selftest_wait_timeout(1000, nil, nil) == 1
    assert lib.mc_selftest_wait_timeout(1000, ctypes.c_void_p(4100), nil) == 1


def test_workspace_sizes(lib):
    a = api.mc_max_logits_mha_workspace_size(8, 1024, 1024, 16, 64, api.MC_BF16)
    # Q and K in fp16 (the scan merges S_max straight into the outputs)
    assert a >= 2 * 8 * 1024 * 1024 * 2
    assert api.mc_max_logits_mha_workspace_size(8, 1024, 1024, 16, 64, api.MC_F32) > a
    shapes = [(7168, 2048), (2048, 7168)]
    b = api.mc_muon_workspace_size(shapes)
    # per matrix: X ping-pong (2048x7168) + A, B (2048^2), bf16
    assert b >= 2 * (2 * 2048 * 7168 * 2 + 2 * 2048 * 2048 * 2)
    assert api.mc_muon_workspace_size(shapes) == b
    L = api.MlaLayer(D=7168, q_lora=1536, kv_lora=512, H=64, nope=128, rope=64, rope_base=5e4,
                     wtype=1)
    # attention: no workspace (S_max is merged straight into the outputs)
    assert api.mc_attention_mha_workspace_size(8, 16) == 0
    assert api.mc_attention_mha_workspace_size(0, 16) == 0
    c = api.mc_max_logits_mla_workspace_size(L, 16, 4096)
    # c_Q, [c_KV|k^R], [q^C|q^R] and k^C of a K2-shaped layer at B=16, T=4096
    assert c >= 65536 * (1536 + 576 + 64 * 192 + 64 * 128) * 2


def test_workspace_sizes_saturate_instead_of_wrapping(lib):
    """Sizes whose scratch does not fit size_t report SIZE_MAX, so no
    workspace (nor the allocation-free scratch) can pass the size check;
    the largest int sizes give B*T*H*dh near 2^62 elements."""
    big = 2 ** 31 - 1
    size_max = 2 ** 64 - 1
    for dt in (api.MC_BF16, api.MC_F32):
        assert api.mc_max_logits_mha_workspace_size(65535, 32767, 64, 32767, 65535, dt) == size_max
    assert api.mc_max_logits_mha_workspace_size(1, big, 64, 1, 64, api.MC_BF16) < size_max
    L = api.MlaLayer(D=7168, q_lora=big, kv_lora=big, H=big, nope=128, rope=64, rope_base=5e4,
                     wtype=1)
    assert api.mc_max_logits_mla_workspace_size(L, big, big) == size_max
