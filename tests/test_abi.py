"""The C-ABI library: it builds, loads, exports every entry point that
include/moeq4.h declares, and its host-side argument checks return the
documented status codes.  No CUDA computation runs here (no GPU needed): every
call below is rejected, or answered, before the library touches a device."""
import ctypes
import os
import re

import pytest

import bit_quantized_moe_q4_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moeq4.h")


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for required in ("moe_q4_pack", "moe_route_topk", "moe_q4_forward_prefill",
                     "moe_w4a8_forward_decode"):
        assert required in names
    assert set(names) == set(moe.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_packed_bytes(lib):
    assert moe.moe_q4_packed_bytes(128, 1536, 2048) == 128 * 1536 * 2048 * 18 // 32
    assert moe.moe_q4_packed_bytes(1, 128, 64) == 4608
    assert moe.moe_q4_packed_bytes(1, 100, 64) == 0
    assert moe.moe_q4_packed_bytes(1, 128, 32) == 0
    assert moe.moe_q4_packed_bytes(0, 128, 64) == 0


def test_workspace_bytes_grow_with_tokens(lib):
    a = moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL, 2048, 2048, 768, 128, 8)
    b = moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL, 4096, 2048, 768, 128, 8)
    assert 0 < a < b
    # y (bf16 [T*k, H]) and h (bf16 [T*k, I]) dominate
    assert a >= 2048 * 8 * (2048 + 768) * 2
    assert moe.moe_workspace_bytes(7, 1, 256, 128, 8, 2) == 0
    assert moe.moe_workspace_bytes(moe.MOE_MODE_DECODE, 1, 2048, 768, 128, 8) > 0


FAKE = 1 << 20  # a 16-byte-aligned address that is never dereferenced on the host


def _prefill(lib, T=4, H=256, I=128, E=8, k=2, flags=1, x=FAKE, wr=FAKE, wgu=FAKE, wd=FAKE,
             out=FAKE * 2, ws=FAKE * 3, ws_bytes=1 << 40, fn="moe_q4_forward_prefill"):
    return getattr(lib, fn)(x, wr, wgu, wd, T, H, I, E, k, flags, out, ws, ws_bytes, None, None)


@pytest.mark.parametrize("fn", ["moe_q4_forward_prefill", "moe_w4a8_forward_decode",
                                "moe_w8a8_forward_decode"])
def test_forward_argument_checks(lib, fn):
    assert _prefill(lib, fn=fn, H=200) == moe.MOE_ERR_SHAPE          # H % 128
    assert _prefill(lib, fn=fn, I=96) == moe.MOE_ERR_SHAPE           # I % 128
    assert _prefill(lib, fn=fn, E=300) == moe.MOE_ERR_SHAPE          # E > 256
    assert _prefill(lib, fn=fn, k=9, E=8) == moe.MOE_ERR_SHAPE       # k > E
    assert _prefill(lib, fn=fn, k=17, E=64) == moe.MOE_ERR_SHAPE     # k > 16
    assert _prefill(lib, fn=fn, k=0) == moe.MOE_ERR_SHAPE
    assert _prefill(lib, fn=fn, T=-1) == moe.MOE_ERR_SHAPE
    assert _prefill(lib, fn=fn, flags=4) == moe.MOE_ERR_INVALID_ARG
    assert _prefill(lib, fn=fn, x=None) == moe.MOE_ERR_INVALID_ARG
    assert _prefill(lib, fn=fn, wd=None) == moe.MOE_ERR_INVALID_ARG
    assert _prefill(lib, fn=fn, x=FAKE + 8) == moe.MOE_ERR_ALIGN
    assert _prefill(lib, fn=fn, out=FAKE) == moe.MOE_ERR_INVALID_ARG   # out aliases x
    assert _prefill(lib, fn=fn, ws_bytes=16) == moe.MOE_ERR_WORKSPACE
    assert _prefill(lib, fn=fn, ws=None) == moe.MOE_ERR_WORKSPACE
    assert _prefill(lib, fn=fn, T=0) == moe.MOE_OK                     # empty input: no-op
    assert b"workspace" in lib.moe_last_error_string() or True
    if fn == "moe_w4a8_forward_decode":
        assert _prefill(lib, fn=fn, T=33) == moe.MOE_ERR_SHAPE       # decode takes <= 32 tokens
    if fn == "moe_w8a8_forward_decode":
        assert _prefill(lib, fn=fn, T=moe.MOE_W8_DECODE_MAX_T + 1) == moe.MOE_ERR_SHAPE
        assert b"8-bit" in lib.moe_last_error_string()
        # the full decode shape fits the on-chip staging at 16 tokens
        assert _prefill(lib, fn=fn, T=16, H=2048, I=768, E=128, k=8, x=None) == moe.MOE_ERR_INVALID_ARG


def _stack(lib, L=2, T=1, H=256, I=128, E=8, k=2, flags=1, x=FAKE, layer=(FAKE, FAKE, FAKE),
           bad_layer=None, out=FAKE * 2, ws=FAKE * 3, ws_bytes=1 << 40):
    ptrs = [list(layer) for _ in range(max(L, 1))]
    if bad_layer is not None:
        ptrs[bad_layer[0]][bad_layer[1]] = bad_layer[2]
    arrs = [(ctypes.c_void_p * len(ptrs))(*[p[j] for p in ptrs]) for j in range(3)]
    return lib.moe_w4a8_forward_decode_stack(x, L, arrs[0], arrs[1], arrs[2], T, H, I, E, k, flags,
                                             out, ws, ws_bytes, None)


def test_decode_stack_argument_checks(lib):
    assert _stack(lib, L=0) == moe.MOE_ERR_SHAPE
    assert _stack(lib, L=moe.MOE_DECODE_MAX_LAYERS + 1) == moe.MOE_ERR_SHAPE
    assert b"L=" in lib.moe_last_error_string()
    assert _stack(lib, T=33) == moe.MOE_ERR_SHAPE
    assert _stack(lib, H=200) == moe.MOE_ERR_SHAPE
    assert _stack(lib, flags=4) == moe.MOE_ERR_INVALID_ARG
    assert _stack(lib, x=None) == moe.MOE_ERR_INVALID_ARG
    assert _stack(lib, bad_layer=(1, 2, None)) == moe.MOE_ERR_INVALID_ARG   # layer 1's wd
    assert b"layer 1" in lib.moe_last_error_string()
    assert _stack(lib, bad_layer=(0, 1, FAKE + 8)) == moe.MOE_ERR_ALIGN
    assert _stack(lib, out=FAKE) == moe.MOE_ERR_INVALID_ARG                 # out aliases x
    assert _stack(lib, ws_bytes=16) == moe.MOE_ERR_WORKSPACE
    assert _stack(lib, T=0) == moe.MOE_OK                                   # empty input: no-op


def test_error_string_names_the_problem(lib):
    assert _prefill(lib, H=200) == moe.MOE_ERR_SHAPE
    assert b"128" in lib.moe_last_error_string()


def test_pack_argument_checks(lib):
    f = lib.moe_q4_pack
    assert f(9, FAKE, FAKE, 1, 128, 64, FAKE, 4608, None) == moe.MOE_ERR_INVALID_ARG
    assert f(0, FAKE, FAKE, 1, 100, 64, FAKE, 4608, None) == moe.MOE_ERR_SHAPE
    assert f(0, FAKE, FAKE, 1, 128, 96, FAKE, 4608, None) == moe.MOE_ERR_SHAPE
    assert f(0, FAKE, None, 1, 128, 64, FAKE, 4608, None) == moe.MOE_ERR_INVALID_ARG
    assert f(1, FAKE, FAKE, 1, 128, 64, FAKE, 4608, None) == moe.MOE_ERR_INVALID_ARG
    assert f(0, FAKE + 4, FAKE, 1, 128, 64, FAKE, 4608, None) == moe.MOE_ERR_ALIGN
    assert f(0, FAKE, FAKE, 1, 128, 64, FAKE, 4607, None) == moe.MOE_ERR_INVALID_ARG


def test_q8_pack_argument_checks(lib):
    assert moe.moe_q8_packed_bytes(128, 1536, 2048) == 128 * 1536 * 2048 * 34 // 32
    assert moe.moe_q8_packed_bytes(1, 128, 64) == 8704
    assert moe.moe_q8_packed_bytes(1, 100, 64) == 0
    assert moe.moe_q8_packed_bytes(1, 128, 32) == 0
    f = lib.moe_q8_pack
    assert f(FAKE, FAKE, 1, 100, 64, FAKE, 8704, None) == moe.MOE_ERR_SHAPE
    assert f(FAKE, FAKE, 1, 128, 96, FAKE, 8704, None) == moe.MOE_ERR_SHAPE
    assert f(FAKE, None, 1, 128, 64, FAKE, 8704, None) == moe.MOE_ERR_INVALID_ARG
    assert f(FAKE + 4, FAKE, 1, 128, 64, FAKE, 8704, None) == moe.MOE_ERR_ALIGN
    assert f(FAKE, FAKE, 1, 128, 64, FAKE, 8703, None) == moe.MOE_ERR_INVALID_ARG


def test_route_argument_checks(lib):
    f = lib.moe_route_topk
    assert f(FAKE, FAKE, 4, 256, 300, 2, FAKE, FAKE, None, None) == moe.MOE_ERR_SHAPE
    assert f(FAKE, FAKE, 4, 256, 8, 9, FAKE, FAKE, None, None) == moe.MOE_ERR_SHAPE
    assert f(FAKE, FAKE, 4, 250, 8, 2, FAKE, FAKE, None, None) == moe.MOE_ERR_SHAPE
    assert f(None, FAKE, 4, 256, 8, 2, FAKE, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 256, 8, 2, FAKE + 4, FAKE, None, None) == moe.MOE_ERR_ALIGN
    assert f(FAKE, FAKE, 0, 256, 8, 2, FAKE, FAKE, None, None) == moe.MOE_OK


def test_quantize_argument_checks(lib):
    q = lib.moe_q4_quantize
    assert q(7, FAKE, 4, 64, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG       # source type
    assert q(0, FAKE, 4, 64, 5, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG       # format
    assert q(0, FAKE, 4, 40, 0, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE             # K % 32
    assert q(0, FAKE, -1, 64, 0, FAKE, FAKE, None) == moe.MOE_ERR_SHAPE            # rows < 0
    assert q(0, None, 4, 64, 0, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG       # null src
    assert q(0, FAKE, 4, 64, 0, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG       # no scales
    assert q(0, FAKE, 4, 64, 1, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG       # block18 + scales
    assert q(0, FAKE + 4, 4, 64, 0, FAKE, FAKE, None) == moe.MOE_ERR_ALIGN
    assert q(0, FAKE, 0, 64, 0, None, None, None) == moe.MOE_OK                     # nothing to do


def _streamed(lib, L=2, T=4, H=256, I=128, E=8, k=2, flags=2, x=FAKE, layer=(FAKE, FAKE, FAKE),
              bad_layer=None, out=FAKE * 2, ws=FAKE * 3, ws_bytes=1 << 40):
    ptrs = [list(layer) for _ in range(max(L, 1))]
    if bad_layer is not None:
        ptrs[bad_layer[0]][bad_layer[1]] = bad_layer[2]
    arrs = [(ctypes.c_void_p * len(ptrs))(*[p[j] for p in ptrs]) for j in range(3)]
    return lib.moe_q4_forward_prefill_stack_streamed(x, L, arrs[0], arrs[1], arrs[2], T, H, I, E, k,
                                                     flags, out, ws, ws_bytes, None)


def test_prefill_stack_streamed_argument_checks(lib):
    # every refusal here comes before the library touches the GPU
    assert _streamed(lib, L=0) == moe.MOE_ERR_SHAPE
    assert _streamed(lib, L=moe.MOE_DECODE_MAX_LAYERS + 1) == moe.MOE_ERR_SHAPE
    assert _streamed(lib, H=200) == moe.MOE_ERR_SHAPE
    assert _streamed(lib, flags=4) == moe.MOE_ERR_INVALID_ARG
    assert _streamed(lib, x=None) == moe.MOE_ERR_INVALID_ARG
    assert _streamed(lib, bad_layer=(1, 1, None)) == moe.MOE_ERR_INVALID_ARG  # layer 1's gate/up
    assert b"layer 1" in lib.moe_last_error_string()
    assert _streamed(lib, bad_layer=(0, 2, FAKE + 8)) == moe.MOE_ERR_ALIGN
    assert _streamed(lib, out=FAKE) == moe.MOE_ERR_INVALID_ARG               # out aliases x
    assert _streamed(lib, ws_bytes=16) == moe.MOE_ERR_WORKSPACE
    assert _streamed(lib, T=0) == moe.MOE_OK                                 # empty input: no-op


def test_streamed_workspace_holds_two_layers_of_experts():
    T, H, I, E, k = 2048, 2048, 768, 128, 8
    pre = moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL, T, H, I, E, k)
    experts = moe.moe_q4_packed_bytes(E, 2 * I, H) + moe.moe_q4_packed_bytes(E, H, I)
    got = moe.moe_workspace_bytes(moe.MOE_MODE_PREFILL_STREAMED, T, H, I, E, k)
    assert pre + 2 * experts + 2 * T * H * 2 <= got <= pre + 2 * experts + 2 * T * H * 2 + 8 * 256
