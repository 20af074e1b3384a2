"""The C-ABI library builds, loads and exports every declared entry point;
host-side argument checks answer without touching a GPU."""
import ctypes as C
import os
import re

import pytest

from int4_weight_kv_w4a16_gb300 import build, futr
from int4_weight_kv_w4a16_gb300.inputs import LLAMA8B, LLAMA70B, TOY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return futr.lib()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(futr_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("futr_pack_weights", "futr_kv_append", "futr_decode_block"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    # the binding exposes the same names
    for n in names:
        assert hasattr(futr, n), n


def test_debug_variant_builds_and_exports_the_same_symbols():
    """libfutr_debug.so (-DFUTR_DEBUG: device bounds checks) builds from the
    same sources and exports every declared entry point."""
    path = build.build(debug=True)
    assert os.path.basename(path) == "libfutr_debug.so"
    D = C.CDLL(path)
    for n in declared_functions():
        assert hasattr(D, n), n
    D.futr_status_string.restype = C.c_char_p
    assert b"bounds" in D.futr_status_string(futr.FUTR_ERR_BOUNDS)
    assert b"guard" in D.futr_status_string(futr.FUTR_ERR_CORRUPT)


def test_struct_sizes_match_binding(L):
    # futr_shape: 9 x 4 bytes; descriptors are plain data with 8-byte fields
    assert C.sizeof(futr.futr_shape) == 36
    assert C.sizeof(futr.futr_kv) % 8 == 0 and C.sizeof(futr.futr_ws) % 8 == 0


def test_status_strings_and_version(L):
    assert futr.futr_status_string(0) == "ok"
    assert "position" in futr.futr_status_string(futr.FUTR_ERR_OUT_OF_RANGE)
    assert futr.futr_status_string(99) == "unknown status"
    assert futr.futr_version() >= 10000


def _blob_bytes(shape):
    units = 0
    q = (shape.n_q_heads + 2 * shape.n_kv_heads) * shape.head_dim
    for rows, cols in ((q, shape.hidden), (shape.hidden, shape.n_q_heads * shape.head_dim),
                       (2 * shape.inter, shape.hidden), (shape.hidden, shape.inter)):
        sec = (rows // 128) * (cols // 128) * 8448
        units += (sec + 255) // 256 * 256
    return 256 + units


@pytest.mark.parametrize("shape", [TOY, LLAMA8B, LLAMA70B], ids=["toy", "8b", "70b"])
def test_weights_size(L, shape):
    n = futr.futr_weights_size(futr.make_shape(shape))
    assert n == _blob_bytes(shape)
    # INT4 codes + fp16 scales of every projection
    params = shape.hidden * shape.qkv_rows + shape.hidden * shape.q_rows + 3 * shape.hidden * shape.inter
    assert n >= params // 2 + params // 128 * 2


def test_unsupported_shapes_rejected(L):
    import dataclasses
    bad = [dataclasses.replace(TOY, head_dim=96), dataclasses.replace(TOY, group=64),
           dataclasses.replace(TOY, hidden=200), dataclasses.replace(TOY, had_block=48),
           dataclasses.replace(TOY, had_block=128), dataclasses.replace(TOY, n_q_heads=3),
           dataclasses.replace(TOY, inter=700)]
    for s in bad:
        n = C.c_size_t()
        assert L.futr_weights_size(C.byref(futr.make_shape(s)), C.byref(n)) == futr.FUTR_ERR_UNSUPPORTED


def test_null_arguments_rejected_without_gpu(L):
    sh = futr.make_shape(TOY)
    n = C.c_size_t()
    assert L.futr_weights_size(C.byref(sh), None) == futr.FUTR_ERR_INVALID_ARG
    args = [None] * 10
    assert L.futr_pack_weights(C.byref(sh), *args, 0, None) == futr.FUTR_ERR_INVALID_ARG
    assert L.futr_kv_size(C.byref(sh), 0, 1, 16, C.byref(n)) == futr.FUTR_ERR_INVALID_ARG
    kv = futr.futr_kv()  # never initialised: magic mismatch
    assert L.futr_kv_append(C.byref(kv), 0, 0, 1, None, 1, None, None, None) == futr.FUTR_ERR_INVALID_ARG
    ws = futr.futr_ws()
    assert L.futr_decode_block(None, None, C.byref(kv), 0, 1, None, None, C.byref(ws), None) == \
        futr.FUTR_ERR_INVALID_ARG


def test_kv_size_formula(L):
    sh = futr.make_shape(LLAMA8B)
    n = futr.futr_kv_size(sh, 2, 3, 1000)  # capacity rounds up to 1008
    streams = 2 * 3 * 8 * 1008 * (128 + 4)
    rope = 1008 * 64 * 8
    # + the error word and three 256-byte guards (one after each region), 256-byte aligned
    assert n >= streams + rope + 16 + 3 * 256 and n <= streams + rope + 2048


def test_kv_size_beyond_32_bits(L):
    # a 70B model's whole cache: 80 layers x 32 sequences x 65536 positions,
    # 8 kv-heads x (128 code bytes + 4 scale bytes) per position -- 177 GB
    n = futr.futr_kv_size(futr.make_shape(LLAMA70B), 80, 32, 65536)
    streams = 80 * 32 * 8 * 65536 * (128 + 4)
    assert streams > 2 ** 32
    assert streams + 65536 * 64 * 8 <= n <= streams + 65536 * 64 * 8 + 2048
    # one position more than the supported capacity is refused
    sz = C.c_size_t(0)
    assert L.futr_kv_size(C.byref(futr.make_shape(LLAMA70B)), 80, 32, 65537, C.byref(sz)) == futr.FUTR_ERR_UNSUPPORTED


def test_no_alloc_rejects_zeroed_cache_descriptor(L):
    """A cache descriptor that was never initialised (all zero, so its shape
    has no kv-heads) is refused before its shape sizes anything."""
    kv = futr.futr_kv()
    buf = (C.c_uint16 * 256)()
    pos = (C.c_int32 * 1)()
    assert L.futr_decode_block_noalloc(C.addressof(buf), C.addressof(buf), C.byref(kv), 0, 1, C.addressof(pos),
                                       C.addressof(buf) + 256, None) == futr.FUTR_ERR_INVALID_ARG
    assert L.futr_decode_block_noalloc(None, None, None, 0, 1, None, None, None) == futr.FUTR_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [TOY, LLAMA8B, LLAMA70B], ids=["toy", "8b", "70b"])
def test_gptq_scratch_size_covers_its_buffers(L, shape):
    """Two float64 K x K matrices for the widest projection input, a float64
    copy of the largest single projection, its block errors and its codes."""
    n = futr.futr_gptq_scratch_size(futr.make_shape(shape))
    kmax = max(shape.hidden, shape.q_rows, shape.inter)
    largest = max(shape.qkv_rows * shape.hidden, shape.hidden * shape.q_rows, shape.inter * shape.hidden,
                  shape.hidden * shape.inter)
    assert n >= 2 * 8 * kmax * kmax + 8 * largest + 2 * largest


def test_gptq_arguments_rejected_without_gpu(L):
    sh = futr.make_shape(TOY)
    fake = C.c_void_p(1 << 20)  # never dereferenced: every check below is on the host
    blob_n = futr.futr_weights_size(sh)
    scr_n = futr.futr_gptq_scratch_size(sh)
    ptrs = [fake] * 13

    def call(damp=0.01, scr=fake, scr_n=scr_n, blob=fake, blob_n=blob_n, ptrs=ptrs):
        return L.futr_pack_weights_gptq(C.byref(sh), *ptrs, C.c_double(damp), scr, scr_n, blob, blob_n, None)

    assert call(damp=0.0) == futr.FUTR_ERR_INVALID_ARG
    assert call(damp=-1.0) == futr.FUTR_ERR_INVALID_ARG
    assert call(damp=float("nan")) == futr.FUTR_ERR_INVALID_ARG
    assert call(scr_n=scr_n - 1) == futr.FUTR_ERR_INVALID_ARG
    assert call(scr=C.c_void_p((1 << 20) + 16)) == futr.FUTR_ERR_INVALID_ARG
    assert call(blob_n=blob_n - 1) == futr.FUTR_ERR_INVALID_ARG
    assert call(scr=None) == futr.FUTR_ERR_INVALID_ARG
    assert call(ptrs=[fake] * 12 + [None]) == futr.FUTR_ERR_INVALID_ARG
    import dataclasses
    bad = futr.make_shape(dataclasses.replace(TOY, head_dim=96))
    assert L.futr_pack_weights_gptq(C.byref(bad), *ptrs, C.c_double(0.01), fake, scr_n, fake, blob_n, None) == \
        futr.FUTR_ERR_UNSUPPORTED
    assert "positive definite" in futr.futr_status_string(futr.FUTR_ERR_NOT_PD)
