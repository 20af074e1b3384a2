"""Thin ctypes binding of libfutr.so (C ABI in include/futr.h).

Every function here only marshals arguments: device buffers are torch CUDA
tensors (passed by ``data_ptr()``), streams are torch streams (or None for the
current stream), descriptors are the ctypes mirrors of the C structs.  All
arithmetic runs in the library's kernels; if the library is missing, ``lib()``
raises and nothing falls back to another implementation.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfutr.so")
LIB_DEBUG_PATH = os.path.join(PKG, "libfutr_debug.so")

FUTR_OK = 0
FUTR_ERR_INVALID_ARG = 1
FUTR_ERR_UNSUPPORTED = 2
FUTR_ERR_CUDA = 3
FUTR_ERR_OUT_OF_RANGE = 4
FUTR_ERR_TIMEOUT = 5
FUTR_ERR_BAD_BLOB = 6
FUTR_ERR_NOT_PD = 7
FUTR_ERR_CORRUPT = 8
FUTR_ERR_BOUNDS = 9

FUTR_PROJ_QKV, FUTR_PROJ_O, FUTR_PROJ_GATE, FUTR_PROJ_UP, FUTR_PROJ_DOWN = range(5)


class futr_shape(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("inter", C.c_int32), ("group", C.c_int32),
                ("had_block", C.c_int32), ("rms_eps", C.c_float), ("rope_theta", C.c_float)]


class futr_kv(C.Structure):
    _fields_ = [("shape", futr_shape), ("n_layers", C.c_int32), ("max_batch", C.c_int32),
                ("capacity", C.c_int32), ("_pad", C.c_int32), ("base", C.c_void_p),
                ("bytes", C.c_uint64), ("stream_bytes", C.c_uint64), ("rope_offset", C.c_uint64),
                ("err_offset", C.c_uint64), ("magic", C.c_uint64)]


class futr_ws(C.Structure):
    _fields_ = [("shape", futr_shape), ("max_batch", C.c_int32), ("capacity", C.c_int32),
                ("n_sm", C.c_int32), ("_pad", C.c_int32), ("base", C.c_void_p), ("bytes", C.c_uint64),
                ("off_err", C.c_uint64), ("off_qrot", C.c_uint64), ("off_o", C.c_uint64),
                ("off_h", C.c_uint64), ("off_a", C.c_uint64), ("off_xin", C.c_uint64),
                ("off_yout", C.c_uint64), ("off_pos", C.c_uint64), ("off_part", C.c_uint64),
                ("part_bytes", C.c_uint64), ("off_apart", C.c_uint64), ("apart_bytes", C.c_uint64),
                ("off_cnt", C.c_uint64), ("cnt_words", C.c_uint64), ("magic", C.c_uint64)]


class FutrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.futr_status_string(status).decode() if _lib else status}")


_lib: Optional[C.CDLL] = None
P = C.c_void_p
I32 = C.c_int32
_SIGS = {
    "futr_status_string": (C.c_char_p, [I32]),
    "futr_version": (I32, []),
    "futr_weights_size": (I32, [C.POINTER(futr_shape), C.POINTER(C.c_size_t)]),
    "futr_pack_weights": (I32, [C.POINTER(futr_shape)] + [P] * 10 + [C.c_size_t, P]),
    "futr_gptq_scratch_size": (I32, [C.POINTER(futr_shape), C.POINTER(C.c_size_t)]),
    "futr_pack_weights_gptq": (I32, [C.POINTER(futr_shape)] + [P] * 13 + [C.c_double, P, C.c_size_t, P,
                                                                          C.c_size_t, P]),
    "futr_unpack_weights": (I32, [C.POINTER(futr_shape), P, I32, P, P, P]),
    "futr_kv_size": (I32, [C.POINTER(futr_shape), I32, I32, I32, C.POINTER(C.c_size_t)]),
    "futr_kv_init": (I32, [C.POINTER(futr_shape), I32, I32, I32, P, C.c_size_t, C.POINTER(futr_kv), P]),
    "futr_kv_append": (I32, [C.POINTER(futr_kv), I32, I32, I32, P, I32, P, P, P]),
    "futr_kv_read": (I32, [C.POINTER(futr_kv), I32, I32, I32, P, P, P, P, P]),
    "futr_workspace_size": (I32, [C.POINTER(futr_shape), I32, I32, C.POINTER(C.c_size_t)]),
    "futr_workspace_init": (I32, [C.POINTER(futr_shape), I32, I32, P, C.c_size_t, C.POINTER(futr_ws), P]),
    "futr_decode_block": (I32, [P, P, C.POINTER(futr_kv), I32, I32, P, P, C.POINTER(futr_ws), P]),
    "futr_decode_block_timed": (I32, [P, P, C.POINTER(futr_kv), I32, I32, P, P, C.POINTER(futr_ws), P,
                                      C.POINTER(C.c_float)]),
    "futr_decode_block_host": (I32, [P, P, C.POINTER(futr_kv), I32, I32, P, P, C.POINTER(futr_ws), P]),
    "futr_check": (I32, [C.POINTER(futr_ws), C.POINTER(futr_kv), P]),
    "futr_decode_block_noalloc": (I32, [P, P, C.POINTER(futr_kv), I32, I32, P, P, P]),
    "futr_decode_step": (I32, [P, P, I32, C.POINTER(C.c_void_p), I32, C.POINTER(futr_kv), I32, P, P, P, P,
                               C.POINTER(futr_ws), P]),
}


def lib() -> C.CDLL:
    """Load libfutr.so (built by ``build.py``), or its debug variant
    libfutr_debug.so (``build.py --debug``: device bounds checks) when the
    environment has FUTR_DEBUG=1; raises if that library is missing."""
    global _lib
    if _lib is None:
        path = LIB_DEBUG_PATH if os.environ.get("FUTR_DEBUG") == "1" else LIB_PATH
        if not os.path.exists(path):
            flag = " --debug" if path == LIB_DEBUG_PATH else ""
            raise RuntimeError(f"{path} is not built; run int4_weight_kv_w4a16_gb300/build.py{flag}")
        h = C.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def _ok(status: int, where: str) -> None:
    if status != FUTR_OK:
        raise FutrError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):  # numpy (host buffers)
        return t.ctypes.data
    raise TypeError(f"cannot pass {type(t)} as a buffer")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(s) -> futr_shape:
    """futr_shape from any object with the BlockShape attributes."""
    return futr_shape(s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.inter, s.group, s.had_block,
                      s.rms_eps, s.rope_theta)


def futr_status_string(status: int) -> str:
    return lib().futr_status_string(status).decode()


def futr_version() -> int:
    return lib().futr_version()


def futr_weights_size(shape: futr_shape) -> int:
    n = C.c_size_t()
    _ok(lib().futr_weights_size(C.byref(shape), C.byref(n)), "futr_weights_size")
    return n.value


def futr_pack_weights(shape, wq, wk, wv, wo, wgate, wup, wdown, g_attn, g_mlp, blob, stream=None):
    _ok(lib().futr_pack_weights(C.byref(shape), *[_ptr(t) for t in (wq, wk, wv, wo, wgate, wup, wdown,
                                                                    g_attn, g_mlp, blob)],
                                blob.numel() * blob.element_size(), _stream(stream)), "futr_pack_weights")


def futr_gptq_scratch_size(shape) -> int:
    n = C.c_size_t()
    _ok(lib().futr_gptq_scratch_size(C.byref(shape), C.byref(n)), "futr_gptq_scratch_size")
    return n.value


def futr_pack_weights_gptq(shape, wq, wk, wv, wo, wgate, wup, wdown, g_attn, g_mlp, h_attn, h_o, h_mlp, h_down,
                           damp, scratch, blob, stream=None):
    _ok(lib().futr_pack_weights_gptq(C.byref(shape), *[_ptr(t) for t in (wq, wk, wv, wo, wgate, wup, wdown,
                                                                         g_attn, g_mlp, h_attn, h_o, h_mlp,
                                                                         h_down)],
                                     float(damp), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                     _ptr(blob), blob.numel() * blob.element_size(), _stream(stream)),
        "futr_pack_weights_gptq")


def futr_unpack_weights(shape, blob, which, codes, scales, stream=None):
    _ok(lib().futr_unpack_weights(C.byref(shape), _ptr(blob), which, _ptr(codes), _ptr(scales),
                                  _stream(stream)), "futr_unpack_weights")


def futr_kv_size(shape, n_layers, max_batch, capacity) -> int:
    n = C.c_size_t()
    _ok(lib().futr_kv_size(C.byref(shape), n_layers, max_batch, capacity, C.byref(n)), "futr_kv_size")
    return n.value


def futr_kv_init(shape, n_layers, max_batch, capacity, kv_mem, stream=None) -> futr_kv:
    kv = futr_kv()
    _ok(lib().futr_kv_init(C.byref(shape), n_layers, max_batch, capacity, _ptr(kv_mem),
                           kv_mem.numel() * kv_mem.element_size(), C.byref(kv), _stream(stream)), "futr_kv_init")
    kv._mem = kv_mem  # keep the device buffer alive with the descriptor
    return kv


def futr_kv_append(kv, layer, seq0, batch, pos, n_tok, k, v, stream=None):
    _ok(lib().futr_kv_append(C.byref(kv), layer, seq0, batch, _ptr(pos), n_tok, _ptr(k), _ptr(v),
                             _stream(stream)), "futr_kv_append")


def futr_kv_read(kv, layer, seq, n_pos, k_codes, k_scales, v_codes, v_scales, stream=None):
    _ok(lib().futr_kv_read(C.byref(kv), layer, seq, n_pos, _ptr(k_codes), _ptr(k_scales), _ptr(v_codes),
                           _ptr(v_scales), _stream(stream)), "futr_kv_read")


def futr_workspace_size(shape, max_batch, capacity) -> int:
    n = C.c_size_t()
    _ok(lib().futr_workspace_size(C.byref(shape), max_batch, capacity, C.byref(n)), "futr_workspace_size")
    return n.value


def futr_workspace_init(shape, max_batch, capacity, ws_mem, stream=None) -> futr_ws:
    ws = futr_ws()
    _ok(lib().futr_workspace_init(C.byref(shape), max_batch, capacity, _ptr(ws_mem),
                                  ws_mem.numel() * ws_mem.element_size(), C.byref(ws), _stream(stream)),
        "futr_workspace_init")
    ws._mem = ws_mem
    return ws


def futr_decode_block(x, blob, kv, layer, batch, pos, y, ws, stream=None):
    _ok(lib().futr_decode_block(_ptr(x), _ptr(blob), C.byref(kv), layer, batch, _ptr(pos), _ptr(y),
                                C.byref(ws), _stream(stream)), "futr_decode_block")


def futr_decode_block_timed(x, blob, kv, layer, batch, pos, y, ws, stream=None) -> Sequence[float]:
    out = (C.c_float * 5)()
    _ok(lib().futr_decode_block_timed(_ptr(x), _ptr(blob), C.byref(kv), layer, batch, _ptr(pos), _ptr(y),
                                      C.byref(ws), _stream(stream), out), "futr_decode_block_timed")
    return list(out)


def futr_decode_block_host(x_host, blob, kv, layer, batch, pos_host, y_host, ws, stream=None):
    _ok(lib().futr_decode_block_host(_ptr(x_host), _ptr(blob), C.byref(kv), layer, batch, _ptr(pos_host),
                                     _ptr(y_host), C.byref(ws), _stream(stream)), "futr_decode_block_host")


def futr_decode_step(tokens, embedding, vocab, blobs, kv, batch, pos, g_final, lm_head, logits, ws, stream=None):
    """One complete decode step (embedding, every block in ``blobs``, final
    norm, bf16 LM head) -> fp32 logits [batch, vocab]."""
    arr = (C.c_void_p * len(blobs))(*[_ptr(b) for b in blobs])
    _ok(lib().futr_decode_step(_ptr(tokens), _ptr(embedding), vocab, arr, len(blobs), C.byref(kv), batch,
                               _ptr(pos), _ptr(g_final), _ptr(lm_head), _ptr(logits), C.byref(ws),
                               _stream(stream)), "futr_decode_step")


def futr_decode_block_noalloc(x, blob, kv, layer, batch, pos, y, stream=None):
    """futr_decode_block with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _ok(lib().futr_decode_block_noalloc(_ptr(x), _ptr(blob), C.byref(kv), layer, batch, _ptr(pos), _ptr(y),
                                        _stream(stream)), "futr_decode_block_noalloc")


def futr_check(ws=None, kv=None, stream=None) -> int:
    """Synchronize and return the device status (0 = ok); does not raise."""
    return lib().futr_check(C.byref(ws) if ws is not None else None, C.byref(kv) if kv is not None else None,
                            _stream(stream))


# ----------------------------------------------------------------------------
# allocation helpers (torch provides the device memory)
# ----------------------------------------------------------------------------

def alloc_bytes(n: int, device="cuda"):
    import torch
    # 256-byte aligned: the caching allocator aligns blocks to at least 512 bytes
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def ws_view(ws: futr_ws, name: str, shape, dtype):
    """A tensor view of one workspace region (e.g. 'h', 'a', 'o', 'qrot')."""
    import torch
    off = getattr(ws, "off_" + name)
    n = 1
    for s in shape:
        n *= s
    esize = torch.empty((), dtype=dtype).element_size()
    return ws._mem[off:off + n * esize].view(dtype).view(*shape)
