"""ctypes binding of liblowrank.so (declared in include/lowrank.h).

Argument marshalling only: each function here has the name of the C entry
point it calls, takes torch tensors (device memory) or raw integers for the
pointer arguments, and raises LowRankError when the call returns a non-zero
lr_status.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind: if the shared library is missing or cannot
be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liblowrank.so")

LR_F32, LR_BF16 = 0, 1
LR_SAVE_FULL, LR_SAVE_CKPT = 0, 1
LR_ACT_SILU, LR_ACT_IDENTITY = 0, 1
STATUS = {
    0: "LR_OK", 1: "LR_ERR_NULL", 2: "LR_ERR_SHAPE", 3: "LR_ERR_ALIGN", 4: "LR_ERR_DTYPE",
    5: "LR_ERR_WORKSPACE", 6: "LR_ERR_CUDA", 7: "LR_ERR_TIMEOUT", 8: "LR_ERR_UNSUPPORTED",
}
EXPORTED = [
    "lr_mlp_saved_bytes", "lr_mlp_fwd_workspace_bytes", "lr_mlp_bwd_workspace_bytes", "lr_mlp_fwd",
    "lr_mlp_bwd", "lr_proj_saved_bytes", "lr_proj_fwd_workspace_bytes", "lr_proj_bwd_workspace_bytes",
    "lr_proj_fwd", "lr_proj_bwd", "lr_stack_workspace_bytes", "lr_stack_step", "lr_last_error",
    "lr_check_device_error", "lr_selftest_wait_timeout", "lr_version", "lr_launch_count",
    "lr_profile_start", "lr_profile_stop", "lr_profile_filter", "lr_profile_count", "lr_profile_entry",
    "lr_proj_fwd_noalloc", "lr_dense_saved_bytes", "lr_dense_fwd_workspace_bytes", "lr_dense_bwd_workspace_bytes",
    "lr_dense_fwd", "lr_dense_bwd", "lr_btp_payload_floats", "lr_btp_workspace_bytes", "lr_btp_partial",
    "lr_btp_finish", "lr_attn_saved_bytes", "lr_attn_workspace_bytes", "lr_attn_fwd", "lr_attn_bwd",
    "lr_block_saved_bytes", "lr_block_workspace_bytes", "lr_block_fwd", "lr_block_bwd",
]


class LowRankError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class lr_pair(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p)]


class lr_pair_grad(ctypes.Structure):
    _fields_ = [("dA", ctypes.c_void_p), ("dB", ctypes.c_void_p)]


class lr_block_weights(ctypes.Structure):
    _fields_ = [("g_attn", ctypes.c_void_p), ("q", lr_pair), ("k", lr_pair), ("v", lr_pair), ("o", lr_pair),
                ("g_mlp", ctypes.c_void_p), ("gate", lr_pair), ("up", lr_pair), ("down", lr_pair)]


class lr_block_grads(ctypes.Structure):
    _fields_ = [("dg_attn", ctypes.c_void_p), ("q", lr_pair_grad), ("k", lr_pair_grad), ("v", lr_pair_grad),
                ("o", lr_pair_grad), ("dg_mlp", ctypes.c_void_p), ("gate", lr_pair_grad), ("up", lr_pair_grad),
                ("down", lr_pair_grad)]


_lib = None

_I, _F, _P, _SZ = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_SIGS = {
    "lr_mlp_saved_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "lr_mlp_fwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "lr_mlp_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "lr_mlp_fwd": (_I, [_I, _I, _I, _I, _I, _I, _I, _F, _P, _P, lr_pair, lr_pair, lr_pair, _P, _P, _SZ, _P, _SZ,
                        _P]),
    "lr_mlp_bwd": (_I, [_I, _I, _I, _I, _I, _I, _I, _F, _P, _P, lr_pair, lr_pair, lr_pair, _P, _SZ, _P, _P, _P,
                        lr_pair_grad, lr_pair_grad, lr_pair_grad, _P, _SZ, _P]),
    "lr_proj_saved_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "lr_proj_fwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "lr_proj_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "lr_proj_fwd": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(lr_pair), _P, _F, _P, ctypes.POINTER(_P), _P,
                         _SZ, _P, _SZ, _P]),
    "lr_proj_bwd": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(lr_pair), _P, _F, _P, _P, _SZ,
                         ctypes.POINTER(_P),
                         _P, _P, ctypes.POINTER(lr_pair_grad), _P, _SZ, _P]),
    "lr_proj_fwd_noalloc": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(lr_pair), _P, _F, _P, ctypes.POINTER(_P),
                                 _P, _SZ, _P]),
    "lr_stack_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "lr_dense_saved_bytes": (_SZ, [_I, _I, _I, _I]),
    "lr_btp_payload_floats": (_SZ, [_I, _I, _I]),
    "lr_btp_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "lr_btp_partial": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(lr_pair), _P, _P, _P, _P, _SZ, _P]),
    "lr_btp_finish": (_I, [_I, _I, _I, _I, _I, _I, _P, _F, _P, _P, _P, _P]),
    "lr_block_saved_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "lr_block_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "lr_block_fwd": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _F, _P, ctypes.POINTER(lr_block_weights), _P, _P, _SZ, _P,
                          _SZ, _P]),
    "lr_block_bwd": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _F, _P, ctypes.POINTER(lr_block_weights), _P, _SZ, _P, _P,
                          ctypes.POINTER(lr_block_grads), _P, _SZ, _P]),
    "lr_attn_saved_bytes": (_SZ, [_I, _I, _I, _I]),
    "lr_attn_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "lr_attn_fwd": (_I, [_I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _SZ, _P, _SZ, _P]),
    "lr_attn_bwd": (_I, [_I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "lr_dense_fwd_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "lr_dense_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "lr_dense_fwd": (_I, [_I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _SZ, _P]),
    "lr_dense_bwd": (_I, [_I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "lr_stack_step": (_I, [_I, _I, _I, _I, _I, _I, _I, _F, _P, _P, ctypes.POINTER(_P), ctypes.POINTER(lr_pair), _P,
                           _P, ctypes.POINTER(_P), ctypes.POINTER(lr_pair_grad), _P, _SZ, _P]),
    "lr_last_error": (ctypes.c_char_p, []),
    "lr_check_device_error": (_I, [_P]),
    "lr_selftest_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "lr_version": (_I, []),
    "lr_launch_count": (ctypes.c_ulonglong, []),
    "lr_profile_start": (_I, []),
    "lr_profile_stop": (_I, []),
    "lr_profile_filter": (_I, [ctypes.c_char_p]),
    "lr_profile_count": (_I, []),
    "lr_profile_entry": (_I, [_I, ctypes.c_char_p, _SZ, ctypes.POINTER(ctypes.c_longlong),
                              ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_double)]),
}


def lib() -> ctypes.CDLL:
    """Load liblowrank.so (built in-tree by rank_bottleneck_block_gb300.build); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m rank_bottleneck_block_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------- marshalling
def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != 0:
        raise LowRankError(status, lib().lr_last_error().decode())


def dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return LR_BF16
    if t.dtype == torch.float32:
        return LR_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def pair(A, B) -> lr_pair:
    return lr_pair(_p(A), _p(B))


def pair_grad(dA, dB) -> lr_pair_grad:
    return lr_pair_grad(_p(dA), _p(dB))


# ---------------------------------------------------------- entry points
def lr_version() -> int:
    return lib().lr_version()


def lr_last_error() -> str:
    return lib().lr_last_error().decode()


def lr_mlp_saved_bytes(dt, mode, T, d, f, r) -> int:
    return lib().lr_mlp_saved_bytes(dt, mode, T, d, f, r)


def lr_mlp_fwd_workspace_bytes(dt, mode, T, d, f, r) -> int:
    return lib().lr_mlp_fwd_workspace_bytes(dt, mode, T, d, f, r)


def lr_mlp_bwd_workspace_bytes(dt, mode, T, d, f, r) -> int:
    return lib().lr_mlp_bwd_workspace_bytes(dt, mode, T, d, f, r)


def lr_mlp_fwd(dt, mode, T, d, f, r, eps, x, g, gate, up, down, out, saved, ws, stream=None, act=None):
    act = LR_ACT_SILU if act is None else act
    _check(lib().lr_mlp_fwd(dt, mode, act, T, d, f, r, eps, _p(x), _p(g), gate, up, down, _p(out), _p(saved),
                            _nbytes(saved), _p(ws), _nbytes(ws), _stream(stream)))


def lr_mlp_bwd(dt, mode, T, d, f, r, eps, x, g, gate, up, down, saved, dout, dx, dg, dgate, dup, ddown, ws,
               stream=None, act=None):
    act = LR_ACT_SILU if act is None else act
    _check(lib().lr_mlp_bwd(dt, mode, act, T, d, f, r, eps, _p(x), _p(g), gate, up, down, _p(saved),
                            _nbytes(saved), _p(dout), _p(dx), _p(dg), dgate, dup, ddown, _p(ws), _nbytes(ws),
                            _stream(stream)))


def lr_proj_saved_bytes(dt, T, d_in, d_out, r, group, norm) -> int:
    return lib().lr_proj_saved_bytes(dt, T, d_in, d_out, r, group, int(norm))


def lr_proj_fwd_workspace_bytes(dt, T, d_in, d_out, r, group, norm) -> int:
    return lib().lr_proj_fwd_workspace_bytes(dt, T, d_in, d_out, r, group, int(norm))


def lr_proj_bwd_workspace_bytes(dt, T, d_in, d_out, r, group, norm) -> int:
    return lib().lr_proj_bwd_workspace_bytes(dt, T, d_in, d_out, r, group, int(norm))


def _pairs(ps: Sequence[lr_pair]):
    arr = (lr_pair * len(ps))(*ps)
    return arr


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[_p(t) for t in ts])


def lr_proj_fwd(dt, T, d_in, d_out, r, pairs: Sequence[lr_pair], g, eps, x, outs, saved, ws, stream=None,
                act=None):
    act = LR_ACT_SILU if act is None else act
    group = len(pairs)
    _check(lib().lr_proj_fwd(dt, act, T, d_in, d_out, r, group, _pairs(pairs), _p(g), eps, _p(x), _ptrs(outs),
                             _p(saved), _nbytes(saved), _p(ws), _nbytes(ws), _stream(stream)))


def lr_proj_bwd(dt, T, d_in, d_out, r, pairs: Sequence[lr_pair], g, eps, x, saved, douts, dx, dg,
                grads: Sequence[lr_pair_grad], ws, stream=None, act=None):
    act = LR_ACT_SILU if act is None else act
    group = len(pairs)
    garr = (lr_pair_grad * group)(*grads)
    _check(lib().lr_proj_bwd(dt, act, T, d_in, d_out, r, group, _pairs(pairs), _p(g), eps, _p(x), _p(saved),
                             _nbytes(saved), _ptrs(douts), _p(dx), _p(dg), garr, _p(ws), _nbytes(ws),
                             _stream(stream)))


def lr_dense_saved_bytes(dt, T, d, f) -> int:
    return lib().lr_dense_saved_bytes(dt, T, d, f)


def lr_dense_fwd_workspace_bytes(dt, T, d, f) -> int:
    return lib().lr_dense_fwd_workspace_bytes(dt, T, d, f)


def lr_dense_bwd_workspace_bytes(dt, T, d, f) -> int:
    return lib().lr_dense_bwd_workspace_bytes(dt, T, d, f)


def lr_dense_fwd(dt, T, d, f, eps, x, g, Wg, Wu, Wd, out, saved, ws, stream=None):
    _check(lib().lr_dense_fwd(dt, T, d, f, eps, _p(x), _p(g), _p(Wg), _p(Wu), _p(Wd), _p(out), _p(saved),
                              _nbytes(saved), _p(ws), _nbytes(ws), _stream(stream)))


def lr_dense_bwd(dt, T, d, f, eps, x, g, Wg, Wu, Wd, saved, dout, dx, dg, dWg, dWu, dWd, ws, stream=None):
    _check(lib().lr_dense_bwd(dt, T, d, f, eps, _p(x), _p(g), _p(Wg), _p(Wu), _p(Wd), _p(saved), _nbytes(saved),
                              _p(dout), _p(dx), _p(dg), _p(dWg), _p(dWu), _p(dWd), _p(ws), _nbytes(ws),
                              _stream(stream)))


def lr_attn_saved_bytes(b, s, H, dh) -> int:
    return lib().lr_attn_saved_bytes(b, s, H, dh)


def lr_attn_workspace_bytes(b, s, H, dh) -> int:
    return lib().lr_attn_workspace_bytes(b, s, H, dh)


def lr_attn_fwd(dt, b, s, H, dh, scale, q, k, v, o, saved, ws, stream=None):
    _check(lib().lr_attn_fwd(dt, b, s, H, dh, scale, _p(q), _p(k), _p(v), _p(o), _p(saved), _nbytes(saved), _p(ws),
                             _nbytes(ws), _stream(stream)))


def lr_attn_bwd(dt, b, s, H, dh, scale, q, k, v, o, saved, dout, dq, dk, dv, ws, stream=None):
    _check(lib().lr_attn_bwd(dt, b, s, H, dh, scale, _p(q), _p(k), _p(v), _p(o), _p(saved), _p(dout), _p(dq),
                             _p(dk), _p(dv), _p(ws), _nbytes(ws), _stream(stream)))


def lr_block_saved_bytes(b, s, H, dh, f, ra, rm) -> int:
    return lib().lr_block_saved_bytes(b, s, H, dh, f, ra, rm)


def lr_block_workspace_bytes(b, s, H, dh, f, ra, rm) -> int:
    return lib().lr_block_workspace_bytes(b, s, H, dh, f, ra, rm)


def lr_block_fwd(dt, b, s, H, dh, f, ra, rm, eps, x, w: lr_block_weights, out, saved, ws, stream=None):
    _check(lib().lr_block_fwd(dt, b, s, H, dh, f, ra, rm, eps, _p(x), ctypes.byref(w), _p(out), _p(saved),
                              _nbytes(saved), _p(ws), _nbytes(ws), _stream(stream)))


def lr_block_bwd(dt, b, s, H, dh, f, ra, rm, eps, x, w: lr_block_weights, saved, dout, dx, g: lr_block_grads, ws,
                 stream=None):
    _check(lib().lr_block_bwd(dt, b, s, H, dh, f, ra, rm, eps, _p(x), ctypes.byref(w), _p(saved), _nbytes(saved),
                              _p(dout), _p(dx), ctypes.byref(g), _p(ws), _nbytes(ws), _stream(stream)))


def lr_btp_payload_floats(T, r, group) -> int:
    return lib().lr_btp_payload_floats(T, r, group)


def lr_btp_workspace_bytes(dt, d_shard, r, group) -> int:
    return lib().lr_btp_workspace_bytes(dt, d_shard, r, group)


def lr_btp_partial(dt, T, d_shard, r, pairs: Sequence[lr_pair], g_shard, x_shard, payload, ws, stream=None):
    group = len(pairs)
    _check(lib().lr_btp_partial(dt, T, d_shard, r, group, _pairs(pairs), _p(g_shard), _p(x_shard), _p(payload),
                                _p(ws), _nbytes(ws), _stream(stream)))


def lr_btp_finish(dt, act, T, d, r, group, payload, eps, u, z, s, stream=None):
    _check(lib().lr_btp_finish(dt, act, T, d, r, group, _p(payload), eps, _p(u), _p(z), _p(s), _stream(stream)))


def lr_stack_workspace_bytes(dt, mode, nblocks, T, d, f, r) -> int:
    return lib().lr_stack_workspace_bytes(dt, mode, nblocks, T, d, f, r)


def lr_stack_step(dt, mode, T, d, f, r, eps, x, target, gs, pairs: Sequence[lr_pair], loss, dx, dgs,
                  grads: Sequence[lr_pair_grad], ws, stream=None):
    nblocks = len(gs)
    parr = (lr_pair * len(pairs))(*pairs)
    garr = (lr_pair_grad * len(grads))(*grads)
    _check(lib().lr_stack_step(dt, mode, nblocks, T, d, f, r, eps, _p(x), _p(target), _ptrs(gs), parr, _p(loss),
                               _p(dx), _ptrs(dgs), garr, _p(ws), _nbytes(ws), _stream(stream)))


def lr_check_device_error(stream=None):
    _check(lib().lr_check_device_error(_stream(stream)))


def lr_selftest_wait_timeout(limit_ns: int, stream=None):
    _check(lib().lr_selftest_wait_timeout(limit_ns, _stream(stream)))


def lr_launch_count() -> int:
    return lib().lr_launch_count()


def lr_profile_start():
    _check(lib().lr_profile_start())


def lr_profile_filter(prefix=None):
    """Record only launches whose kernel name starts with `prefix` (None: all)."""
    _check(lib().lr_profile_filter(prefix.encode() if prefix else None))


def lr_profile_stop():
    """Stop profiling and return {kernel name: dict(launches, ms, flops, bytes)}."""
    _check(lib().lr_profile_stop())
    out = {}
    for i in range(lib().lr_profile_count()):
        name = ctypes.create_string_buffer(128)
        n = ctypes.c_longlong()
        ms, fl, by = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        _check(lib().lr_profile_entry(i, name, 128, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(fl),
                                      ctypes.byref(by)))
        out[name.value.decode()] = dict(launches=n.value, ms=ms.value, flops=fl.value, bytes=by.value)
    return out


LR_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def lr_proj_fwd_noalloc(dt, T, d_in, d_out, r, pairs: Sequence[lr_pair], g, eps, x, outs, saved, stream=None):
    """lr_proj_fwd without a workspace, for callers that cannot allocate device memory: its scratch is a
    fixed device array of LR_NOALLOC_SCRATCH_BYTES inside the library, shared by all calls (serialise them)."""
    group = len(pairs)
    _check(lib().lr_proj_fwd_noalloc(dt, T, d_in, d_out, r, group, _pairs(pairs), _p(g), eps, _p(x), _ptrs(outs),
                                     _p(saved), _nbytes(saved), _stream(stream)))
