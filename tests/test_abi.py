"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/lowrank.h declares; size queries and argument validation need no device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lowrank.h")


@pytest.fixture(scope="module")
def L():
    from rank_bottleneck_block_gb300 import build

    build.build()
    from rank_bottleneck_block_gb300 import lowrank

    lowrank.lib()
    return lowrank


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lr_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared()
    assert len(names) >= 15
    lib = L.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(L.EXPORTED) == names


def test_size_queries(L):
    T, d, f, r = 16384, 2048, 5632, 512
    ck = L.lr_mlp_saved_bytes(L.LR_BF16, L.LR_SAVE_CKPT, T, d, f, r)
    full = L.lr_mlp_saved_bytes(L.LR_BF16, L.LR_SAVE_FULL, T, d, f, r)
    # checkpoint keeps u (3r columns, bf16) and s (fp32) per token
    assert ck == pytest.approx(T * (3 * r * 2 + 4), rel=1e-3)
    assert full > 5 * ck
    assert L.lr_mlp_saved_bytes(L.LR_BF16, L.LR_SAVE_CKPT, T, 2047, f, r) == 0  # d not a multiple of 8
    assert L.lr_mlp_saved_bytes(7, 0, T, d, f, r) == 0
    assert L.lr_stack_workspace_bytes(L.LR_BF16, 1, 24, T, d, f, r) < \
        L.lr_stack_workspace_bytes(L.LR_BF16, 0, 24, T, d, f, r) / 3
    assert L.lr_proj_saved_bytes(L.LR_BF16, T, 4096, 4096, 1024, 3, 1) > 0
    assert L.lr_proj_saved_bytes(L.LR_BF16, T, 4096, 4096, 1024, 4, 1) == 0  # group > 3


def _call_mlp_fwd(L, **over):
    p = 0x10000  # a 16-byte aligned fake address: validation must fail before any launch
    args = dict(dt=L.LR_BF16, mode=1, act=0, T=64, d=64, f=128, r=16, x=p, g=p, out=p, saved=p,
                saved_bytes=1 << 30, ws=p, ws_bytes=1 << 30)
    args.update(over)
    pr = L.lr_pair(args.pop("A", p), p)
    lib = L.lib()
    return lib.lr_mlp_fwd(args["dt"], args["mode"], args["act"], args["T"], args["d"], args["f"], args["r"], 1e-6,
                          args["x"],
                          args["g"], pr, L.lr_pair(p, p), L.lr_pair(p, p), args["out"], args["saved"],
                          args["saved_bytes"], args["ws"], args["ws_bytes"], None)


def test_validation_codes(L):
    assert _call_mlp_fwd(L, x=None) == 1
    assert _call_mlp_fwd(L, A=None) == 1
    assert _call_mlp_fwd(L, d=60) == 2
    assert _call_mlp_fwd(L, T=0) == 2
    assert _call_mlp_fwd(L, x=0x10004) == 3
    assert _call_mlp_fwd(L, dt=5) == 4
    assert _call_mlp_fwd(L, mode=9) == 4
    assert _call_mlp_fwd(L, act=2) == 4
    assert _call_mlp_fwd(L, ws_bytes=16) == 5
    assert "ws" in L.lr_last_error()
    assert _call_mlp_fwd(L, saved_bytes=16) == 5


def test_no_device_is_reported_not_faulted(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert _call_mlp_fwd(L) == 8  # LR_ERR_UNSUPPORTED: validated arguments, but no device
    assert L.lib().lr_version() == 100


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    from rank_bottleneck_block_gb300 import lowrank

    monkeypatch.setattr(lowrank, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(lowrank, "_lib", None)
    with pytest.raises(RuntimeError):
        lowrank.lib()


def test_attention_shape_rules(L):
    assert L.lr_attn_saved_bytes(2, 256, 3, 128) == 2 * 3 * 256 * 4
    R = 2 * 3 * 256
    assert L.lr_attn_workspace_bytes(2, 256, 3, 128) >= 2 * R * 256 + 4 * R  # dh 128: bf16 dS^T and D
    assert L.lr_attn_workspace_bytes(2, 256, 3, 128) < 3 * R * 256
    assert L.lr_attn_workspace_bytes(2, 256, 3, 256) > 6 * R * 256  # other dh: fp32 S and bf16 P
    assert L.lr_attn_saved_bytes(1, 200, 1, 128) == 0  # s not a multiple of 256
    assert L.lr_attn_workspace_bytes(1, 256, 1, 64) == 0  # dh not a multiple of 128
    assert L.lr_attn_saved_bytes(1 << 15, 256, 1 << 8, 128) == 0  # b*H*s = 2^31 score rows
    assert L.lr_attn_saved_bytes(1 << 14, 256, 1 << 8, 128) > 0  # 2^30: the largest allowed
    assert L.lr_attn_saved_bytes(1, 1 << 16, 1 << 9, 128) == 0  # b*H*s*s = 2^41
    # tokens b*s and channels H*dh bounded before anything forms them in int
    assert L.lr_attn_saved_bytes(1 << 16, 512, 1, 128) == 0  # b*s = 2^25 tokens
    assert L.lr_attn_saved_bytes(1 << 15, 512, 1, 128) > 0  # 2^24: the largest allowed
    assert L.lr_attn_workspace_bytes(1, 256, 1 << 20, 4096) == 0  # H*dh = 2^32 would wrap an int
    assert L.lr_attn_saved_bytes(1, 256, 1 << 17, 128) > 0  # H*dh = 2^24: the largest allowed
    assert L.lr_attn_saved_bytes(1, 256, (1 << 17) + 1, 128) == 0  # one head more
    lib = L.lib()
    null = None
    assert lib.lr_attn_fwd(L.LR_F32, 1, 256, 1, 128, 1.0, null, null, null, null, null, 0, null, 0, null) == 8
    assert lib.lr_attn_fwd(L.LR_BF16, 1, 100, 1, 128, 1.0, null, null, null, null, null, 0, null, 0, null) == 2
    assert lib.lr_attn_fwd(L.LR_BF16, 1, 256, 1, 128, 1.0, null, null, null, null, null, 0, null, 0, null) == 1


def test_block_shape_rules(L):
    dims = (1, 256, 2, 128, 344, 32, 48)
    assert L.lr_block_saved_bytes(*dims) > 4 * 256 * 256 * 2  # q, k, v, o at least
    assert L.lr_block_workspace_bytes(*dims) >= L.lr_attn_workspace_bytes(1, 256, 2, 128)
    assert L.lr_block_saved_bytes(1, 200, 2, 128, 344, 32, 48) == 0  # s not a multiple of 256
    assert L.lr_block_saved_bytes(1, 256, 2, 128, 343, 32, 48) == 0  # f not a multiple of 8
    assert L.lr_block_saved_bytes(1 << 16, 512, 1, 128, 344, 32, 48) == 0  # b*s = 2^25 tokens
    assert L.lr_block_workspace_bytes(1, 256, 1 << 20, 4096, 344, 32, 48) == 0  # H*dh = 2^32
    lib = L.lib()
    w, g = L.lr_block_weights(), L.lr_block_grads()
    assert lib.lr_block_fwd(L.LR_F32, *dims, 1e-6, None, ctypes.byref(w), None, None, 0, None, 0, None) == 8
    assert lib.lr_block_fwd(L.LR_BF16, *dims, 1e-6, None, ctypes.byref(w), None, None, 0, None, 0, None) == 1
    assert lib.lr_block_bwd(L.LR_BF16, *dims, 1e-6, None, ctypes.byref(w), None, 0, None, None, ctypes.byref(g),
                            None, 0, None) == 1
