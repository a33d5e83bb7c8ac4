"""Seeded synthetic inputs (weights, token ids, stand-in KV contents).

Both the GPU path and the CPU oracle get their inputs from here: the host
functions fill numpy arrays, the device functions fill torch CUDA tensors, and
the two implement one counter-based generator (splitmix64, defined in
include/mk_synth.h) independently; the tests check them bit for bit.  Nothing
in this module computes any part of the decoder.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

from .configs import (  # noqa: F401  (re-exported)
    TINY_D128,
    TINY_FFN6K,
    TINY_G8,
    TINY_LONGFF,
    TINY_MHA,
    TINY_WIDE,
    LAYER_TIDS,
    TID_EMBED,
    TID_FINAL_NORM,
    TID_LM_HEAD,
    WORKLOADS,
    ModelCfg,
    Workload,
    kv_tid,
    layer_shapes,
    layer_tid,
    token_tid,
    weight_bytes,
    with_random_gains,
)

_HERE = Path(__file__).resolve().parent
_ROOT = _HERE.parent
LIB_PATH = _HERE / "libmk_synth.so"
_SOURCES = [_HERE / "synth.c", _HERE / "synth_cuda.cu", _ROOT / "include" / "mk_synth.h"]
GAIN_STD = 0.1


def build(force: bool = False) -> Path:
    """Compile libmk_synth.so (host C + device CUDA) in-tree."""
    if not force and LIB_PATH.exists():
        mtime = LIB_PATH.stat().st_mtime
        if all(s.stat().st_mtime <= mtime for s in _SOURCES):
            return LIB_PATH
    bdir = _HERE / "_build"
    bdir.mkdir(exist_ok=True)
    inc = str(_ROOT / "include")
    obj_c = bdir / "synth.o"
    obj_cu = bdir / "synth_cuda.o"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-fopenmp", "-ffp-contract=off", "-std=c11", "-I", inc,
                           "-c", str(_HERE / "synth.c"), "-o", str(obj_c)])
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-Xcompiler", "-fPIC",
                           "-fmad=false", "-I", inc, "-c", str(_HERE / "synth_cuda.cu"), "-o", str(obj_cu)])
    tmp = LIB_PATH.with_suffix(".so.tmp")
    subprocess.check_call(["nvcc", "-shared", "-o", str(tmp), str(obj_c), str(obj_cu), "-lgomp", "-lcudart"])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(LIB_PATH))
        u64, i64, f32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        L.mk_synth_scale.restype = f32
        L.mk_synth_scale.argtypes = [ctypes.c_double]
        L.mk_synth_u64_host.argtypes = [u64, u64, u64, i64, vp]
        L.mk_synth_stream_host.argtypes = [u64, u64, i64, vp]
        L.mk_synth_normal_bf16_host.argtypes = [vp, i64, u64, u64, u64, f32, f32]
        L.mk_synth_normal_bf16_device.argtypes = [vp, i64, u64, u64, u64, f32, f32, vp]
        L.mk_synth_tokens_host.argtypes = [vp, i64, u64, u64, u64, ctypes.c_int32]
        L.mk_synth_kv_pages_device.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, u64, u64, f32, vp]
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def scale(sigma: float) -> float:
    return float(lib().mk_synth_scale(sigma))


def stream(state: int, i0: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _check(lib().mk_synth_stream_host(state, i0, n, out.ctypes.data), "mk_synth_stream_host")
    return out


def u64(seed: int, tid: int, i0: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _check(lib().mk_synth_u64_host(seed, tid, i0, n, out.ctypes.data), "mk_synth_u64_host")
    return out


def normal_bf16(shape, seed: int, tid: int, sigma: float, offset: float = 0.0, i0: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of the normal generator, host memory."""
    out = np.empty(shape, dtype=np.uint16)
    _check(lib().mk_synth_normal_bf16_host(out.ctypes.data, out.size, seed, tid, i0, scale(sigma), offset),
           "mk_synth_normal_bf16_host")
    return out


def tokens(n: int, seed: int, seq: int, vocab: int, i0: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _check(lib().mk_synth_tokens_host(out.ctypes.data, n, seed, token_tid(seq), i0, vocab), "mk_synth_tokens_host")
    return out


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- weights

def _gain_args(m: ModelCfg):
    # gains: exactly 1.0 (sigma 0 gives z = 0) or 1 + N(0, 0.1)
    return (GAIN_STD if m.random_gains else 0.0), 1.0


def host_layer_weights(m: ModelCfg, seed: int, layer: int) -> dict:
    out = {}
    for name, shape in layer_shapes(m).items():
        if name.endswith("norm"):
            sig, off = _gain_args(m)
            out[name] = normal_bf16(shape, seed, layer_tid(layer, name), sig, off)
        else:
            out[name] = normal_bf16(shape, seed, layer_tid(layer, name), m.weight_std)
    return out


def host_weights(m: ModelCfg, seed: int = 0) -> dict:
    """All weights as host bf16 bit arrays: {'embed','lm_head','final_norm','layers':[...]}."""
    emb = normal_bf16((m.vocab, m.hidden), seed, TID_EMBED, m.weight_std)
    lm = emb if m.tied_embeddings else normal_bf16((m.vocab, m.hidden), seed, TID_LM_HEAD, m.weight_std)
    sig, off = _gain_args(m)
    fin = normal_bf16((m.hidden,), seed, TID_FINAL_NORM, sig, off)
    layers = [host_layer_weights(m, seed, l) for l in range(m.n_layers)]
    return {"embed": emb, "lm_head": lm, "final_norm": fin, "layers": layers}


def _fill_device(t, seed: int, tid: int, sigma: float, offset: float = 0.0, stream=None) -> None:
    import torch

    assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check(lib().mk_synth_normal_bf16_device(t.data_ptr(), t.numel(), seed, tid, 0, scale(sigma), offset, s),
           "mk_synth_normal_bf16_device")


def device_weights(m: ModelCfg, seed: int = 0, device: str = "cuda") -> dict:
    """All weights as torch bf16 CUDA tensors, filled on the device."""
    import torch

    def new(shape, tid, sigma, offset=0.0):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        _fill_device(t, seed, tid, sigma, offset)
        return t

    sig, off = _gain_args(m)
    emb = new((m.vocab, m.hidden), TID_EMBED, m.weight_std)
    lm = emb if m.tied_embeddings else new((m.vocab, m.hidden), TID_LM_HEAD, m.weight_std)
    fin = new((m.hidden,), TID_FINAL_NORM, sig, off)
    layers = []
    for l in range(m.n_layers):
        lw = {}
        for name, shape in layer_shapes(m).items():
            if name.endswith("norm"):
                lw[name] = new(shape, layer_tid(l, name), sig, off)
            else:
                lw[name] = new(shape, layer_tid(l, name), m.weight_std)
        layers.append(lw)
    return {"embed": emb, "lm_head": lm, "final_norm": fin, "layers": layers}


# ------------------------------------------------------- stand-in KV cache

def kv_sigma(m: ModelCfg) -> float:
    """Std of the stand-in K/V values: that of W x-hat for x-hat of unit RMS."""
    return m.weight_std * (m.hidden ** 0.5)


def host_kv(m: ModelCfg, seed: int, layer: int, which: str, batch: int, ctx: int) -> np.ndarray:
    """Logical stand-in cache [batch][ctx][n_kv_heads][head_dim] (bf16 bits)."""
    return normal_bf16((batch, ctx, m.n_kv_heads, m.head_dim), seed, kv_tid(layer, which), kv_sigma(m))


def device_kv_pages(pool_layer, page_table, m: ModelCfg, seed: int, layer: int, which: str, batch: int,
                    max_pages: int, ctx: int, page_size: int) -> None:
    import torch

    s = torch.cuda.current_stream().cuda_stream
    _check(lib().mk_synth_kv_pages_device(pool_layer.data_ptr(), page_table.data_ptr(), batch, max_pages, ctx,
                                          m.n_kv_heads, page_size, m.head_dim, seed, kv_tid(layer, which),
                                          scale(kv_sigma(m)), s), "mk_synth_kv_pages_device")
