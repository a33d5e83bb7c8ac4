"""fp64 CPU oracle of the Llama-style decode step (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The GPU
library neither imports nor links it, and it neither imports nor links the
GPU library: the two share only the seeded inputs from ``synth``.

Every function cites, in oracle.c, the page passage it follows.  Parity is
pinned by the tests in tests/test_oracle_pins.py (closed forms, invariants,
brute force on tiny inputs, special cases of the whole decoder); the end-to-end
logits of the random-init models have no printed value on the pages and are
pinned only through those properties.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_DEFAULT_LIB = _HERE / "liboracle.so"
# The mutation tests point this at deliberately broken builds of oracle.c.
LIB_PATH = Path(os.environ.get("MK_ORACLE_LIB", str(_DEFAULT_LIB)))

_i, _d, _p = ctypes.c_int, ctypes.c_double, ctypes.c_void_p


def compile_source(src: Path, out: Path) -> Path:
    tmp = out.with_suffix(".so.tmp")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
                           str(src), "-o", str(tmp), "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> Path:
    if LIB_PATH != _DEFAULT_LIB:
        return LIB_PATH
    src = _HERE / "oracle.c"
    if not force and LIB_PATH.exists() and src.stat().st_mtime <= LIB_PATH.stat().st_mtime:
        return LIB_PATH
    return compile_source(src, LIB_PATH)


class _Cfg(ctypes.Structure):
    _fields_ = [("n_layers", _i), ("hidden", _i), ("n_q_heads", _i), ("n_kv_heads", _i), ("head_dim", _i),
                ("ffn_dim", _i), ("vocab", _i), ("rms_eps", _d), ("rope_theta", _d), ("kv_bf16", _i)]


class _LayerW(ctypes.Structure):
    _fields_ = [(n, _p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _p), ("lm_head", _p), ("final_norm", _p), ("layers", ctypes.POINTER(_LayerW))]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(LIB_PATH))
        L.orc_num_threads.restype = _i
        L.orc_num_threads.argtypes = []
        L.orc_set_num_threads.restype = None
        L.orc_set_num_threads.argtypes = [_i]
        L.orc_bf16.restype = _d
        L.orc_bf16.argtypes = [ctypes.c_uint16]
        L.orc_round_bf16.restype = _d
        L.orc_round_bf16.argtypes = [_d]
        L.orc_rmsnorm.argtypes = [_i, _p, _p, _d, _p]
        L.orc_matvec.argtypes = [_i, _i, _p, _p, _p]
        L.orc_rope.argtypes = [_i, _p, _i, _d]
        L.orc_silu.restype = _d
        L.orc_silu.argtypes = [_d]
        L.orc_attention_head.argtypes = [_i, _i, _p, _p, _p, _i, _p]
        L.orc_layer_step.argtypes = [_p, _p, _p, _p, _i, _i, _p]
        L.orc_embed.argtypes = [_p, _p, _i, _p]
        L.orc_head.argtypes = [_p, _p, _p, _p, _p]
        L.orc_decode_step.argtypes = [_p, _p, _p, _p, _i, _i, _i, _p]
        L.orc_full_forward.argtypes = [_p, _p, _i, _p, _p]
        _lib = L
    return _lib


def num_threads() -> int:
    """Threads the oracle's parallel loops run with in this process."""
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's later parallel loops (timing runs only)."""
    lib().orc_set_num_threads(int(n))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "weights are bf16 bit patterns (uint16)"
    return a


# ------------------------------------------------------------- components

def rmsnorm(x, g_bits, eps: float) -> np.ndarray:
    x, g = _f64(x), _u16(g_bits)
    y = np.empty_like(x)
    lib().orc_rmsnorm(x.size, x.ctypes.data, g.ctypes.data, eps, y.ctypes.data)
    return y


def matvec(w_bits, x) -> np.ndarray:
    w, x = _u16(w_bits), _f64(x)
    y = np.empty(w.shape[0], dtype=np.float64)
    lib().orc_matvec(w.shape[0], w.shape[1], w.ctypes.data, x.ctypes.data, y.ctypes.data)
    return y


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = _f64(v).copy()
    lib().orc_rope(v.size, v.ctypes.data, pos, theta)
    return v


def silu(z: float) -> float:
    return float(lib().orc_silu(z))


def attention_head(q, K, V) -> np.ndarray:
    """q[d], K/V[C][d] -> out[d]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    out = np.empty(q.size, dtype=np.float64)
    lib().orc_attention_head(K.shape[0], q.size, q.ctypes.data, K.ctypes.data, V.ctypes.data, q.size,
                             out.ctypes.data)
    return out


def bf16_value(bits: int) -> float:
    return float(lib().orc_bf16(bits))


def round_bf16(x: float) -> float:
    """The bf16 value nearest to x (ties to even)."""
    return float(lib().orc_round_bf16(float(x)))


# ---------------------------------------------------------------- decoder

class Model:
    """A decoder shape plus host bf16 weights, laid out for oracle.c.

    ``weights`` is the dict of ``synth.host_weights``.  For models too large
    for host memory, build with ``layers=None`` and drive ``layer_step`` with
    per-layer weights instead.  ``kv_bf16``: the cache stores every appended
    key and value rounded to the nearest bf16 (a bf16 KV cache); otherwise it
    keeps them in fp64.
    """

    def __init__(self, cfg, weights: dict, kv_bf16: bool = False):
        self.cfg = cfg
        self.kv_bf16 = bool(kv_bf16)
        self._c = _Cfg(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                       cfg.vocab, cfg.rms_eps, cfg.rope_theta, int(kv_bf16))
        self._keep = []
        self.embed = _u16(weights["embed"])
        self.lm_head = _u16(weights["lm_head"])
        self.final_norm = _u16(weights["final_norm"])
        layers = weights.get("layers")
        self._w = None
        if layers is not None:
            arr = (_LayerW * cfg.n_layers)()
            for l, lw in enumerate(layers):
                arr[l] = self._layer_struct(lw, self._keep)
            self._layers = arr
            self._w = _Weights(self.embed.ctypes.data, self.lm_head.ctypes.data, self.final_norm.ctypes.data, arr)

    @staticmethod
    def _layer_struct(lw: dict, keep: list) -> _LayerW:
        vals = []
        for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"):
            a = _u16(lw[n])
            keep.append(a)
            vals.append(a.ctypes.data)
        return _LayerW(*vals)

    def new_cache(self, max_seq: int):
        c = self.cfg
        shape = (c.n_layers, max_seq, c.n_kv_heads, c.head_dim)
        return np.zeros(shape, dtype=np.float64), np.zeros(shape, dtype=np.float64)

    def decode_step(self, kcache, vcache, token: int, pos: int) -> np.ndarray:
        assert self._w is not None
        assert kcache.flags.c_contiguous and kcache.dtype == np.float64 and kcache.shape == vcache.shape
        logits = np.empty(self.cfg.vocab, dtype=np.float64)
        rc = lib().orc_decode_step(ctypes.byref(self._c), ctypes.byref(self._w), kcache.ctypes.data,
                                   vcache.ctypes.data, kcache.shape[1], int(token), int(pos), logits.ctypes.data)
        if rc != 0:
            raise ValueError(f"orc_decode_step rejected token={token} pos={pos}")
        return logits

    def prefill(self, kcache, vcache, tokens) -> np.ndarray:
        """Decode steps at positions 0..n-1; returns the logits of the last."""
        logits = None
        for p, t in enumerate(tokens):
            logits = self.decode_step(kcache, vcache, int(t), p)
        return logits

    def full_forward(self, tokens) -> np.ndarray:
        assert self._w is not None
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty((toks.size, self.cfg.vocab), dtype=np.float64)
        rc = lib().orc_full_forward(ctypes.byref(self._c), ctypes.byref(self._w), toks.size, toks.ctypes.data,
                                    out.ctypes.data)
        if rc != 0:
            raise ValueError("orc_full_forward rejected its input")
        return out

    # layer-wise driving (weights supplied per layer)
    def embed_token(self, token: int) -> np.ndarray:
        x = np.empty(self.cfg.hidden, dtype=np.float64)
        if lib().orc_embed(ctypes.byref(self._c), self.embed.ctypes.data, int(token), x.ctypes.data) != 0:
            raise ValueError("token out of range")
        return x

    def layer_step(self, layer_weights: dict, kc_layer, vc_layer, pos: int, x) -> None:
        """x (float64[hidden]) updated in place; kc/vc_layer [max_seq][nkv][d]."""
        keep: list = []
        st = self._layer_struct(layer_weights, keep)
        assert x.dtype == np.float64 and x.flags.c_contiguous
        assert kc_layer.flags.c_contiguous and kc_layer.dtype == np.float64
        rc = lib().orc_layer_step(ctypes.byref(self._c), ctypes.byref(st), kc_layer.ctypes.data,
                                  vc_layer.ctypes.data, kc_layer.shape[0], int(pos), x.ctypes.data)
        if rc != 0:
            raise ValueError("orc_layer_step rejected its input")

    def head(self, x) -> np.ndarray:
        logits = np.empty(self.cfg.vocab, dtype=np.float64)
        lib().orc_head(ctypes.byref(self._c), self.final_norm.ctypes.data, self.lm_head.ctypes.data,
                       _f64(x).ctypes.data, logits.ctypes.data)
        return logits
