"""Python binding of the persistent decode megakernel (libmk.so, C ABI in include/mk.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libmk.so.  The functions below carry the C names; ``Plan`` is a
small convenience holder that keeps torch tensors (device memory) alive for
the plan's lifetime.  There is no CPU fallback: if libmk.so cannot be built or
loaded, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes

from .build import LIB, build

MK_OK, MK_ERR_INVALID, MK_ERR_CUDA, MK_ERR_LAUNCH, MK_ERR_TIMEOUT, MK_ERR_BOUNDS, MK_ERR_OOM, MK_ERR_UNSUPPORTED = range(8)
OP_QKV, OP_ATTN, OP_O, OP_GU, OP_DOWN, OP_LM, OP_EMBED, OP_KVA = range(1, 9)
TC_TILE_M, TC_TILE_K = 128, 64  # batched path: weight rows x columns per unit

_i32, _f32, _vp = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class mk_model_cfg(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("hidden", _i32), ("n_q_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("ffn_dim", _i32), ("vocab", _i32), ("rms_eps", _f32), ("rope_theta", _f32),
                ("tied_embeddings", _i32), ("batch", _i32), ("max_seq", _i32), ("page_size", _i32)]


_PP = ctypes.POINTER(_vp)


class mk_weight_ptrs(ctypes.Structure):
    _fields_ = [("embed", _vp), ("lm_head", _vp), ("final_norm", _vp), ("attn_norm", _PP), ("wq", _PP),
                ("wk", _PP), ("wv", _PP), ("wo", _PP), ("mlp_norm", _PP), ("w_gate", _PP), ("w_up", _PP),
                ("w_down", _PP)]


class mk_kv_cache(ctypes.Structure):
    _fields_ = [("k_pool", _vp), ("v_pool", _vp), ("page_table", _vp), ("num_pages", _i32),
                ("max_pages_per_seq", _i32)]


class mk_plan_options(ctypes.Structure):
    _fields_ = [("num_ctas", _i32), ("attn_splits", _i32), ("slot_bytes", _i32), ("num_slots", _i32),
                ("timeout_ms", _i32), ("planner_seed", ctypes.c_uint32), ("l2_prefetch_kb", _i32),
                ("test_unreachable_event", _i32), ("trace", _i32), ("tensor_cores", _i32), ("max_inflight", _i32),
                ("kv_append", _i32), ("prefill_by_decode", _i32), ("jit", _i32),
                ("test_poison_scratch", _i32), ("tc_tile_split", _i32), ("tc_k_subtiles", _i32),
                ("reserved", _i32 * 1)]


class mk_device_error(ctypes.Structure):
    _fields_ = [("status", _i32), ("site", _i32), ("cta", _i32), ("detail", _i32)]


class mk_task_info(ctypes.Structure):
    _fields_ = [(n, _i32) for n in ("cta", "op", "layer", "wait_event", "wait_count", "signal_event", "a0", "a1",
                                    "a2", "a3")]


_lib = None
EXPORTS = ("mk_plan_create", "mk_plan_create_ex", "mk_decode_step", "mk_decode_step_ablation",
           "mk_decode_step_host", "mk_decode_step_greedy_host", "mk_prefill", "mk_prefill_row", "mk_greedy_next", "mk_plan_last_error",
           "mk_status_string", "mk_error_site_string", "mk_plan_destroy", "mk_plan_describe", "mk_plan_trace",
           "mk_decode_step_noalloc", "mk_decode_step_greedy", "mk_pages_create", "mk_pages_admit",
           "mk_pages_extend", "mk_pages_retire", "mk_pages_free_count", "mk_pages_scratch_page", "mk_pages_table",
           "mk_pages_sync", "mk_pages_destroy")


def lib():
    """Loads libmk.so (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(LIB))
        P = ctypes.POINTER
        L.mk_plan_create.argtypes = [P(mk_model_cfg), P(mk_weight_ptrs), P(_vp)]
        L.mk_plan_create_ex.argtypes = [P(mk_model_cfg), P(mk_weight_ptrs), P(mk_plan_options), P(_vp)]
        step = [_vp, _vp, _vp, P(mk_kv_cache), _vp, _vp]
        L.mk_decode_step.argtypes = step
        L.mk_decode_step_ablation.argtypes = step
        L.mk_decode_step_greedy.argtypes = step
        L.mk_decode_step_host.argtypes = step
        L.mk_decode_step_greedy_host.argtypes = step
        L.mk_prefill.argtypes = [_vp, _vp, _i32, P(mk_kv_cache), _vp, _vp]
        L.mk_greedy_next.argtypes = [_vp, _vp, _vp, _vp, _vp]
        L.mk_plan_last_error.argtypes = [_vp, _vp, P(mk_device_error)]
        L.mk_status_string.restype = ctypes.c_char_p
        L.mk_status_string.argtypes = [ctypes.c_int]
        L.mk_error_site_string.restype = ctypes.c_char_p
        L.mk_error_site_string.argtypes = [_i32]
        L.mk_plan_destroy.argtypes = [_vp]
        L.mk_plan_destroy.restype = None
        L.mk_plan_describe.argtypes = [P(mk_model_cfg), P(mk_plan_options), _i32, P(mk_task_info), _i32,
                                       P(_i32), P(_i32)]
        L.mk_plan_trace.argtypes = [_vp, _vp, _vp, ctypes.c_int64, P(_i32), P(_i32)]
        L.mk_decode_step_noalloc.argtypes = [P(mk_model_cfg), P(mk_weight_ptrs), _vp, _vp, P(mk_kv_cache), _vp, _vp]
        L.mk_prefill_row.argtypes = [_vp, _i32, _vp, _i32, P(mk_kv_cache), _vp, _vp]
        L.mk_pages_create.argtypes = [_i32, _i32, _i32, _i32, P(_vp)]
        L.mk_pages_admit.argtypes = [_vp, _i32, _i32]
        L.mk_pages_extend.argtypes = [_vp, _i32, _i32]
        L.mk_pages_retire.argtypes = [_vp, _i32]
        L.mk_pages_free_count.argtypes = [_vp]
        L.mk_pages_scratch_page.argtypes = [_vp]
        L.mk_pages_table.argtypes = [_vp, _vp, ctypes.c_int64]
        L.mk_pages_sync.argtypes = [_vp, _vp, _vp]
        L.mk_pages_destroy.argtypes = [_vp]
        L.mk_pages_destroy.restype = None
        for n in EXPORTS:
            if n not in ("mk_plan_destroy", "mk_status_string", "mk_error_site_string", "mk_pages_destroy"):
                getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


class MKError(RuntimeError):
    def __init__(self, status: int, what: str, info: "mk_device_error | None" = None):
        msg = f"{what}: {mk_status_string(status)} ({status})"
        if info is not None and info.status:
            msg += f" at {lib().mk_error_site_string(info.site).decode()} (cta {info.cta}, detail {info.detail})"
        super().__init__(msg)
        self.status = status
        self.info = info


def mk_status_string(status: int) -> str:
    return lib().mk_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != MK_OK:
        raise MKError(status, what)


def model_cfg(m, batch: int, max_seq: int, page_size: int = 64) -> mk_model_cfg:
    """mk_model_cfg from a synth.configs.ModelCfg-like object."""
    return mk_model_cfg(m.n_layers, m.hidden, m.n_q_heads, m.n_kv_heads, m.head_dim, m.ffn_dim, m.vocab,
                        m.rms_eps, m.rope_theta, int(m.tied_embeddings), batch, max_seq, page_size)


def _stream_ptr(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def mk_plan_describe(cfg: mk_model_cfg, num_ctas: int, opts: "mk_plan_options | None" = None):
    """Host-only task graph: (list of mk_task_info, n_events)."""
    n, ne = _i32(0), _i32(0)
    po = ctypes.byref(opts) if opts is not None else None
    st = lib().mk_plan_describe(ctypes.byref(cfg), po, num_ctas, None, 0, ctypes.byref(n), ctypes.byref(ne))
    if st not in (MK_OK, MK_ERR_INVALID) or n.value <= 0:
        _check(st, "mk_plan_describe")
    arr = (mk_task_info * max(1, n.value))()
    _check(lib().mk_plan_describe(ctypes.byref(cfg), po, num_ctas, arr, n.value, ctypes.byref(n), ctypes.byref(ne)),
           "mk_plan_describe")
    return list(arr)[: n.value], ne.value


class KVCache:
    """Paged bf16 KV cache in device memory (torch tensors) + its descriptor."""

    def __init__(self, m, batch: int, max_seq: int, page_size: int = 64, num_pages: int | None = None,
                 shuffle_seed: int | None = None, device="cuda"):
        import torch

        self.page_size = page_size
        self.max_pages = (max_seq + page_size - 1) // page_size
        self.num_pages = num_pages or batch * self.max_pages
        shape = (m.n_layers, self.num_pages, m.n_kv_heads, page_size, m.head_dim)
        self.k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        ids = torch.arange(batch * self.max_pages, dtype=torch.int32)
        if shuffle_seed is not None:
            g = torch.Generator().manual_seed(shuffle_seed)
            ids = ids[torch.randperm(ids.numel(), generator=g)]
        self.page_table = ids.view(batch, self.max_pages).contiguous().to(device)
        self.desc = mk_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.page_table.data_ptr(), self.num_pages,
                                self.max_pages)


class PagePool:
    """Host-side allocator of a KV pool's pages and of the batch's page table
    (mk_pages_* in include/mk.h): rows are admitted, extended and retired
    between decode steps; sync() copies the table to the device."""

    def __init__(self, num_pages: int, batch: int, max_pages: int, page_size: int = 64):
        self.batch, self.max_pages = batch, max_pages
        h = _vp()
        _check(lib().mk_pages_create(num_pages, batch, max_pages, page_size, ctypes.byref(h)), "mk_pages_create")
        self.h = h

    def admit(self, row: int, n_tokens: int) -> int:
        return lib().mk_pages_admit(self.h, row, n_tokens)

    def extend(self, row: int, n_tokens: int) -> int:
        return lib().mk_pages_extend(self.h, row, n_tokens)

    def retire(self, row: int) -> int:
        return lib().mk_pages_retire(self.h, row)

    @property
    def free_count(self) -> int:
        return int(lib().mk_pages_free_count(self.h))

    @property
    def scratch_page(self) -> int:
        return int(lib().mk_pages_scratch_page(self.h))

    def table(self):
        import numpy as np

        out = np.empty((self.batch, self.max_pages), dtype=np.int32)
        _check(lib().mk_pages_table(self.h, out.ctypes.data, out.size), "mk_pages_table")
        return out

    def sync(self, page_table_dev, stream=None) -> None:
        _check(lib().mk_pages_sync(self.h, page_table_dev.data_ptr(), _stream_ptr(stream)), "mk_pages_sync")

    def close(self):
        if self.h:
            lib().mk_pages_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Plan:
    """Owns an mk_plan plus references to the weight tensors it points at."""

    def __init__(self, m, weights: dict, batch: int, max_seq: int, page_size: int = 64,
                 opts: "mk_plan_options | None" = None):
        self.m = m
        self.cfg = model_cfg(m, batch, max_seq, page_size)
        self.batch, self.max_seq = batch, max_seq
        self._weights = weights
        L = m.n_layers
        names = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")
        self._arrs = {k: (_vp * L)(*[weights["layers"][l][k].data_ptr() for l in range(L)]) for k in names}
        self.wp = mk_weight_ptrs(weights["embed"].data_ptr(), weights["lm_head"].data_ptr(),
                                 weights["final_norm"].data_ptr(),
                                 *[ctypes.cast(self._arrs[k], _PP) for k in names])
        h = _vp()
        if opts is None:
            st = lib().mk_plan_create(ctypes.byref(self.cfg), ctypes.byref(self.wp), ctypes.byref(h))
        else:
            st = lib().mk_plan_create_ex(ctypes.byref(self.cfg), ctypes.byref(self.wp), ctypes.byref(opts),
                                         ctypes.byref(h))
        _check(st, "mk_plan_create")
        self.h = h

    def close(self):
        if self.h:
            lib().mk_plan_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # thin wrappers: torch tensors in, status checked
    def decode_step(self, tokens, positions, kv: KVCache, logits, stream=None):
        _check(lib().mk_decode_step(self.h, tokens.data_ptr(), positions.data_ptr(), ctypes.byref(kv.desc),
                                    logits.data_ptr(), _stream_ptr(stream)), "mk_decode_step")

    def decode_step_greedy(self, tokens, positions, kv: KVCache, logits, stream=None):
        """A decode step, then tokens = argmax(logits), positions += 1 in place."""
        _check(lib().mk_decode_step_greedy(self.h, tokens.data_ptr(), positions.data_ptr(), ctypes.byref(kv.desc),
                                           logits.data_ptr(), _stream_ptr(stream)), "mk_decode_step_greedy")

    def decode_step_ablation(self, tokens, positions, kv: KVCache, logits, stream=None):
        _check(lib().mk_decode_step_ablation(self.h, tokens.data_ptr(), positions.data_ptr(), ctypes.byref(kv.desc),
                                             logits.data_ptr(), _stream_ptr(stream)), "mk_decode_step_ablation")

    def decode_step_host(self, tokens_host, positions_host, kv: KVCache, logits_host, stream=None):
        """numpy (or pinned torch CPU) buffers; synchronises; raises on device errors."""
        ptr = lambda a: a.ctypes.data if hasattr(a, "ctypes") else a.data_ptr()
        st = lib().mk_decode_step_host(self.h, ptr(tokens_host), ptr(positions_host), ctypes.byref(kv.desc),
                                       ptr(logits_host), _stream_ptr(stream))
        _check(st, "mk_decode_step_host")

    def decode_step_greedy_host(self, tokens_host, positions_host, kv: KVCache, next_tokens_host, stream=None):
        """Host int32 buffers: tokens and positions in, the step's greedy picks out; synchronises."""
        ptr = lambda a: a.ctypes.data if hasattr(a, "ctypes") else a.data_ptr()
        st = lib().mk_decode_step_greedy_host(self.h, ptr(tokens_host), ptr(positions_host), ctypes.byref(kv.desc),
                                              ptr(next_tokens_host), _stream_ptr(stream))
        _check(st, "mk_decode_step_greedy_host")

    def prefill(self, tokens, kv: KVCache, last_logits, stream=None):
        T = tokens.shape[-1]
        _check(lib().mk_prefill(self.h, tokens.data_ptr(), T, ctypes.byref(kv.desc), last_logits.data_ptr(),
                                _stream_ptr(stream)), "mk_prefill")

    def prefill_row(self, row: int, tokens, kv: KVCache, logits, stream=None):
        """Prefill one batch row's prompt (device int32 [T]) into its pages; logits: device fp32 [vocab]."""
        T = tokens.shape[-1]
        _check(lib().mk_prefill_row(self.h, row, tokens.data_ptr(), T, ctypes.byref(kv.desc), logits.data_ptr(),
                                    _stream_ptr(stream)), "mk_prefill_row")

    def greedy_next(self, logits, tokens, positions, stream=None):
        _check(lib().mk_greedy_next(self.h, logits.data_ptr(), tokens.data_ptr(), positions.data_ptr(),
                                    _stream_ptr(stream)), "mk_greedy_next")

    def last_error(self, stream=None) -> mk_device_error:
        info = mk_device_error()
        lib().mk_plan_last_error(self.h, _stream_ptr(stream), ctypes.byref(info))
        return info

    def trace(self, stream=None):
        """numpy uint64 [num_ctas][max_tasks][8] of the last step (plan built with trace=1)."""
        import numpy as np

        nc, mt = _i32(0), _i32(0)
        lib().mk_plan_trace(self.h, _stream_ptr(stream), None, 0, ctypes.byref(nc), ctypes.byref(mt))
        out = np.zeros((nc.value, mt.value, 8), dtype=np.uint64)
        _check(lib().mk_plan_trace(self.h, _stream_ptr(stream), out.ctypes.data, out.size, ctypes.byref(nc),
                                   ctypes.byref(mt)), "mk_plan_trace")
        return out

    def check(self, stream=None) -> None:
        info = self.last_error(stream)
        if info.status != MK_OK:
            raise MKError(info.status, "device", info)
