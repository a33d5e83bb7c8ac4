"""The allocation-free decode step (mk_decode_step_noalloc) against the plan
path (mk_decode_step).

mk_decode_step_noalloc is for callers that cannot call cudaMalloc when they
need a decode step, for example code running while a memory pool or a CUDA
graph owns the device's allocations. Its scratch is one fixed array compiled
into the library, and every call reuses it. So this test makes two calls in a
row and checks each against the plan path on an identical KV cache. The
second call also checks that nothing left over from the first changes the
result. The file is named so that pytest collects it last. It builds
everything it uses itself, so it passes alone in a fresh process as well as
after the other tests.
"""
import ctypes

import numpy as np
import pytest

import persistent_decode_megakernel_04_b300 as mk
import synth
from synth import WORKLOADS
from tests import harness

pytestmark = pytest.mark.gpu


def test_noalloc_step_matches_plan_step_twice(cuda_device):
    import torch

    m = WORKLOADS["tiny"].model
    max_seq = 128
    plan, kv_ref = harness.gpu_plan(m, max_seq)
    kv_na = mk.KVCache(m, 1, max_seq, shuffle_seed=1)
    # identical caches: prefill one, copy it into the other
    prompt = torch.tensor(synth.tokens(37, 0, 11, m.vocab), dtype=torch.int32, device=cuda_device).view(1, -1)
    logits_ref = torch.empty((1, m.vocab), dtype=torch.float32, device=cuda_device)
    plan.prefill(prompt, kv_ref, logits_ref)
    plan.check()
    kv_na.k.copy_(kv_ref.k)
    kv_na.v.copy_(kv_ref.v)
    kv_na.page_table.copy_(kv_ref.page_table)
    torch.cuda.synchronize()

    logits_na = torch.empty_like(logits_ref)
    tok = torch.empty(1, dtype=torch.int32, device=cuda_device)
    pos = torch.tensor([37], dtype=torch.int32, device=cuda_device)
    tok.fill_(int(np.argmax(logits_ref.cpu().numpy()[0])))
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        plan.decode_step(tok, pos, kv_ref, logits_ref)
        plan.check()
        logits_na.fill_(float("nan"))
        st = mk.lib().mk_decode_step_noalloc(ctypes.byref(plan.cfg), ctypes.byref(plan.wp), tok.data_ptr(),
                                            pos.data_ptr(), ctypes.byref(kv_na.desc), logits_na.data_ptr(), stream)
        assert st == mk.MK_OK, f"call {call}: {mk.mk_status_string(st)}"
        got, ref = logits_na.cpu().numpy()[0], logits_ref.cpu().numpy()[0]
        harness.compare_logits(got, ref, f"no-alloc call {call} vs plan step")
        # the appended K/V of this position agree as well
        assert torch.equal(kv_na.k, kv_ref.k) and torch.equal(kv_na.v, kv_ref.v)
        tok.fill_(int(np.argmax(ref)))
        pos += 1


def test_noalloc_rejects_batched_and_oversized_shapes(cuda_device):
    import torch

    m = WORKLOADS["tiny"].model
    plan, kv = harness.gpu_plan(m, 64)
    logits = torch.empty((1, m.vocab), dtype=torch.float32, device=cuda_device)
    t = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    batched = mk.model_cfg(m, 2, 64)
    assert mk.lib().mk_decode_step_noalloc(ctypes.byref(batched), ctypes.byref(plan.wp), t.data_ptr(), t.data_ptr(),
                                           ctypes.byref(kv.desc), logits.data_ptr(), None) == mk.MK_ERR_UNSUPPORTED
    # a context whose RoPE table alone exceeds the fixed scratch
    huge = mk.model_cfg(m, 1, 1 << 20)
    big_kv = mk.mk_kv_cache(kv.desc.k_pool, kv.desc.v_pool, kv.desc.page_table, kv.desc.num_pages, (1 << 20) // 64)
    assert mk.lib().mk_decode_step_noalloc(ctypes.byref(huge), ctypes.byref(plan.wp), t.data_ptr(), t.data_ptr(),
                                           ctypes.byref(big_kv), logits.data_ptr(), None) == mk.MK_ERR_OOM


def test_noalloc_call_keeps_a_larger_plan_launchable(cuda_device):
    """The kernel's dynamic shared-memory limit is shared by every plan and
    call in the process.  A plan made with a larger ring than the
    allocation-free call uses must still launch after that call."""
    import torch

    m = WORKLOADS["tiny"].model
    max_seq = 128
    big, kv = harness.gpu_plan(m, max_seq, opts=mk.mk_plan_options(slot_bytes=33792))
    model = harness.oracle_model(m)
    prompt = synth.tokens(20, 0, 12, m.vocab)
    kc, vc = model.new_cache(max_seq)
    ref = model.prefill(kc, vc, prompt)
    logits = torch.empty((1, m.vocab), dtype=torch.float32, device=cuda_device)
    big.prefill(torch.tensor(prompt, dtype=torch.int32, device=cuda_device).view(1, -1), kv, logits)
    big.check()
    harness.compare_logits(logits.cpu().numpy()[0], ref, "larger-ring plan before the no-alloc call")
    # the allocation-free call (default ring, less shared memory), on a cache of its own
    kv_na = mk.KVCache(m, 1, max_seq, shuffle_seed=1)
    t = torch.tensor([int(np.argmax(ref))], dtype=torch.int32, device=cuda_device)
    p0 = torch.tensor([0], dtype=torch.int32, device=cuda_device)
    out = torch.empty_like(logits)
    st = mk.lib().mk_decode_step_noalloc(ctypes.byref(big.cfg), ctypes.byref(big.wp), t.data_ptr(), p0.data_ptr(),
                                        ctypes.byref(kv_na.desc), out.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert st == mk.MK_OK, mk.mk_status_string(st)
    # the larger plan's next step still launches and still matches the oracle
    nxt = int(np.argmax(ref))
    ref = model.decode_step(kc, vc, nxt, len(prompt))
    big.decode_step(t, torch.tensor([len(prompt)], dtype=torch.int32, device=cuda_device), kv, logits)
    big.check()
    harness.compare_logits(logits.cpu().numpy()[0], ref, "larger-ring plan after the no-alloc call")
