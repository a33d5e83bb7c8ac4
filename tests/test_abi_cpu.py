"""CPU checks of the C-ABI library: it builds, loads, exports every function
include/mk.h declares, and its host-only parts behave (no GPU needed)."""
import ctypes
import re
import subprocess
from pathlib import Path

import pytest

import persistent_decode_megakernel_04_b300 as mk
import synth

ROOT = Path(__file__).resolve().parent.parent


def _declared(header: str):
    text = (ROOT / "include" / header).read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(mk_\w+)\s*\(", text, flags=re.M)))


def _exported(lib: Path):
    out = subprocess.run(["nm", "-D", "--defined-only", str(lib)], capture_output=True, text=True, check=True).stdout
    return {l.split()[-1] for l in out.splitlines() if l.strip()}


def test_libmk_exports_every_declared_function():
    mk.lib()
    names = _declared("mk.h")
    assert "mk_decode_step" in names and "mk_plan_create" in names and len(names) >= 12
    exported = _exported(mk.LIB)
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared in mk.h but not exported: {missing}"
    for n in names:
        getattr(mk.lib(), n)


def test_libmk_synth_exports_every_declared_function():
    synth.lib()
    names = _declared("mk_synth.h")
    exported = _exported(synth.LIB_PATH)
    assert names and not [n for n in names if n not in exported]


def test_status_strings():
    for s in range(8):
        assert mk.mk_status_string(s)
    assert "unknown" in mk.mk_status_string(99)
    assert mk.lib().mk_error_site_string(1)


def test_plan_create_rejects_null_and_bad_shapes_without_gpu():
    h = ctypes.c_void_p()
    assert mk.lib().mk_plan_create(None, None, ctypes.byref(h)) == mk.MK_ERR_INVALID
    bad = mk.model_cfg(synth.WORKLOADS["tiny"].model, 1, 64)
    bad.n_q_heads = 3  # not a multiple of n_kv_heads
    wp = mk.mk_weight_ptrs()
    assert mk.lib().mk_plan_create(ctypes.byref(bad), ctypes.byref(wp), ctypes.byref(h)) == mk.MK_ERR_INVALID
    good = mk.model_cfg(synth.WORKLOADS["tiny"].model, 1, 64)
    # null weight pointers are rejected before any CUDA call
    assert mk.lib().mk_plan_create(ctypes.byref(good), ctypes.byref(wp), ctypes.byref(h)) == mk.MK_ERR_INVALID
    assert not h.value


def test_unsupported_shapes_are_reported():
    c = mk.model_cfg(synth.WORKLOADS["tiny"].model, 1, 64)
    c.head_dim = 48
    with pytest.raises(mk.MKError) as e:
        mk.mk_plan_describe(c, 148)
    assert e.value.status == mk.MK_ERR_UNSUPPORTED


def test_null_step_arguments_rejected():
    assert mk.lib().mk_decode_step(None, None, None, None, None, None) == mk.MK_ERR_INVALID
    for fn in ("mk_decode_step_greedy", "mk_decode_step_host", "mk_decode_step_greedy_host",
               "mk_decode_step_ablation"):
        assert getattr(mk.lib(), fn)(None, None, None, None, None, None) == mk.MK_ERR_INVALID, fn
    assert mk.lib().mk_prefill(None, None, 4, None, None, None) == mk.MK_ERR_INVALID
    assert mk.lib().mk_prefill_row(None, 0, None, 4, None, None, None) == mk.MK_ERR_INVALID
    assert mk.lib().mk_greedy_next(None, None, None, None, None) == mk.MK_ERR_INVALID


def test_plan_options_layout_matches_the_header():
    """The binding's options struct has the header's fields in order (the
    header's field names, read from mk.h, against the ctypes fields)."""
    text = (ROOT / "include" / "mk.h").read_text()
    body = text[text.index("typedef struct {\n    int32_t num_ctas;"):text.index("} mk_plan_options;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"\b(?:int32_t|uint32_t)\s+(\w+)", body)
    assert [n for n, _ in mk.mk_plan_options._fields_] == names
    assert ctypes.sizeof(mk.mk_plan_options) == 4 * (len(names) - 1 + 1)  # reserved[1] is one word


@pytest.mark.parametrize("bad", [dict(tc_k_subtiles=3), dict(tc_k_subtiles=-1), dict(num_slots=1), dict(jit=17)])
def test_out_of_range_options_rejected_on_host(bad):
    c = mk.model_cfg(synth.WORKLOADS["tiny"].model, 8, 64)
    with pytest.raises(mk.MKError) as e:
        mk.mk_plan_describe(c, 148, mk.mk_plan_options(**bad))
    assert e.value.status == mk.MK_ERR_INVALID
