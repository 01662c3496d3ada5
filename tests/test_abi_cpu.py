"""The C-ABI library loads, exports every declared symbol, and validates on the host.

No compute call here touches a GPU: create/persistent_bytes/workspace_bytes/
strerror/path_for are host-only.
"""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from latent_moe_layer_gb300 import build, k3moe
    build.build()
    return k3moe.lib()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(k3moe_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    from latent_moe_layer_gb300 import k3moe
    declared = _declared()
    assert len(declared) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", k3moe.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (k3moe_\w+)", out))
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    for n in declared:
        getattr(lib, n)
    assert set(k3moe.EXPORTS) <= set(declared)


def _cfg(**kw):
    from latent_moe_layer_gb300 import k3moe, synth
    c = k3moe.make_config(synth.CONFIGS[1])
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _create(lib, cfg):
    h = C.c_void_p()
    rc = lib.k3moe_create(C.byref(cfg), C.byref(h))
    return rc, h


@pytest.mark.parametrize("field,value,code", [
    ("hidden", 7000, -2), ("latent", 3590, -2), ("inter", 3000, -2), ("n_experts", 0, -1),
    ("top_k", 0, -1), ("top_k", 33, -2), ("n_experts", 2048, -2), ("act", 5, -9),
    ("router_dtype", 7, -1), ("path", 9, -1), ("shared_inter", 6000, -2)])
def test_create_rejects_bad_configs(lib, field, value, code):
    rc, h = _create(lib, _cfg(**{field: value}))
    assert rc == code and not h.value


def test_create_and_sizes_k3(lib):
    from latent_moe_layer_gb300 import k3moe
    rc, h = _create(lib, _cfg())
    assert rc == 0 and h.value
    try:
        assert lib.k3moe_persistent_bytes(h) > 6 * 896 * 8
        w16 = lib.k3moe_workspace_bytes(h, 16)
        w256 = lib.k3moe_workspace_bytes(h, 256)
        assert 0 < w16 < w256
        assert lib.k3moe_workspace_bytes(h, 0) > 0
        assert lib.k3moe_path_for(h, 16) == k3moe.PATH_GENERIC   # nothing loaded yet
    finally:
        lib.k3moe_destroy(h)
    lib.k3moe_destroy(None)


def test_calls_out_of_order_are_rejected(lib):
    rc, h = _create(lib, _cfg())
    try:
        rc = lib.k3moe_forward(h, None, 4, None, None, None, None, 0, None)
        assert rc == -11                                  # STATE: no weights yet
        assert lib.k3moe_load_weights(h, None, None, 0, None) == -1
        assert lib.k3moe_status(h, None) == -11
    finally:
        lib.k3moe_destroy(h)


def test_strerror_names_every_code(lib):
    from latent_moe_layer_gb300 import k3moe
    for code in k3moe.ERR:
        s = lib.k3moe_strerror(code).decode()
        assert s and s != "unknown error"
    assert lib.k3moe_strerror(12345).decode() == "unknown error"


def test_debug_dequant_argument_checks(lib):
    assert lib.k3moe_debug_dequant(None, None, 1, 32, None, None) == -1
    one = C.c_void_p(16)
    assert lib.k3moe_debug_dequant(one, one, 1, 33, one, None) == -2


def test_ep_plan_argument_checks(lib):
    from latent_moe_layer_gb300 import k3moe
    rc, h = _create(lib, _cfg())
    try:
        one = C.c_void_p(16)
        plan = k3moe.EpPlan(16, 16, 16, 16, 16)
        empty = k3moe.EpPlan(16, 16, 16, None, 16)
        assert lib.k3moe_ep_plan_compute(h, None, 8, 16, C.byref(plan), None) == -1
        assert lib.k3moe_ep_plan_compute(h, one, 8, 16, C.byref(empty), None) == -1
        assert lib.k3moe_ep_plan_compute(h, one, 8, 16, C.byref(plan), None) == -11   # no weights: no status word
        assert lib.k3moe_ep_dispatch(h, one, 16, 0, one, 8, C.byref(plan), one, one, one, 1 << 20, None) == -11
        assert lib.k3moe_ep_dispatch(h, None, 16, 0, one, 8, C.byref(plan), one, one, one, 1 << 20, None) == -1
        # 896 experts, 16 tokens: 1 chunk of per-expert counts plus the bases and totals
        assert lib.k3moe_ep_dispatch_workspace_bytes(h, 16) >= 3 * 896 * 4
        assert lib.k3moe_ep_dispatch_workspace_bytes(h, 0) == 0
    finally:
        lib.k3moe_destroy(h)
