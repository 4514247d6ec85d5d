"""Host-only checks of the C ABI: the library loads, exports every symbol
include/h2o.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "h2o.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:h2o|lsh|sh|fg)_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from kv_cache_eviction_h2o_gb300 import build as b
    b.build()
    from kv_cache_eviction_h2o_gb300 import binding
    return binding


def test_header_declares_the_api():
    names = _declared()
    for must in ("h2o_init", "h2o_prefill", "h2o_decode_step", "lsh_decode_step", "lsh_init",
                 "lsh_prefill", "h2o_get_state", "h2o_set_state", "h2o_sync", "h2o_destroy",
                 "h2o_last_error", "h2o_init_gqa", "sh_init", "sh_prefill", "sh_decode_step",
                 "fg_init", "fg_prefill", "fg_decode_step", "fg_get_policy"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    lib = L.lib()
    for name in _declared():
        assert hasattr(lib, name), name
    # the binding wraps exactly the declared set
    assert set(L.SIGNATURES) == set(_declared())
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T ((?:h2o|lsh|sh|fg)_\w+)$", out, flags=re.M))
    assert set(_declared()) <= exported


def test_library_has_sm103a_code(L):
    # the fat binary is tagged with the architecture it was built for
    out = subprocess.run(["strings", L.LIB_PATH], capture_output=True, text=True).stdout
    assert "sm_103a" in out


@pytest.mark.parametrize("args,frag", [
    ((0, 0, 0, 1, 1, 128, 1, 0.1), "budget"),
    ((10, 5, 6, 1, 1, 128, 1, 0.1), "heavy + recent"),
    ((10, 5, 5, 1, 1, 96, 1, 0.1), "head_dim"),
    ((10, 5, 5, 1, 1, 128, 7, 0.1), "dtype"),
    ((10, 5, 5, 0, 1, 128, 1, 0.1), "batch"),
    ((10, 5, 5, 1, 1, 128, 1, -1.0), "scale"),
    ((10, 5, 11, 1, 1, 128, 1, 0.1), "recent"),
])
def test_init_rejects_bad_arguments(L, args, frag):
    with pytest.raises(L.H2OError) as e:
        L.h2o_init(*args)
    assert e.value.code == L.H2O_ERR_ARG
    assert frag in str(e.value)


def test_lsh_init_requires_projection(L):
    with pytest.raises(L.H2OError) as e:
        L.lsh_init(10, 5, 1, 1, 128, 1, 0.1, None)
    assert e.value.code == L.H2O_ERR_ARG


def test_null_handle_is_rejected(L):
    lib = L.lib()
    assert lib.h2o_prefill(None, None, None, None, 4) == L.H2O_ERR_ARG
    assert lib.h2o_decode_step(None, None, None, None, None, None) == L.H2O_ERR_ARG
    assert lib.lsh_decode_step(None, None, None, None, None, None) == L.H2O_ERR_ARG
    assert lib.h2o_sync(None) == L.H2O_ERR_ARG
    assert lib.h2o_get_state(None, None, None, None, None, None, None, None) == L.H2O_ERR_ARG
    assert lib.h2o_set_decode_split(None, 2) == L.H2O_ERR_ARG
    lib.h2o_destroy(None)          # no-op
    assert "NULL" in L.h2o_last_error()


def test_out_pointer_is_required(L):
    lib = L.lib()
    assert lib.h2o_init(None, 10, 5, 5, 1, 1, 128, 1, 0.1, None) == L.H2O_ERR_ARG


@pytest.mark.parametrize("groups,budget,frag", [
    (0, 64, "groups"),
    (17, 64, "groups"),
    (4, 1025, "1024 slots"),
])
def test_grouped_query_init_rejects_bad_groups(L, groups, budget, frag):
    with pytest.raises(L.H2OError) as e:
        L.h2o_init_gqa(budget, budget // 2, budget - budget // 2, 1, 2, groups, 128, 1, 0.1)
    assert e.value.code == L.H2O_ERR_ARG
    assert frag in str(e.value)


def test_persistence_rule_init_checks(L):
    with pytest.raises(L.H2OError) as e:
        L.sh_init(10, 5, 6, 1, 1, 128, 1, 0.1)          # heavy + recent != budget
    assert e.value.code == L.H2O_ERR_ARG
    for flag in (L.H2O_KV8, L.H2O_KV4):
        with pytest.raises(L.H2OError) as e:
            L.sh_init(10, 5, 5, 1, 1, 128, 1 | flag, 0.1)
        assert e.value.code == L.H2O_ERR_UNSUPPORTED
    lib = L.lib()
    assert lib.sh_prefill(None, None, None, None, 4) == L.H2O_ERR_ARG
    assert lib.sh_decode_step(None, None, None, None, None, None) == L.H2O_ERR_ARG
    assert lib.sh_init(None, 10, 5, 5, 1, 1, 128, 1, 0.1, None) == L.H2O_ERR_ARG


def test_binding_checks_host_buffers(L):
    import numpy as np
    # a handle shape recorded as the init call records it (no device needed:
    # every check below fails before the library is called)
    h = L._remember(0xDEAD0, "h2o", 4, 8, 64, L.H2O_BF16)
    try:
        with pytest.raises(TypeError, match="score"):
            L.h2o_get_state(h, score=np.empty(32, np.float32))
        with pytest.raises(ValueError, match="pos"):
            L.h2o_get_state(h, pos=np.empty(31, np.int32))
        with pytest.raises(TypeError, match="K"):
            L.h2o_set_state(h, K=np.empty(4 * 8 * 64, np.float32))      # bf16 rows are uint16 on the host
        with pytest.raises(ValueError, match="occupancy"):
            L.h2o_set_state(h, occupancy=np.empty(5, np.int32))
        with pytest.raises(ValueError, match="kscale"):
            L.h2o_get_kv_scales(h, np.empty(31, np.float32))
        with pytest.raises(ValueError, match="c"):
            L.h2o_get_prefill_stats(h, c=np.empty(1))
        with pytest.raises(TypeError, match="numpy"):
            L.h2o_get_state(h, score=[0.0] * 32)
    finally:
        L._meta.pop(h, None)
    with pytest.raises(ValueError, match="unknown handle"):
        L.h2o_get_state(0xDEAD0, score=np.empty(32))


def test_per_head_policy_init_checks(L):
    lib = L.lib()
    for args, frag in (((10, 5, 6, 64, 0.95), "heavy + recent"), ((10, 5, 5, 0, 0.95), "full_budget"),
                       ((10, 5, 5, 64, 0.0), "tau"), ((10, 5, 5, 64, 1.5), "tau")):
        with pytest.raises(L.H2OError) as e:
            L.fg_init(*args, 1, 1, 128, 1, 0.1)
        assert e.value.code == L.H2O_ERR_ARG and frag in str(e.value)
    for flag in (L.H2O_KV8, L.H2O_KV4):
        with pytest.raises(L.H2OError) as e:
            L.fg_init(10, 5, 5, 64, 0.95, 1, 1, 128, 1 | flag, 0.1)
        assert e.value.code == L.H2O_ERR_UNSUPPORTED
    assert lib.fg_prefill(None, None, None, None, 4) == L.H2O_ERR_ARG
    assert lib.fg_decode_step(None, None, None, None, None, None) == L.H2O_ERR_ARG
    assert lib.fg_get_policy(None, None, None, None) == L.H2O_ERR_ARG


def test_quantised_flags_are_exclusive(L):
    for init in (lambda dt: L.h2o_init(8, 4, 4, 1, 2, 64, dt, 0.125),
                 lambda dt: L.lsh_init(8, 4, 1, 2, 64, dt, 0.125, None)):
        with pytest.raises(L.H2OError) as e:
            init(L.H2O_BF16 | L.H2O_KV8 | L.H2O_KV4)
        assert e.value.code == L.H2O_ERR_ARG and "H2O_KV4" in str(e.value)


def test_binding_sizes_4bit_rows(L):
    import numpy as np
    # a 4-bit handle's rows are d/2 bytes on the host
    h = L._remember(0xDEAD4, "h2o", 4, 8, 64, L.H2O_BF16 | L.H2O_KV4)
    try:
        with pytest.raises(ValueError, match="K"):
            L.h2o_get_state(h, K=np.empty(4 * 8 * 64, np.uint8))
        with pytest.raises(TypeError, match="V"):
            L.h2o_get_state(h, V=np.empty(4 * 8 * 32, np.int8))
    finally:
        L._meta.pop(h, None)
