"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and validates arguments / injects host-side faults before touching a device."""
import ctypes
import os
import re

import pytest

import ftgen
import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def F():
    from expert_cache_host_softmax_b300 import build
    build.build()
    import expert_cache_host_softmax_b300 as F
    return F


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(ft_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(F):
    declared = _declared()
    assert len(declared) >= 15
    L = F.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(F.EXPORTED) == declared


def test_blob_bytes_agree_three_ways(F):
    for fmt in ("bf16", "nvfp4", "mxfp4"):
        for H, I in ((256, 512), (2048, 768), (7168, 2048), (6144, 2048)):
            lib = F.blob_bytes(fmt, H, I)
            assert lib == ftgen.blob_bytes(fmt, H, I) == O.blob_bytes(ftgen.FMT_NAMES[fmt], H, I)
    assert F.blob_bytes("bf16", 200, 512) == -1


def _create(F, *args):
    h = ctypes.c_void_p()
    rc = F.lib().ft_moe_create(*args, ctypes.byref(h))
    return rc, h


def test_create_validates_before_touching_a_device(F):
    ok = (2048, 128, 8, 768, 1, 1024, 48, 1)
    bad = [
        ((2000,) + ok[1:], F.FT_ERR_ARG),                 # hidden not a multiple of 256
        (ok[:1] + (0,) + ok[2:], F.FT_ERR_ARG),           # no experts
        (ok[:1] + (600,) + ok[2:], F.FT_ERR_ARG),         # more than 512 experts
        (ok[:2] + (0,) + ok[3:], F.FT_ERR_ARG),           # top_k 0
        (ok[:2] + (129,) + ok[3:], F.FT_ERR_ARG),         # top_k > E
        (ok[:4] + (4,) + ok[5:], F.FT_ERR_ARG),           # unknown format
        (ok[:5] + (7,) + ok[6:], F.FT_ERR_CACHE_TOO_SMALL),  # 7 slots < 8 experts of one call
        (ok[:7] + (0,), F.FT_ERR_ARG),                    # max_tokens 0
    ]
    for args, want in bad:
        rc, h = _create(F, *args)
        assert rc == want, (args, rc, F.lib().ft_last_error(None))
        assert not h.value
        assert F.lib().ft_last_error(None)


def test_injected_allocation_failure(F, monkeypatch):
    monkeypatch.setenv("FT_FAULT", "alloc")
    rc, h = _create(F, 2048, 128, 8, 768, 1, 1024, 48, 1)
    assert rc == F.FT_ERR_OOM and not h.value
    assert b"FT_FAULT=alloc" in F.lib().ft_last_error(None)


def test_null_handle_and_stateless_validation(F):
    L = F.lib()
    assert L.ft_moe_load_pool(None, None) == F.FT_ERR_ARG
    assert L.ft_moe_forward(None, 0, 1, None, None, None, None) == F.FT_ERR_ARG
    assert L.ft_cache_stats(None, None, None) == F.FT_ERR_ARG
    assert L.ft_cache_reset(None, 1) == F.FT_ERR_ARG
    assert L.ft_moe_set_mode(None, 0) == F.FT_ERR_ARG
    assert L.ft_moe_resize_slots(None, 8) == F.FT_ERR_ARG
    assert L.ft_moe_set_prefill_hit_d2d(None, 1) == F.FT_ERR_ARG
    assert L.ft_moe_prefill_hit_d2d(None) == F.FT_ERR_ARG
    assert L.ft_moe_set_keep_activations(None, 1) == F.FT_ERR_ARG
    assert L.ft_moe_destroy(None) == F.FT_OK
    assert L.ft_moe_slot_stride(None) == -1
    assert L.ft_topk_softmax(None, 4, 600, 2, None, None, None) == F.FT_ERR_ARG
    assert L.ft_topk_softmax(None, 4, 8, 9, None, None, None) == F.FT_ERR_ARG
    need = L.ft_permute_workspace_bytes(100, 8, 128)
    assert need == 2 * 4 * 128 * ((100 + 31) // 32)
    assert L.ft_permute(None, 100, 8, 128, None, None, None, None, 0, None) == F.FT_ERR_ARG


def test_package_import_fails_loudly_without_library(F, tmp_path, monkeypatch):
    monkeypatch.setattr(F, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(F, "_lib", None)
    with pytest.raises(ImportError):
        F.lib()


def test_binding_checks_tensors_before_calling_the_library(F):
    """forward and load_pool reject wrong shapes, dtypes and devices in the
    binding itself (a stack object without a handle stands in; nothing
    reaches the library)."""
    import torch

    class NoHandle(F.MoELayerStack):
        def __init__(self):
            self.H, self.E, self.L, self._h = 256, 8, 2, None

    s = NoHandle()
    x = torch.zeros(3, 256, dtype=torch.bfloat16)
    lg = torch.zeros(3, 8, dtype=torch.float32)
    out = torch.zeros(3, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="x must be"):
        s.forward(0, x, lg, out)                     # host tensors
    with pytest.raises(ValueError, match="pool pointers"):
        s.load_pool([1, 2, 3])
