"""The C ABI library: it loads, exports every function include/attn.h declares,
and validates arguments on the host.  No compute call (no GPU needed)."""
import ctypes
import importlib
import os
import re

import pytest

import transformer_self_attention_gb300 as tsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:attn_status|int|const char\s*\*)\s*(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("attn_create", "attn_forward", "attn_destroy", "attn_status_string"):
        assert required in names
    assert set(names) == set(tsa.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(tsa.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for s in range(6):
        assert tsa.attn_status_string(s) and tsa.attn_status_string(s) != "unknown status"
    assert tsa.attn_status_string(99) == "unknown status"


@pytest.mark.parametrize("args,status", [
    ((1, 4, 3, 128, tsa.MASK_CAUSAL, 0, []), tsa.ATTN_ERR_INVALID_ARG),         # Hq % Hkv != 0
    ((0, 4, 4, 128, tsa.MASK_CAUSAL, 0, []), tsa.ATTN_ERR_INVALID_ARG),         # B < 1
    ((1, 4, 4, 0, tsa.MASK_CAUSAL, 0, []), tsa.ATTN_ERR_INVALID_ARG),           # S < 1
    ((1, 4, 4, 128, tsa.MASK_SLIDING, -1, []), tsa.ATTN_ERR_INVALID_ARG),       # negative window
    ((1, 4, 4, 128, tsa.MASK_LOCAL_GLOBAL, 3, [128]), tsa.ATTN_ERR_INVALID_ARG),  # global out of range
    ((1, 4, 4, 128, tsa.MASK_LOCAL_GLOBAL, 3, [-1]), tsa.ATTN_ERR_INVALID_ARG),
    ((1, 4, 4, 128, tsa.MASK_CAUSAL, 0, [5]), tsa.ATTN_ERR_INVALID_ARG),        # globals need LOCAL_GLOBAL
    ((1, 4, 4, 128, 7, 0, []), tsa.ATTN_ERR_INVALID_ARG),                       # unknown kind
])
def test_schedule_argument_validation(args, status):
    with pytest.raises(tsa.AttnError) as e:
        tsa.attn_schedule_host(*args)
    assert e.value.status == status


def test_create_rejects_bad_arguments_before_any_cuda_call():
    # these fail validation on the host, so they behave the same with or without a GPU
    bad = [
        dict(B=1, Hq=4, Hkv=4, S=128, d_k=96, dtype=tsa.ATTN_BF16, scale=0.1, kind=0),   # d_k unsupported
        dict(B=1, Hq=4, Hkv=4, S=128, d_k=64, dtype=tsa.ATTN_BF16, scale=0.0, kind=0),   # scale <= 0
        dict(B=1, Hq=4, Hkv=4, S=128, d_k=64, dtype=tsa.ATTN_BF16, scale=float("nan"), kind=0),
        dict(B=1, Hq=4, Hkv=4, S=128, d_k=64, dtype=5, scale=0.1, kind=0),               # dtype
        dict(B=1, Hq=4, Hkv=3, S=128, d_k=64, dtype=tsa.ATTN_BF16, scale=0.1, kind=0),
    ]
    expect = [tsa.ATTN_ERR_UNSUPPORTED, tsa.ATTN_ERR_INVALID_ARG, tsa.ATTN_ERR_INVALID_ARG,
              tsa.ATTN_ERR_INVALID_ARG, tsa.ATTN_ERR_INVALID_ARG]
    for kw, st in zip(bad, expect):
        with pytest.raises(tsa.AttnError) as e:
            tsa.attn_create(**kw)
        assert e.value.status == st


def test_forward_rejects_null_handle_and_pointers():
    assert tsa.attn_forward(0, 16, 16, 16, 16) == tsa.ATTN_ERR_INVALID_ARG
    assert tsa.attn_destroy(0) == tsa.ATTN_OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(tsa, "LIB_PATH", str(tmp_path / "libattn.so"))
    with pytest.raises(ImportError):
        tsa._load()


def test_kernel_setup_is_made_once_per_device():
    """The shared-memory opt-in of a kernel belongs to a device context: the launchers' registry
    runs it once per (device, kernel), from any number of host threads, and again after a
    failure (fake device ids; no GPU is touched)."""
    assert tsa.attn_selftest_device_once() == 0
