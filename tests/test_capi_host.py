"""The C-ABI library on the host: it loads, exports every declared entry point,
and its host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import diffusion_transformer_joint_txt_b300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flux_attn.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FLUX_ATTN_API\s+[\w\s\*]+?\b(flux_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("flux_attn_create", "flux_attn_forward", "flux_attn_destroy", "flux_attn_sync_status",
                     "flux_attn_prologue", "flux_attn_attend", "flux_attn_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(fa.library_path())
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_uses_the_c_names():
    for n in declared_symbols():
        assert hasattr(fa, n), "binding lacks %s" % n


def test_status_strings():
    assert fa.flux_attn_status_string(0) == "ok"
    assert "timed out" in fa.flux_attn_status_string(fa.FLUX_ATTN_ERR_DEVICE_TIMEOUT)
    assert fa.flux_attn_status_string(999) == "unknown status"


def _create_status(**kw):
    cfg = dict(batch=1, num_heads=2, max_tokens=320)
    cfg.update(kw)
    try:
        h = fa.flux_attn_create(**cfg)
    except fa.FluxAttnError as e:
        return e.status, str(e)
    fa.flux_attn_destroy(h)
    return 0, ""


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), fa.FLUX_ATTN_ERR_UNSUPPORTED),
    (dict(batch=0), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(num_heads=0), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(max_tokens=0), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(axes_dim=(16, 56, 54)), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(axes_dim=(15, 57, 56)), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(axes_dim=(12, 60, 56)), fa.FLUX_ATTN_ERR_UNSUPPORTED),
    (dict(rope_theta=0.0), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(rms_eps=-1.0), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(precision=7), fa.FLUX_ATTN_ERR_INVALID_ARG),
    (dict(batch=1000, num_heads=100), fa.FLUX_ATTN_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config(kw, status):
    got, msg = _create_status(**kw)
    assert got == status, msg
    assert fa.flux_attn_last_error() != ""


def test_calls_on_a_null_handle_are_rejected():
    with pytest.raises(fa.FluxAttnError) as e:
        fa.flux_attn_attend(None, 16, 16, 16, 1, 16, stream=0)
    assert e.value.status == fa.FLUX_ATTN_ERR_INVALID_ARG
    with pytest.raises(fa.FluxAttnError):
        fa.flux_attn_forward(None, 16, 16, 16, 1, 1, 1, 0, 0, None, 16, 16, 16, stream=0)
    assert fa.flux_attn_sync_status(None, stream=0) == fa.FLUX_ATTN_ERR_INVALID_ARG
    fa.flux_attn_destroy(None)  # accepted
    assert fa.flux_attn_workspace_bytes(None) == 0
    assert fa.flux_attn_launches_per_forward(None, 10) == 0


def test_create_without_a_b300_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    got, msg = _create_status()
    assert got in (fa.FLUX_ATTN_ERR_CUDA, fa.FLUX_ATTN_ERR_UNSUPPORTED), msg
