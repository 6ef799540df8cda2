"""Host-side checks of the C-ABI library that need no GPU.

The library must load, export every entry point ``include/qd.h`` declares, and
reject bad configurations during validation, before any device work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qd():
    import __graft_entry__
    __graft_entry__.build_library()
    import transformer_autoregressive_decode_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "qd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qd_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("qd_create", "qd_prefill", "qd_decode_step", "qd_grow_kv", "qd_reset", "qd_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(qd):
    lib = ctypes.CDLL(qd.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(qd.EXPORTS) == _declared()


def test_status_strings(qd):
    for st in range(0, -8, -1):
        assert qd.qd_status_string(st).startswith("QD_")
    assert qd.qd_status_string(5) == "unknown status"


def _cfg(qd, **kw):
    base = dict(hidden=256, n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=768, vocab=1024,
                embed_rows=1024, bf16=False, qk_norm=True, buckets=(128,))
    base.update(kw)
    return qd.make_config(**base)


@pytest.mark.parametrize("bad,expect", [
    (dict(n_q_heads=3), "QD_EINVAL"),
    (dict(head_dim=96), "QD_EUNSUPPORTED"),
    (dict(hidden=300), "QD_EUNSUPPORTED"),
    (dict(ffn=10240), "QD_EUNSUPPORTED"),
    (dict(buckets=(128, 64)), "QD_EINVAL"),
    (dict(buckets=(100,)), "QD_EINVAL"),
    (dict(n_heads_out=17), "QD_EINVAL"),
    (dict(eos_mask_id=1024), "QD_EINVAL"),
    (dict(rep_penalty=0.0), "QD_EINVAL"),
    (dict(n_layers=0), "QD_EINVAL"),
    (dict(weight_q8=True), "QD_EUNSUPPORTED"),               # 8-bit rows need bf16
    (dict(bf16=True, weight_q8=2), "QD_EINVAL"),
])
def test_create_validates_config_before_device_work(qd, bad, expect):
    q8 = bad.pop("weight_q8", None) if bad.get("weight_q8") == 2 else None
    cfg = _cfg(qd, **bad)
    if q8 is not None:
        cfg.weight_q8 = q8                                     # past make_config's bool
    out = ctypes.c_void_p(123)
    st = qd._lib.qd_create(None, ctypes.byref(cfg), None, ctypes.byref(out))
    assert qd.qd_status_string(st).startswith(expect)
    assert out.value is None


def test_null_handle_calls_are_rejected(qd):
    assert qd._lib.qd_reset(None) == qd.QD_EINVAL
    assert qd._lib.qd_decode_step(None, None, 0, 0, None) == qd.QD_EINVAL
    assert qd._lib.qd_grow_kv(None, 256) == qd.QD_EINVAL
    assert qd._lib.qd_destroy(None) == qd.QD_OK
    assert qd._lib.qd_create(None, None, None, None) == qd.QD_EINVAL


def test_product_package_does_not_use_the_oracle():
    pkg = os.path.join(ROOT, "transformer_autoregressive_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle." not in text.replace("the oracle", ""), f
                assert "liboracle" not in text, f
