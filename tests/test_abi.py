"""The C-ABI library builds, loads without a GPU and exports every declared entry point."""
import glob
import os
import re

import pytest

import block_sparse_kv_bsr_gb300 as bsr
from block_sparse_kv_bsr_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(bsr_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return bsr.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("bsr_attn_plan", "bsr_attn_run", "bsr_merge_states", "bsr_append_kv",
              "bsr_schedule_destroy", "bsr_last_device_error", "bsr_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert set(bsr.EXPORTED_SYMBOLS) == declared_functions()


def test_status_strings(lib):
    assert bsr.bsr_status_string(0) == "ok"
    for code in range(-7, 0):
        assert bsr.bsr_status_string(code) not in ("ok", "unknown status")
    assert bsr.bsr_status_string(-99) == "unknown status"


def _plan_host(**kw):
    base = dict(indptr=[0, 2, 3], indices=[0, 1, 2], last_page_len=[5, 16], num_qo_heads=8,
                num_kv_heads=2, head_dim=128, page_size=16, num_pages=3, num_sms=4)
    base.update(kw)
    return bsr.bsr_attn_plan_host(**base)


def test_plan_host_accepts_a_valid_table(lib):
    info, units = _plan_host()
    assert info["active_tokens"] == 16 + 5 + 16
    assert units.shape[1] == 8


@pytest.mark.parametrize("kw,code", [
    (dict(indices=[0, 1, 3]), -3),                       # page id outside the pool
    (dict(indices=[0, -1, 2]), -3),                      # negative page id
    (dict(last_page_len=[0, 16]), -3),                   # empty last page
    (dict(last_page_len=[17, 16]), -3),                  # last page longer than P
    (dict(indptr=[0, 3, 2], indices=[0, 1, 2]), -3),     # decreasing indptr
    (dict(indptr=[1, 2, 3]), -3),                        # indptr must start at 0
    (dict(head_dim=96), -2),
    (dict(page_size=12), -2),
    (dict(page_size=512), -2),
    (dict(num_qo_heads=6, num_kv_heads=4), -2),          # Hq not a multiple of Hk
    (dict(num_qo_heads=64, num_kv_heads=2), -2),         # group of 32 > 16
    (dict(num_sms=0), -1),
    (dict(qo_indptr=[0, 40, 41], causal=True), -3),      # more queries than keys
    (dict(rope_theta=-1.0), -1),
    (dict(num_pages=1 << 27), -2),                       # pool rows beyond 32-bit indexing
])
def test_plan_host_rejects(lib, kw, code):
    with pytest.raises(bsr.BsrError) as e:
        _plan_host(**kw)
    assert e.value.code == code


def test_entry_points_reject_bad_arguments_without_a_gpu(lib):
    assert lib.bsr_attn_run(None, None, None, None, 1.0, 0.0, 0, None, 0, None, None) == -1
    assert lib.bsr_merge_states(None, None, None, None, 1, 1, 96, 0, None, None, None) == -2
    assert lib.bsr_append_kv(None, None, None, None, None, None, 1, 1, 1, 128, 3, 1, 0,
                             None, None, None, None) == -2
    assert lib.bsr_selftest_bounded_wait(None, 1000, None) == -1
    # FP8 without a GPU: head_dim 64 is outside the FP8 kernel's set; a zero scale is refused
    assert lib.bsr_attn_decode_noalloc_kv8(None, None, None, None, None, None, 1, 8, 2, 64, 16,
                                           4, 0.125, 1.0, 1.0, None, 0, None, None, None) == -2
    assert lib.bsr_attn_decode_noalloc_kv8(None, None, None, None, None, None, 1, 8, 2, 128, 16,
                                           4, 0.125, 0.0, 1.0, None, 0, None, None, None) == -1
    # the general entry: an unknown cache dtype and a negative window are refused
    assert lib.bsr_attn_decode_noalloc_ex(None, None, None, None, None, None, 1, 8, 2, 128, 16,
                                          4, 0.125, 7, 1.0, 1.0, 0, None, 0, None, None,
                                          None) == -1
    assert lib.bsr_attn_decode_noalloc_ex(None, None, None, None, None, None, 1, 8, 2, 128, 16,
                                          4, 0.125, 0, 1.0, 1.0, -5, None, 0, None, None,
                                          None) == -1
    # an unknown page layout
    assert lib.bsr_append_kv(None, None, None, None, None, None, 1, 1, 1, 128, 16, 1, 7,
                             None, None, None, None) == -1
