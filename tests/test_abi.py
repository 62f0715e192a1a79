"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/mla.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_attention_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_what_binding_lists():
    assert header_functions() == sorted(mla.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = mla.library()
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    lib = mla.library()
    for code, name in mla.STATUS.items():
        assert lib.mla_status_string(code).decode().startswith(name)
    assert b"unknown" in lib.mla_status_string(99)


FAKE = 0x100000  # never dereferenced: every call below is rejected before any device work


def _kv(**over):
    kw = dict(pool=FAKE, num_pages=16, page_size=64, page_table=FAKE, page_table_stride=16,
              seq_lens=FAKE, kv_scale=1.0)
    kw.update(over)
    return mla.mla_kv_t(**kw)


@pytest.mark.parametrize("kv,B,H,status", [
    (None, 1, 12, 1),
    (_kv(pool=None), 1, 12, 1),
    (_kv(page_table=None), 1, 12, 1),
    (_kv(page_size=48), 1, 12, 2),
    (_kv(page_size=0), 1, 12, 2),
    (_kv(num_pages=-1), 1, 12, 1),
    (_kv(pool=FAKE + 4), 1, 12, 1),
    (_kv(), 1, 0, 2),
    (_kv(), 1, 17, 2),
    (_kv(), -1, 12, 1),
])
def test_decode_rejects_bad_arguments(kv, B, H, status):
    lib = mla.library()
    ref = ctypes.byref(kv) if kv is not None else None
    assert lib.mla_decode(ref, FAKE, B, H, 0.1, FAKE, FAKE, FAKE, 1 << 30, None) == status
    assert lib.mla_last_launch_count() == 0


@pytest.mark.parametrize("n_q", [0, 5, -1])
def test_verify_rejects_positions(n_q):
    lib = mla.library()
    kv = _kv()
    assert lib.mla_verify(ctypes.byref(kv), FAKE, 1, n_q, 12, 0.1, FAKE, FAKE, FAKE, 1 << 30,
                          None) == 2


def test_misaligned_and_missing_buffers():
    lib = mla.library()
    kv = _kv()
    assert lib.mla_decode(ctypes.byref(kv), FAKE + 2, 1, 12, 0.1, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.mla_decode(ctypes.byref(kv), FAKE, 1, 12, 0.1, None, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.mla_decode(ctypes.byref(kv), FAKE, 1, 12, 0.1, FAKE, FAKE, None, 1 << 30, None) == 3
    assert lib.mla_decode(ctypes.byref(kv), FAKE, 1, 12, 0.1, FAKE, FAKE, FAKE + 16, 1 << 30, None) == 3
    assert lib.mla_prefill(ctypes.byref(kv), FAKE, 8, 20, 0.1, FAKE, FAKE, FAKE, 1 << 20, None) == 2
    assert lib.mla_prefill(ctypes.byref(kv), FAKE, 8, 12, 0.1, FAKE, FAKE, FAKE, 4, None) == 3
    assert lib.mla_merge_lse(FAKE, FAKE, -1, 4, FAKE, FAKE, None) == 1
    assert lib.mla_merge_lse(None, FAKE, 2, 4, FAKE, FAKE, None) == 1


def test_workspace_size_rejects_unsupported():
    lib = mla.library()
    assert lib.mla_workspace_size(0, 1, 0, 1, 0) == 0
    assert lib.mla_workspace_size(1, 1, 12, 5, 0) == 0
    assert lib.mla_workspace_size(2, 2, 12, 8, 0) == 0


def test_read_status_rejects_small_workspace():
    lib = mla.library()
    assert lib.mla_read_status(FAKE, 4, None) == 3


def test_cache_append_rejects_bad_arguments():
    lib = mla.library()
    ok = dict(pool=FAKE, num_pages=4, page_size=64, x=FAKE, slots=FAKE, n=3, kv_scale=0.5,
              status=None)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.mla_cache_append(a["pool"], a["num_pages"], a["page_size"], a["x"], a["slots"],
                                    a["n"], a["kv_scale"], a["status"], None)

    assert call(n=-1) == 1
    assert call(page_size=0) == 1
    assert call(kv_scale=0.0) == 1
    assert call(kv_scale=float("inf")) == 1
    assert call(kv_scale=float("nan")) == 1
    assert call(pool=None) == 1
    assert call(x=FAKE + 8) == 1      # bf16 rows are read 16 bytes at a time
    assert call(slots=FAKE + 4) == 1  # int64 slots
    assert call(status=FAKE + 2) == 1
    assert call(n=0, pool=None, x=None, slots=None) == 0  # nothing to do
    assert lib.mla_last_launch_count() == 0


def test_top_k_renorm_rejects_bad_arguments():
    lib = mla.library()
    assert lib.mla_top_k_renorm_prob(FAKE, FAKE, -1, 10, None, 3, None) == 1
    assert lib.mla_top_k_renorm_prob(FAKE, FAKE, 2, -5, None, 3, None) == 1
    assert lib.mla_top_k_renorm_prob(None, FAKE, 2, 10, None, 3, None) == 1
    assert lib.mla_top_k_renorm_prob(FAKE + 2, FAKE, 2, 10, None, 3, None) == 1
    assert lib.mla_top_k_renorm_prob(FAKE, FAKE, 2, 10, FAKE + 1, 3, None) == 1
    assert lib.mla_top_k_renorm_prob(None, None, 0, 10, None, 3, None) == 0  # nothing to do
    assert lib.mla_last_launch_count() == 0


def test_verify_f32_rejects_bad_arguments():
    lib = mla.library()
    kv = mla.mla_kv_t(FAKE, 4, 64, FAKE, 4, FAKE, 1.0)
    call = lib.mla_verify_f32
    assert call(ctypes.byref(kv), FAKE, 1, 5, 12, 1.0, FAKE, FAKE, FAKE, 1 << 20, None) == 2  # n_q > 4
    assert call(ctypes.byref(kv), FAKE, 1, 1, 0, 1.0, FAKE, FAKE, FAKE, 1 << 20, None) == 2   # H < 1
    assert call(ctypes.byref(kv), FAKE, 1, 1, 12, 1.0, None, FAKE, FAKE, 1 << 20, None) == 1  # no out
    assert call(ctypes.byref(kv), FAKE, 1, 1, 12, 1.0, FAKE + 4, FAKE, FAKE, 1 << 20, None) == 1
    assert lib.mla_last_launch_count() == 0


def test_prefill_mha_rejects_bad_arguments():
    lib = mla.library()
    kv = mla.mla_kv_t(FAKE, 4, 64, FAKE, 4, FAKE, 1.0)
    call = lib.mla_prefill_mha
    ws = 1 << 30
    assert call(ctypes.byref(kv), 100, FAKE, 200, 12, FAKE, 1.0, FAKE, FAKE, FAKE, ws, None) == 1  # L < T
    assert call(ctypes.byref(kv), 300, FAKE, 200, 12, FAKE, 1.0, FAKE, FAKE, FAKE, ws, None) == 1  # L > capacity
    assert call(ctypes.byref(kv), 200, FAKE, 100, 17, FAKE, 1.0, FAKE, FAKE, FAKE, ws, None) == 2  # H > 16
    assert call(ctypes.byref(kv), 200, FAKE, 100, 12, None, 1.0, FAKE, FAKE, FAKE, ws, None) == 1  # no weights
    assert call(ctypes.byref(kv), 200, FAKE + 8, 100, 12, FAKE, 1.0, FAKE, FAKE, FAKE, ws, None) == 1
    assert call(ctypes.byref(kv), 200, FAKE, 100, 12, FAKE, 1.0, FAKE, FAKE, FAKE + 16, ws, None) == 3
    assert call(ctypes.byref(kv), 200, FAKE, 0, 12, FAKE, 1.0, FAKE, FAKE, FAKE, ws, None) == 0  # T = 0
    assert lib.mla_last_launch_count() == 0
    assert lib.mla_prefill_mha_workspace_size(-1, 12, 0) == 0
