"""The C-ABI library builds, loads and exports every entry point include/sfi.h
declares; host-side argument validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sfi.h")


@pytest.fixture(scope="module")
def libsfi():
    from sparse_kv_long_sfi_gb300 import _abi, build
    build.build()
    return _abi.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^SFI_API\s+[\w\s\*]+?\b(sfi_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_five_hot_path_calls():
    names = declared_functions()
    for n in ["sfi_paged_kv_append", "sfi_fast_decode_attn", "sfi_slow_dense_attn_with_scores", "sfi_select_topk",
              "sfi_compact_gather"]:
        assert n in names


def test_library_exports_every_declared_symbol(libsfi):
    from sparse_kv_long_sfi_gb300 import _abi
    names = declared_functions()
    assert set(names) == set(_abi.PROTOTYPES)
    for n in names:
        assert hasattr(libsfi, n), n


def test_library_exports_nothing_else(libsfi):
    import subprocess
    from sparse_kv_long_sfi_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    assert exported == set(declared_functions())


def test_version_and_status_strings(libsfi):
    assert libsfi.sfi_version() == 1
    assert libsfi.sfi_status_string(0) == b"SFI_OK"
    assert libsfi.sfi_status_string(3) == b"SFI_ERR_WORKSPACE"
    assert libsfi.sfi_status_string(99) == b"SFI_ERR_UNKNOWN"


def _shape(hq=16, hkv=8, d=128, p=16):
    from sparse_kv_long_sfi_gb300 import _abi
    return _abi.sfi_attn_shape(hq, hkv, d, p, 0.0)


def _paged(npages=4, maxp=4):
    from sparse_kv_long_sfi_gb300 import _abi
    # dummy, 16-byte aligned host addresses: validation never dereferences them
    return _abi.sfi_paged_kv(4096, 8192, npages, maxp, 12288, 16384)


@pytest.mark.parametrize("shape_args,expect", [
    ((16, 8, 96, 16), 2),    # head_dim 96 unsupported
    ((16, 8, 128, 32), 2),   # page size 32 unsupported
    ((48, 4, 128, 16), 2),   # G = 12 unsupported
    ((16, 5, 128, 16), 1),   # Hq not a multiple of Hkv
    ((0, 8, 128, 16), 1),
])
def test_shape_validation_before_launch(libsfi, shape_args, expect):
    sh = _shape(*shape_args)
    kv = _paged()
    st = libsfi.sfi_slow_dense_attn_with_scores(ctypes.byref(sh), ctypes.byref(kv), 4, 32, 4096, None, None, 8192,
                                                None, None, 0, None, 1, 0, 0, 0, None, 0, None, None)
    assert st == expect


def test_null_and_negative_arguments(libsfi):
    from sparse_kv_long_sfi_gb300 import _abi
    sh, kv = _shape(), _paged()
    assert libsfi.sfi_paged_kv_append(None, ctypes.byref(kv), 4096, 4096, None, 1, None, None) == 1
    assert libsfi.sfi_paged_kv_append(ctypes.byref(sh), None, 4096, 4096, None, 1, None, None) == 1
    assert libsfi.sfi_paged_kv_append(ctypes.byref(sh), ctypes.byref(kv), None, 4096, None, 1, None, None) == 1
    assert libsfi.sfi_paged_kv_append(ctypes.byref(sh), ctypes.byref(kv), 4097, 4096, None, 1, None, None) == 1
    comp = _abi.sfi_compact_kv(4096, 4096, 100, 4096, 4096, 4096)
    assert libsfi.sfi_fast_decode_attn(ctypes.byref(sh), ctypes.byref(kv), ctypes.byref(comp), -1, 32, 4096, None,
                                       None, 4096, None, None, 1, 0, 0, 0, None, 0, None, None) == 1
    assert libsfi.sfi_fast_decode_attn(ctypes.byref(sh), ctypes.byref(kv), None, 4, 32, 4096, None, None, 4096,
                                       None, None, 1, 0, 0, 0, None, 0, None, None) == 1
    # k_new without v_new
    assert libsfi.sfi_fast_decode_attn(ctypes.byref(sh), ctypes.byref(kv), ctypes.byref(comp), 4, 32, 4096, 4096,
                                       None, 4096, None, None, 1, 0, 0, 0, None, 0, None, None) == 1
    assert libsfi.sfi_select_topk(None, 16, 8, 4096, 4, 32, 4096, 8, 4096, 4096, None, 1, None, None) == 1
    assert libsfi.sfi_select_topk(4096, 0, 8, 4096, 4, 32, 4096, 8, 4096, 4096, None, 1, None, None) == 1
    assert libsfi.sfi_compact_gather(ctypes.byref(sh), ctypes.byref(kv), 4096, 4096, -1, 4, ctypes.byref(comp),
                                     None, 1, None, None) == 1
    bad_pages = _abi.sfi_paged_kv(4096, 8192, 0, 4, 12288, 16384)
    assert libsfi.sfi_paged_kv_append(ctypes.byref(sh), ctypes.byref(bad_pages), 4096, 4096, None, 1, None,
                                      None) == 1


def test_empty_batch_is_a_no_op(libsfi):
    sh, kv = _shape(), _paged()
    assert libsfi.sfi_paged_kv_append(ctypes.byref(sh), ctypes.byref(kv), 4096, 4096, None, 0, None, None) == 0
    assert libsfi.sfi_select_topk(4096, 16, 8, 4096, 4, 32, 4096, 8, 4096, 4096, None, 0, None, None) == 0


def test_workspace_size_rejects_bad_shapes(libsfi):
    sh = _shape(16, 8, 96)
    assert libsfi.sfi_workspace_size(ctypes.byref(sh), 4, 1024, 0) == 0
    assert libsfi.sfi_plan_splits(ctypes.byref(sh), 4, 1024, 0) == 0
    assert libsfi.sfi_plan_splits(ctypes.byref(_shape()), 4, 0, 0) == 1  # no token bound: one split
    assert libsfi.sfi_plan_splits(ctypes.byref(_shape()), 4, 4096, 3) == 3  # explicit request honoured
    for bad in (0, -1, 9, 16):
        assert libsfi.sfi_attn_cluster_capacity(bad) == 0


def test_cluster_capacity_needs_a_device(libsfi):
    """The capacity query answers 0 for every valid size when there is no CUDA device
    (so automatic plans keep the slot-count rule), and a positive count with one."""
    import torch
    caps = [libsfi.sfi_attn_cluster_capacity(c) for c in range(1, 9)]
    if torch.cuda.is_available():
        assert all(c > 0 for c in caps)
    else:
        assert caps == [0] * 8
        assert libsfi.sfi_plan_splits(ctypes.byref(_shape()), 4, 4096, 3) == 3  # plans still answer


def test_multi_token_calls_validate_on_the_host(libsfi):
    from sparse_kv_long_sfi_gb300 import _abi
    sh, kv = _shape(), _paged()  # G = 2: at most 8 tokens
    comp = _abi.sfi_compact_kv(4096, 4096, 100, 4096, 4096, 4096)

    def verify(T, batch=1, scores=None, stride=0):
        return libsfi.sfi_dense_verify_attn(ctypes.byref(sh), ctypes.byref(kv), 4, 32, 4096, T, None, None, 8192, None,
                                            scores, stride, None, batch, 0, 0, 0, None, 0, None, None)

    def draft(T, c=comp, batch=1):
        return libsfi.sfi_sparse_draft_attn(ctypes.byref(sh), ctypes.byref(kv), c and ctypes.byref(c), 4, 32, 4096,
                                            T, None, None, 8192, None, None, batch, 0, 0, 0, None, 0, None, None)

    assert verify(0) == 1 and verify(17) == 1
    assert verify(9) == 2                      # 9 tokens x G = 2 > 16 rows
    assert verify(8, batch=0) == 0             # empty batch: nothing to do
    assert verify(4, scores=4096, stride=0) == 1
    assert draft(0) == 1 and draft(9) == 2 and draft(4, c=None) == 1
    assert draft(8, batch=0) == 0
    sh8 = _shape(32, 4)                        # G = 8: two tokens
    assert libsfi.sfi_dense_verify_attn(ctypes.byref(sh8), ctypes.byref(kv), 4, 32, 4096, 3, None, None, 8192, None,
                                        None, 0, None, 1, 0, 0, 0, None, 0, None, None) == 2
    # k_new without v_new
    assert libsfi.sfi_dense_verify_attn(ctypes.byref(sh), ctypes.byref(kv), 4, 32, 4096, 2, 4096, None, 8192, None,
                                        None, 0, None, 1, 0, 0, 0, None, 0, None, None) == 1
    assert libsfi.sfi_paged_kv_append_tokens(ctypes.byref(sh), ctypes.byref(kv), 4096, 4096, 0, None, 1, None,
                                             None) == 1
    assert libsfi.sfi_paged_kv_append_tokens(ctypes.byref(sh), ctypes.byref(kv), 4096, 4096, 5, None, 0, None,
                                             None) == 0
    assert libsfi.sfi_multi_workspace_size(ctypes.byref(sh), 4, 0, 1024, 0) == 0


def test_select_compact_validates_on_the_host(libsfi):
    from sparse_kv_long_sfi_gb300 import _abi
    sh, kv = _shape(), _paged()
    comp = _abi.sfi_compact_kv(4096, 4096, 100, 4096, 4096, 4096)

    def call(scores=4096, stride=16, k=4096, idx=4096, cnt=4096, c=comp, batch=1, sink=4):
        return libsfi.sfi_select_compact(ctypes.byref(sh), ctypes.byref(kv), scores, stride, sink, 32, k, 8, idx, cnt,
                                         c and ctypes.byref(c), None, batch, None, None)

    assert call(scores=None) == 1 and call(stride=0) == 1 and call(k=None) == 1 and call(idx=None) == 1
    assert call(cnt=None) == 1 and call(c=None) == 1 and call(sink=-1) == 1
    assert call(c=_abi.sfi_compact_kv(4097, 4096, 100, 4096, 4096, 4096)) == 1  # unaligned compact K
    assert call(batch=0) == 0


def test_binding_constants_match_the_header():
    """Every numeric #define and status enumerator of include/sfi.h has the same value
    in the Python binding."""
    from sparse_kv_long_sfi_gb300 import _abi
    text = open(os.path.join(os.path.dirname(__file__), "..", "include", "sfi.h")).read()
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define (SFI_(?:DEV|ATTN|MAX)_\w+) (\d+)u?\b", text, re.M)}
    enums = {m.group(1): int(m.group(2)) for m in re.finditer(r"^\s+(SFI_(?:OK|ERR_\w+)) = (\d+)", text, re.M)}
    assert len(defines) >= 10 and len(enums) == 5
    for name, value in {**defines, **enums}.items():
        assert getattr(_abi, name) == value, name
