"""The C-ABI library loads (no GPU needed) and exports every declared entry point."""
import glob
import os
import re

from continuous_batching_ragged_gb300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_DECL = re.compile(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**(cb_[A-Za-z0-9_]+)\s*\(", re.M)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names.update(_DECL.findall(open(h).read()))
    return names


def test_headers_declare_the_expected_entry_points():
    names = declared_functions()
    for required in ("cb_append_kv", "cb_ragged_attention", "cb_build_batch"):
        assert required in names
    assert names == set(native.EXPORTS)


def test_library_exports_every_declared_symbol(native_lib):
    for name in declared_functions():
        assert hasattr(native_lib, name), name


def test_status_codes_match_header():
    text = open(os.path.join(ROOT, "include", "cb.h")).read()
    for code, name in native.STATUS_NAMES.items():
        assert re.search(rf"{name}\s*=\s*{code}\b", text), name


def test_host_errors_need_no_gpu(native_lib):
    import ctypes
    # a null cache pointer is rejected before any CUDA call
    assert native_lib.cb_append_kv(None, None, None, 4, None, None) == native.CB_ERR_INVALID
    assert b"null cache" in native_lib.cb_last_error()
    c = native.cb_kv_cache(None, None, 16, 16, 32, 128, native.CB_DTYPE_BF16)
    st = native_lib.cb_ragged_attention(None, ctypes.byref(c), None, None, None, 2, 2, 4, 1, 64,
                                        0.1, None, None, 0, None)
    assert st == native.CB_ERR_INVALID
    c.head_dim = 96
    st = native_lib.cb_ragged_attention(None, ctypes.byref(c), None, None, None, 2, 2, 4, 1, 64,
                                        0.1, None, None, 0, None)
    assert st == native.CB_ERR_UNSUPPORTED
    # empty step: nothing to do
    c.head_dim = 128
    assert native_lib.cb_ragged_attention(None, ctypes.byref(c), None, None, None, 0, 0, 0, 0, 0,
                                          0.1, None, None, 0, None) == native.CB_OK
    assert native_lib.cb_append_kv(None, None, None, 0, ctypes.byref(c), None) == native.CB_OK


def test_workspace_size_rules(native_lib):
    import ctypes
    c = native.cb_kv_cache(None, None, 16, 16, 32, 128, native.CB_DTYPE_BF16)

    def a256(x):
        return (x + 255) // 256 * 256

    def bf16_step(S, T, max_ctx, H=32, A=128):
        # header + decode items and their unsorted copy [S*splits] + prefill
        # chunk records and their unsorted copy [T/256 + min(S, T/2) + 1]
        # (int2 each) + prefill entries [that * H + 1024] (int4) + segment
        # tickets [1024, 8] + segment partials [1024, A+2, 256] fp32 (a prefill
        # chunk with contexts past 2048 keys only) + tickets [S,H] + split
        # partials, all for the shortest split (512 keys)
        splits = (max_ctx + 511) // 512
        pre_cap = T // 256 + min(S, T // 2) + 1
        seg = 1024 * 256 * (A + 2) * 4 if T > S and max_ctx > 2048 else 0
        partials = S * H * splits * (A + 2) * 4 if splits > 1 else 0
        return (256 + 2 * a256(S * splits * 8) + 2 * a256(pre_cap * 8) + a256((pre_cap * H + 1024) * 16)
                + 32768 + seg + a256(S * H * 4) + partials)

    # one split per row: no split partials, no segments
    assert native_lib.cb_attention_workspace_size(ctypes.byref(c), 8, 8, 512) == bf16_step(8, 8, 512) == 54016
    # decode rows with up to 9 splits: partials [S,H,splits,A+2] fp32 dominate
    n = native_lib.cb_attention_workspace_size(ctypes.byref(c), 256, 256, 4097)
    assert n == bf16_step(256, 256, 4097) == (256 + 36864 + 2560 + 82944 + 32768 + 32768
                                              + 256 * 32 * 9 * 130 * 4)
    # a prefill chunk over a long context: the segment partials come in
    n = native_lib.cb_attention_workspace_size(ctypes.byref(c), 1, 2048, 32768)
    assert n == bf16_step(1, 2048, 32768) > 1024 * 256 * 130 * 4
    assert native_lib.cb_attention_workspace_size(ctypes.byref(c), 1, 2048, 2048) == bf16_step(1, 2048, 2048)
    c.dtype = native.CB_DTYPE_F32
    c.head_dim = 64
    n = native_lib.cb_attention_workspace_size(ctypes.byref(c), 3, 6, 1024)
    assert n == 768 + 6 * 32 * 2 * 66 * 4   # f32 rows: per-row split partials, no step plan
