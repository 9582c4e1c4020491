"""CPU-side checks of the boundary: the library builds, loads without a GPU and
exports every function include/csa2.h declares; the binding fails loudly when
the library is missing."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    from fp4_kv_cache_csa2_gb300 import build
    return build.build()


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for call in ("csa2_compress_quantize", "csa2_index_score", "csa2_block_topk", "csa2_select_topk",
                 "csa2_sparse_swa_attn", "csa2_decode", "csa2_sync_status", "csa2_status_string"):
        assert call in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(lib_path):
    import fp4_kv_cache_csa2_gb300 as csa2
    assert sorted(csa2.exported_symbols()) == declared_functions()


def test_host_only_calls_without_gpu(lib_path):
    import fp4_kv_cache_csa2_gb300 as csa2
    lib = csa2.load(lib_path)
    assert lib.csa2_layout_version() == 1
    assert lib.csa2_status_string(6) == b"CSA2_ERR_BOUNDS"
    assert lib.csa2_attn_workspace_size(1, 1, 512) >= 256
    assert lib.csa2_block_topk_workspace_size(2, 3, 100) == 256 + 512    # 2*3*13*4 = 312 bytes -> 512
    assert lib.csa2_select_topk_workspace_size(2, 3, 16384) == 256       # short rows: header only
    # long rows: per row and kind a 4096-bin histogram + 16 counters, 2048 sure picks, 8192 candidates
    per = 2 * 6 * (4096 * 4 + 64 + 2048 * 4 + 8192 * 8)
    assert lib.csa2_select_topk_workspace_size(2, 3, 16385) >= 256 + per
    assert lib.csa2_block_topk_workspace_size(2, 3, 1 << 20) == lib.csa2_select_topk_workspace_size(2, 3, 1 << 20)
    # argument validation happens before any CUDA call
    assert lib.csa2_index_score(None, None, None, None, None, 0, None, 1, 1, 10, None, 0, None) == 1


def test_variant_calls_host_logic_without_gpu(lib_path):
    """Workspace arithmetic and argument checks of the HISA and FP8-window calls
    (all return before any CUDA call)."""
    import fp4_kv_cache_csa2_gb300 as csa2
    lib = csa2.load(lib_path)
    # HISA: header + view positions (int64 per query) + summary rows (int32 per
    # sequence) + one score per summary row, each rounded to 256 bytes
    assert lib.csa2_hisa_blocks_workspace_size(2, 3, 1000) == 256 + 256 + 256 + 3072   # 6 x 125 x 4 = 3000
    per_rows = lib.csa2_select_topk_workspace_size(2, 3, 1 << 20) - 256               # long-row lists
    scores = -(-6 * 4097 * 4 // 256) * 256                                               # 98,328 -> 98,560
    assert lib.csa2_hisa_blocks_workspace_size(2, 3, 8 * 4097) == 256 + 256 + 256 + scores + per_rows
    assert lib.csa2_hisa_blocks_workspace_size(-1, 3, 10) == 0
    fake = ctypes.c_void_p(1 << 20)                     # never dereferenced: the calls fail on arguments
    n = ctypes.c_int32(0)
    cache = csa2.CacheStruct(fake.value, fake.value, fake.value, 64, ctypes.addressof(n), 1)
    ws = ctypes.c_void_p(1 << 24)
    # block summary: sum_cap must be a multiple of 8; negative counts
    assert lib.csa2_block_summary(ctypes.byref(cache), fake, 1, 1, fake, fake, 12, ws, 1 << 16, None) == 1
    assert lib.csa2_block_summary(ctypes.byref(cache), fake, -1, 1, fake, fake, 8, ws, 1 << 16, None) == 1
    assert lib.csa2_block_summary(ctypes.byref(cache), fake, 1, 1, fake, fake, 8, None, 0, None) == 3
    # HISA blocks: M outside 1..2048; store shorter than ceil(cap / 8) rows
    ws_need = lib.csa2_hisa_blocks_workspace_size(1, 1, 64)
    args = (fake, fake, fake, 1, 1, 64)                 # q_idx, w_head, q_pos, B, Q, max_n
    assert lib.csa2_hisa_blocks(ctypes.byref(cache), fake, fake, 8, *args, 0, fake, ws, ws_need, None) == 2
    assert lib.csa2_hisa_blocks(ctypes.byref(cache), fake, fake, 0, *args, 4, fake, ws, ws_need, None) == 1
    assert lib.csa2_hisa_blocks(ctypes.byref(cache), fake, fake, 8, *args, 4, fake, ws, ws_need - 1, None) == 3
    # FP8 window: alignment and counts
    assert lib.csa2_swa_quantize_fp8(fake, 4, ctypes.c_void_p((1 << 20) + 8), None) == 1
    assert lib.csa2_swa_quantize_fp8(fake, -4, fake, None) == 1
    assert lib.csa2_swa_quantize_fp8(None, 0, None, None) == 0   # nothing to do
    # decode: swa_fp8 must be 0 or 1
    a = csa2.DecodeArgs()
    a.mode, a.B, a.Q, a.M, a.K, a.S, a.max_n, a.scale = 2, 1, 1, 8, 8, 128, 64, 0.04
    for f in ("q_pos", "q", "swa", "swa_base_pos", "sel", "out"):
        setattr(a, f, fake.value)
    a.swa_fp8 = 2
    need = lib.csa2_decode_workspace_size(2, 1, 1, 64, 8, 8)
    assert lib.csa2_decode(ctypes.byref(cache), ctypes.byref(a), ws, need, None) == 1
    # decode: attn_split must not be negative, and a split call holds at most 128 queries
    a.swa_fp8 = 0
    a.attn_split = -1
    assert lib.csa2_decode(ctypes.byref(cache), ctypes.byref(a), ws, need, None) == 1
    a.B, a.attn_split = 129, 5
    need = lib.csa2_decode_workspace_size(2, 129, 1, 64, 8, 8)
    assert lib.csa2_decode(ctypes.byref(cache), ctypes.byref(a), ws, need, None) == 2
    # the partial states of a split call are part of the workspace up to 128 queries, none beyond
    per_query = 2 * (2 * 64 + 64 * 512) * 4                       # K = 8: the window and one run, 2 CTAs
    assert (lib.csa2_decode_workspace_size(2, 128, 1, 64, 8, 8) - lib.csa2_decode_workspace_size(2, 1, 1, 64, 8, 8)
            >= 127 * per_query)
    assert lib.csa2_decode_workspace_size(2, 129, 1, 64, 8, 8) < per_query


def test_query_count_limit_and_concurrent_argument_checks(lib_path):
    """More than 2^26 queries in one call is refused before anything is
    enqueued (every grid is one-dimensional), by the regular and the
    allocation-free candidate-block calls alike.  Host threads calling the
    argument checks at once all get the same answers (ctypes releases the GIL
    for the foreign calls, so the calls do overlap)."""
    import threading
    import fp4_kv_cache_csa2_gb300 as csa2
    lib = csa2.load(lib_path)
    fake = ctypes.c_void_p(1 << 20)                     # never dereferenced: the calls fail on arguments
    n = ctypes.c_int32(0)
    cache = csa2.CacheStruct(fake.value, fake.value, fake.value, 64, ctypes.addressof(n), 1)
    ws = ctypes.c_void_p(1 << 24)
    big_b, big_q = 1 << 13, (1 << 13) + 1               # 67,117,056 queries > 2^26
    cases = [
        (lambda: lib.csa2_block_topk_static(ctypes.byref(cache), fake, fake, big_b, big_q, 0, 4, fake, None), 2),
        (lambda: lib.csa2_block_topk(ctypes.byref(cache), fake, fake, big_b, big_q, 0, 4, fake, ws, 1 << 30,
                                     None), 2),
        (lambda: lib.csa2_select_topk(ctypes.byref(cache), fake, fake, None, 0, 8, fake, big_b, big_q, 0, ws,
                                      1 << 30, None), 2),
        (lambda: lib.csa2_block_topk_static(ctypes.byref(cache), fake, fake, 1, 1, 8, 0, fake, None), 2),
        (lambda: lib.csa2_block_topk_static(None, fake, fake, 1, 1, 8, 4, fake, None), 1),
        (lambda: lib.csa2_select_topk(ctypes.byref(cache), fake, fake, None, 0, 8, fake, 1, 1, 64, None, 0, None),
         3),
    ]
    for call, want in cases:
        assert call() == want
    errors = []

    def worker():
        try:
            for _ in range(300):
                for call, want in cases:
                    got = call()
                    if got != want:
                        errors.append((want, got))
        except Exception as e:                          # pragma: no cover - reported below
            errors.append(e)
    threads = [threading.Thread(target=worker) for _ in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:5]


def test_rope_table_matches_oracle_bit_for_bit(lib_path):
    """The library's table builder and the oracle's are separate restatements of
    cos/sin(p * theta^(-2i/64)); their binary32 tables agree."""
    import numpy as np
    import fp4_kv_cache_csa2_gb300 as csa2
    import oracle
    got = csa2.rope_table(70000).numpy()
    want = oracle.rope_table(70000)
    np.testing.assert_array_equal(got, want)


def test_missing_library_fails_loudly(tmp_path):
    import fp4_kv_cache_csa2_gb300 as csa2
    saved = csa2._lib
    csa2._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            csa2.load(str(tmp_path / "libcsa2.so"))
    finally:
        csa2._lib = saved


def _c_layout(tmp_path, struct: str, fields: list[str]) -> list[int]:
    """sizeof(struct) followed by offsetof(struct, f) for each field, from a
    small C program compiled against include/csa2.h with the host compiler."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    src = tmp_path / "layout.c"
    body = "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "csa2.h"\n'
                   f'int main(void) {{\n  printf("%zu\\n", sizeof({struct}));\n{body}  return 0;\n}}\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    return [int(x) for x in out]


def test_binding_structs_match_the_c_layout(tmp_path):
    """The ctypes mirrors of csa2_cache and csa2_decode_args (including the
    packed_sel field appended last) have the C structs' sizes and offsets."""
    import fp4_kv_cache_csa2_gb300 as csa2
    for cls, struct in ((csa2.DecodeArgs, "csa2_decode_args"), (csa2.CacheStruct, "csa2_cache")):
        names = [f[0] for f in cls._fields_]
        c = _c_layout(tmp_path, struct, names)
        assert c[0] == ctypes.sizeof(cls), struct
        assert c[1:] == [getattr(cls, n).offset for n in names], struct
