"""Python binding of the CSA2 C-ABI library (``libcsa2.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  Importing this package
does not build anything; ``load()`` raises if the library has not been built
(``python -m fp4_kv_cache_csa2_gb300.build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa2.so")

D_LATENT, D_ROPE, N_HEADS = 512, 64, 64
N_INDEX_HEADS, D_INDEX = 32, 128
BLOCK, WINDOW = 8, 128
MAIN_ENTRY_BYTES, INDEX_CODE_BYTES, INDEX_SCALE_BYTES = 288, 64, 4
MAX_K, MAX_M = 512, 2048
WS_HEADER_BYTES = 256
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2

STATUS_NAMES = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED",
                3: "CSA2_ERR_WORKSPACE", 4: "CSA2_ERR_CUDA", 5: "CSA2_ERR_TIMEOUT",
                6: "CSA2_ERR_BOUNDS"}


class Csa2Error(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class CacheStruct(ctypes.Structure):
    _fields_ = [("main_kv", ctypes.c_void_p), ("idx_codes", ctypes.c_void_p),
                ("idx_scales", ctypes.c_void_p), ("cap", ctypes.c_int64),
                ("n_entries", ctypes.c_void_p), ("m", ctypes.c_int32)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("B", ctypes.c_int), ("Q", ctypes.c_int),
                ("M", ctypes.c_int), ("K", ctypes.c_int), ("S", ctypes.c_int),
                ("max_n", ctypes.c_int64), ("scale", ctypes.c_float),
                ("q_pos", ctypes.c_void_p), ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("w_head", ctypes.c_void_p), ("swa", ctypes.c_void_p),
                ("swa_base_pos", ctypes.c_void_p), ("pool_blocks", ctypes.c_void_p),
                ("sel", ctypes.c_void_p), ("out", ctypes.c_void_p), ("packed_sel", ctypes.c_void_p),
                ("swa_fp8", ctypes.c_int32), ("attn_split", ctypes.c_int32)]


_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_SIGNATURES = {
    "csa2_layout_version": (ctypes.c_int, []),
    "csa2_status_string": (ctypes.c_char_p, [_I]),
    "csa2_workspace_init": (_I, [_P, _SZ, _P]),
    "csa2_sync_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int64)]),
    "csa2_rope_table": (_I, [_P, _I64, ctypes.c_double]),
    "csa2_compress_quantize": (_I, [ctypes.POINTER(CacheStruct), _P, _I, _I, _P, _P, _P, _P, _I64,
                                    _P, _P, _SZ, _P]),
    "csa2_index_score": (_I, [ctypes.POINTER(CacheStruct), _P, _P, _P, _P, _I, _P, _I, _I, _I64,
                              _P, _SZ, _P]),
    "csa2_block_topk_workspace_size": (_SZ, [_I, _I, _I64]),
    "csa2_block_topk": (_I, [ctypes.POINTER(CacheStruct), _P, _P, _I, _I, _I64, _I, _P, _P, _SZ, _P]),
    "csa2_block_topk_static": (_I, [ctypes.POINTER(CacheStruct), _P, _P, _I, _I, _I64, _I, _P, _P]),
    "csa2_select_topk_workspace_size": (_SZ, [_I, _I, _I64]),
    "csa2_select_topk": (_I, [ctypes.POINTER(CacheStruct), _P, _P, _P, _I, _I, _P, _I, _I, _I64,
                              _P, _SZ, _P]),
    "csa2_attn_workspace_size": (_SZ, [_I, _I, _I]),
    "csa2_sparse_swa_attn": (_I, [ctypes.POINTER(CacheStruct), _P, _P, _I, _P, _P, _I, _P, _F, _P,
                                  _I, _I, _P, _SZ, _P]),
    "csa2_swa_quantize_fp8": (_I, [_P, _I64, _P, _P]),
    "csa2_block_summary": (_I, [ctypes.POINTER(CacheStruct), _P, _I64, _I, _P, _P, _I64, _P, _SZ, _P]),
    "csa2_hisa_blocks_workspace_size": (_SZ, [_I, _I, _I64]),
    "csa2_hisa_blocks": (_I, [ctypes.POINTER(CacheStruct), _P, _P, _I64, _P, _P, _P, _I, _I, _I64, _I, _P,
                              _P, _SZ, _P]),
    "csa2_decode_workspace_size": (_SZ, [_I, _I, _I, _I64, _I, _I]),
    "csa2_decode": (_I, [ctypes.POINTER(CacheStruct), ctypes.POINTER(DecodeArgs), _P, _SZ, _P]),
    "csa2_test_withhold_arrival": (_I, [_I]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcsa2.so; raises if it is missing (no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"CSA2 CUDA library not built: {path} is missing "
                               "(run `python -m fp4_kv_cache_csa2_gb300.build`)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols() -> list[str]:
    return sorted(_SIGNATURES)


def _check(call: str, status: int) -> None:
    if status != 0:
        raise Csa2Error(call, status)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ------------------------------------------------------------------ objects
class Cache:
    """One source layer's global cache in device memory (caller-owned tensors)."""

    def __init__(self, B: int, cap: int, m: int, device="cuda"):
        import torch
        cap = -(-int(cap) // BLOCK) * BLOCK        # the library needs cap % 8 == 0
        self.B, self.cap, self.m = B, cap, m
        self.main_kv = torch.zeros((B, cap, MAIN_ENTRY_BYTES), dtype=torch.uint8, device=device)
        self.idx_codes = torch.zeros((B, cap, INDEX_CODE_BYTES), dtype=torch.uint8, device=device)
        self.idx_scales = torch.zeros((B, cap, INDEX_SCALE_BYTES), dtype=torch.uint8, device=device)
        self.n_entries = torch.zeros((B,), dtype=torch.int32, device=device)

    def struct(self) -> CacheStruct:
        return CacheStruct(self.main_kv.data_ptr(), self.idx_codes.data_ptr(),
                           self.idx_scales.data_ptr(), self.cap, self.n_entries.data_ptr(), self.m)

    def sequence(self, b: int) -> "Cache":
        """Sequence b as a batch-1 cache sharing this cache's memory (for writing
        one sequence, or one chunk of it, at a time)."""
        v = Cache.__new__(Cache)
        v.B, v.cap, v.m = 1, self.cap, self.m
        v.main_kv = self.main_kv[b:b + 1]
        v.idx_codes = self.idx_codes[b:b + 1]
        v.idx_scales = self.idx_scales[b:b + 1]
        v.n_entries = self.n_entries[b:b + 1]
        return v


class Workspace:
    """Device scratch with the status header, initialised on creation."""

    def __init__(self, nbytes: int, device="cuda", stream=None):
        import torch
        nbytes = max(int(nbytes), WS_HEADER_BYTES)
        # 256-byte alignment: torch's caching allocator returns 512-byte aligned blocks
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        assert self.buf.data_ptr() % 256 == 0
        self.nbytes = nbytes
        _check("csa2_workspace_init", load().csa2_workspace_init(self.buf.data_ptr(), nbytes, _stream(stream)))

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def sync_status(self, stream=None) -> tuple[int, int]:
        detail = ctypes.c_int64(0)
        st = load().csa2_sync_status(self.ptr, _stream(stream), ctypes.byref(detail))
        return st, detail.value


# ------------------------------------------------------------------ calls
def rope_table(P: int, theta: float = 160000.0):
    """Host RoPE table [P, 32, 2] float32 (torch CPU tensor)."""
    import torch
    cs = torch.empty((P, 32, 2), dtype=torch.float32)
    _check("csa2_rope_table", load().csa2_rope_table(cs.data_ptr(), P, float(theta)))
    return cs


def compress_quantize(cache: Cache, x, entry_start, w0, w1, rope_cs, w_idx, ws: Workspace, stream=None):
    B, T = x.shape[0], x.shape[1]
    c = cache.struct()
    _check("csa2_compress_quantize", load().csa2_compress_quantize(
        ctypes.byref(c), _ptr(x), B, T, _ptr(entry_start), _ptr(w0), _ptr(w1), _ptr(rope_cs),
        rope_cs.shape[0], _ptr(w_idx), ws.ptr, ws.nbytes, _stream(stream)))


def index_score(cache: Cache, q_idx, w_head, q_pos, scores, max_n: int, ws: Workspace,
                pool_blocks=None, M: int = 0, stream=None):
    B, Q = q_pos.shape
    c = cache.struct()
    _check("csa2_index_score", load().csa2_index_score(
        ctypes.byref(c), _ptr(q_idx), _ptr(w_head), _ptr(q_pos), _ptr(pool_blocks), M, _ptr(scores),
        B, Q, max_n, ws.ptr, ws.nbytes, _stream(stream)))


def block_topk_workspace_size(B: int, Q: int, max_n: int) -> int:
    return load().csa2_block_topk_workspace_size(B, Q, max_n)


def block_topk(cache: Cache, scores, q_pos, max_n: int, M: int, pool_blocks, ws: Workspace, stream=None):
    B, Q = q_pos.shape
    c = cache.struct()
    _check("csa2_block_topk", load().csa2_block_topk(
        ctypes.byref(c), _ptr(scores), _ptr(q_pos), B, Q, max_n, M, _ptr(pool_blocks), ws.ptr,
        ws.nbytes, _stream(stream)))


def block_topk_static(cache: Cache, scores, q_pos, max_n: int, M: int, pool_blocks, stream=None) -> int:
    """Candidate blocks without a workspace (library-held 4 MiB scratch); returns
    the status code (CSA2_ERR_WORKSPACE = 3 when the request exceeds the scratch)."""
    B, Q = q_pos.shape
    c = cache.struct()
    return load().csa2_block_topk_static(ctypes.byref(c), _ptr(scores), _ptr(q_pos), B, Q, max_n, M,
                                         _ptr(pool_blocks), _stream(stream))


def select_topk_workspace_size(B: int, Q: int, max_n: int) -> int:
    return load().csa2_select_topk_workspace_size(B, Q, max_n)


def select_topk(cache: Cache, scores, q_pos, K: int, sel, max_n: int, ws: Workspace,
                pool_blocks=None, M: int = 0, stream=None):
    B, Q = q_pos.shape
    c = cache.struct()
    _check("csa2_select_topk", load().csa2_select_topk(
        ctypes.byref(c), _ptr(scores), _ptr(q_pos), _ptr(pool_blocks), M, K, _ptr(sel), B, Q, max_n,
        ws.ptr, ws.nbytes, _stream(stream)))


def attn_workspace_size(B: int, Q: int, K: int) -> int:
    return load().csa2_attn_workspace_size(B, Q, K)


def sparse_swa_attn(cache: Cache, q, sel, swa, swa_base_pos, q_pos, scale: float, out, ws: Workspace,
                    stream=None):
    B, Q = q_pos.shape
    K = 0 if sel is None else sel.shape[-1]
    c = cache.struct()
    _check("csa2_sparse_swa_attn", load().csa2_sparse_swa_attn(
        ctypes.byref(c), _ptr(q), _ptr(sel), K, _ptr(swa), _ptr(swa_base_pos), swa.shape[1], _ptr(q_pos),
        float(scale), _ptr(out), B, Q, ws.ptr, ws.nbytes, _stream(stream)))


class BlockSummaries:
    """HISA summary store of a cache: one MXFP4 key per block of 8 entries
    (caller-owned tensors, [B][sum_cap][64] codes and [B][sum_cap][4] scales)."""

    def __init__(self, cache: Cache, device="cuda"):
        import torch
        self.B = cache.B
        rows = -(-cache.cap // BLOCK)                 # one row per block
        self.sum_cap = -(-rows // BLOCK) * BLOCK      # the library needs sum_cap % 8 == 0
        self.codes = torch.zeros((cache.B, self.sum_cap, INDEX_CODE_BYTES), dtype=torch.uint8, device=device)
        self.scales = torch.zeros((cache.B, self.sum_cap, INDEX_SCALE_BYTES), dtype=torch.uint8, device=device)


def block_summary(cache: Cache, summaries: BlockSummaries, first_block, n_blocks: int, ws: Workspace,
                  stream=None):
    """Recompute blocks first_block[b] .. first_block[b] + n_blocks - 1 of every sequence."""
    c = cache.struct()
    _check("csa2_block_summary", load().csa2_block_summary(
        ctypes.byref(c), _ptr(first_block), n_blocks, cache.B, _ptr(summaries.codes), _ptr(summaries.scales),
        summaries.sum_cap, ws.ptr, ws.nbytes, _stream(stream)))


def swa_quantize_fp8(x, out, stream=None):
    """FP8 window rows: out (uint8 [..., 512]) = E4M3 of x (bf16 as int16, same shape)."""
    n_rows = x.numel() // D_LATENT
    assert out.numel() == x.numel()
    _check("csa2_swa_quantize_fp8", load().csa2_swa_quantize_fp8(_ptr(x), n_rows, _ptr(out), _stream(stream)))


def hisa_blocks_workspace_size(B: int, Q: int, max_n: int) -> int:
    return load().csa2_hisa_blocks_workspace_size(B, Q, max_n)


def hisa_blocks(cache: Cache, summaries: BlockSummaries, q_idx, w_head, q_pos, max_n: int, M: int, pool_blocks,
                ws: Workspace, stream=None):
    B, Q = q_pos.shape
    c = cache.struct()
    _check("csa2_hisa_blocks", load().csa2_hisa_blocks(
        ctypes.byref(c), _ptr(summaries.codes), _ptr(summaries.scales), summaries.sum_cap, _ptr(q_idx),
        _ptr(w_head), _ptr(q_pos), B, Q, max_n, M, _ptr(pool_blocks), ws.ptr, ws.nbytes, _stream(stream)))


def decode_workspace_size(mode: int, B: int, Q: int, max_n: int, M: int, K: int) -> int:
    return load().csa2_decode_workspace_size(mode, B, Q, max_n, M, K)


def decode(mode: int, cache: Cache, *, q_pos, q, swa, swa_base_pos, scale: float, sel, out,
           ws: Workspace, M: int = 0, max_n: int = 0, q_idx=None, w_head=None, pool_blocks=None,
           packed_sel=None, swa_fp8: bool = False, attn_split: int = 0, stream=None):
    """swa: bf16 rows [B][S][512] (as int16), or with swa_fp8 the uint8 rows of
    swa_quantize_fp8.  attn_split: CTAs per query in the attention (0 / 1: one;
    S >= 2 splits the query's key chunks over S CTAs and merges their states)."""
    B, Q = q_pos.shape
    a = DecodeArgs(mode, B, Q, M, sel.shape[-1], swa.shape[1], max_n, float(scale), _ptr(q_pos),
                   _ptr(q), _ptr(q_idx), _ptr(w_head), _ptr(swa), _ptr(swa_base_pos),
                   _ptr(pool_blocks), _ptr(sel), _ptr(out), _ptr(packed_sel), 1 if swa_fp8 else 0,
                   int(attn_split))
    c = cache.struct()
    _check("csa2_decode", load().csa2_decode(ctypes.byref(c), ctypes.byref(a), ws.ptr, ws.nbytes,
                                             _stream(stream)))
