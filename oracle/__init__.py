"""CPU oracle for the CSA2 global-attention layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the package's ``smoke()`` check and the benchmark's CPU-baseline
leg may import this package.  The CUDA library and its Python binding never
import it; the two share no code.  Inputs come from the seeded generators in
``synth``; nothing here consumes an output of the CUDA path.

What it computes (plain, slow, in the order the pages state it):

  cache write     -> ``compress_quantize`` (C, binary32 in a fixed order, see
                     ``cache_write.c``), bytes must match bit for bit
  index score     -> ``index_scores``: s(t,j) = sum_h w_h * ReLU(q_h . k_j), binary64,
                     q_h MXFP4-quantised like the index keys
  block top-M     -> ``block_topm``: g_r = max over blocks of 8 (last block padded
                     with -inf), newest visible block forced to +inf, top-M blocks
  HISA variant    -> ``block_summary`` (mean index key per block of 8, MXFP4) and
                     ``hisa_blocks`` (top-M blocks by the score of their mean key)
  top-K           -> ``select_topk``: Full over all visible entries, Reindex over
                     the candidate pool only; order (score desc, index asc)
  attention       -> ``attention``: one softmax over [selected main-KV entries ||
                     SWA window], K = V = the shared 512-d latent, binary64
  FP8 window      -> ``swa_fp8_quantize`` (every window value to E4M3 on its own);
                     ``attention`` takes such rows (uint8) in place of bf16 rows
  modes           -> ``decode``: Full / Reindex / Reuse composition

Sources (web pages about DeepSeek-V4.1-Flash):
  [zartbot]  "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致": §2.3.2 modes,
             §2.3.4 HSI (block max, forced newest block, pool bitmap),
             §3.2 mode access table, §3.3.1-3.3.2 joint sparse+SWA readout with
             key = value.
  [dilfish]  "4. 层维度(下):CSA2 与每 token 890 字节": §4.2 compressor, §4.3 modes and
             layer schedule, §4.4 entry sizes and 890 B/token, §4.5 FP4 range,
             §4.6 3514 -> 890 steps, §4.7 HSI formulas g_r, TopM, P_t.

Parity of each function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

from . import native
from .native import ptr

D = 512            # shared latent (key = value), last 64 dims carry RoPE
D_ROPE = 64
H_MAIN = 64        # main query heads
H_IDX = 32         # index heads
D_IDX = 128        # index head dim
BLOCK = 8          # candidate_block_size
WINDOW = 128       # SWA window
MAIN_ENTRY = 288   # 256 B E2M1 codes + 32 B E4M3 scales
IDX_CODES = 64
IDX_SCALES = 4
ROPE_THETA = 160000.0


# ------------------------------------------------------------ accounting
def entry_bytes(d: int, group: int) -> float:
    """b(D, G) = D/2 (4-bit payload) + D/G (one scale byte per group). [dilfish §4.4]"""
    return d / 2 + d / group


def global_bytes_per_token(ratios) -> float:
    """Sum over source layers of (main + index entry bytes) / m. [dilfish §4.4]"""
    per_entry = entry_bytes(D, 16) + entry_bytes(D_IDX, 32)
    return sum(per_entry / m for m in ratios)


def v4flash_bytes_per_token() -> float:
    """DeepSeek-V4-Flash global KV per token: 21 CSA layers at m=4 with index K,
    20 HCA layers at m=128 without; 584 B main entries, 68 B index entries.
    [dilfish §4.6]"""
    main_v4 = 448 * 1 + 64 * 2 + 8
    return 21 * (main_v4 + 68) / 4 + 20 * main_v4 / 128


# ------------------------------------------------------------ formats
def e2m1_values() -> np.ndarray:
    """Value of each 4-bit E2M1 code (sign bit 3, exponent bits 2:1 with bias 1,
    mantissa bit 0; exponent 0 is subnormal: 0.5 * mantissa)."""
    out = np.zeros(16)
    for code in range(16):
        e, m = (code >> 1) & 3, code & 1
        mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        out[code] = -mag if code & 8 else mag
    return out


def e4m3_values() -> np.ndarray:
    """Value of each E4M3 byte (bias 7; exponent 0 subnormal m * 2^-9; 0x7F and
    0xFF are NaN)."""
    out = np.zeros(256)
    for code in range(256):
        e, m = (code >> 3) & 15, code & 7
        mag = m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8)
        if (code & 0x7F) == 0x7F:
            mag = np.nan
        out[code] = -mag if code & 0x80 else mag
    return out


_E2M1 = e2m1_values()
_E4M3 = e4m3_values()


def _unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., nbytes] -> [..., 2*nbytes] codes; element 2k is the low nibble of byte k."""
    lo = codes & 0x0F
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)


def dequant_main(entries: np.ndarray) -> np.ndarray:
    """Main-KV entries [..., 288] -> binary64 latents [..., 512] (exact)."""
    codes = _unpack_nibbles(entries[..., :256])
    scales = _E4M3[entries[..., 256:288]]
    return _E2M1[codes] * np.repeat(scales, 16, axis=-1)


def dequant_index(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP4 rows: codes [..., 64], E8M0 scales [..., 4] -> binary64 [..., 128]."""
    vals = _E2M1[_unpack_nibbles(codes)]
    return vals * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)


def mxfp4_quantize(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Rows of 128 binary32 values -> (codes [..., 64], scales [..., 4]) by the
    OCP MX rule (C implementation, shared by index K and indexer queries)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    lead = v.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    codes = np.zeros((n, IDX_CODES), np.uint8)
    scales = np.zeros((n, IDX_SCALES), np.uint8)
    native.lib().oracle_mxfp4_rows(ptr(v), n, ptr(codes), ptr(scales))
    return codes.reshape(*lead, IDX_CODES), scales.reshape(*lead, IDX_SCALES)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ cache write
def rope_table(P: int, theta: float = ROPE_THETA) -> np.ndarray:
    """cos/sin of p * theta^(-2i/64) for p < P, i < 32, binary32 [P, 32, 2]."""
    cs = np.zeros((P, 32, 2), np.float32)
    native.lib().oracle_rope_table(P, float(theta), ptr(cs))
    return cs


def compress_quantize(x: np.ndarray, m: int, w0: np.ndarray, w1: np.ndarray,
                      w_idx: np.ndarray, entry0: int = 0, theta: float = ROPE_THETA,
                      cs: np.ndarray | None = None):
    """Cache write for one sequence chunk.

    x bf16 bits [T, 512] (T even when m = 2), w0/w1 float32 [512], w_idx bf16 bits
    [128, 512].  Entry j (0-based) pools tokens (2j, 2j+1) for m = 2 and is token j
    for m = 1; its RoPE position is ``entry0 + j``.  Returns (main_kv [T/m, 288],
    idx_codes [T/m, 64], idx_scales [T/m, 4]).  [dilfish §4.2, §4.4; zartbot §2.4.4]
    """
    x = np.ascontiguousarray(x, np.uint16)
    T = x.shape[0]
    assert m in (1, 2) and T % m == 0
    n = T // m
    if cs is None:
        cs = rope_table(entry0 + n, theta)
    assert cs.shape[0] >= entry0 + n
    main = np.zeros((n, MAIN_ENTRY), np.uint8)
    codes = np.zeros((n, IDX_CODES), np.uint8)
    scales = np.zeros((n, IDX_SCALES), np.uint8)
    native.lib().oracle_compress_quantize(
        ptr(x), T, m, ptr(np.ascontiguousarray(w0, np.float32)),
        ptr(np.ascontiguousarray(w1, np.float32)), ptr(np.ascontiguousarray(w_idx, np.uint16)),
        entry0, ptr(np.ascontiguousarray(cs, np.float32)), ptr(main), ptr(codes), ptr(scales))
    return main, codes, scales


def entry_stages(x0, x1, m, w0, w1, cs_row, w_idx):
    """Binary32 intermediates of one entry: (compressed, normalised, rotated, index K)."""
    c = np.zeros(D, np.float32)
    yn = np.zeros(D, np.float32)
    yr = np.zeros(D, np.float32)
    k = np.zeros(D_IDX, np.float32)
    x0 = np.ascontiguousarray(x0, np.uint16)
    x1 = np.ascontiguousarray(x1 if x1 is not None else x0, np.uint16)
    native.lib().oracle_entry_stages(
        ptr(x0), ptr(x1), m, ptr(np.ascontiguousarray(w0, np.float32)),
        ptr(np.ascontiguousarray(w1, np.float32)),
        ptr(np.ascontiguousarray(cs_row, np.float32)),
        ptr(np.ascontiguousarray(w_idx, np.uint16)), ptr(c), ptr(yn), ptr(yr), ptr(k))
    return c, yn, yr, k


# ------------------------------------------------------------ indexer
def visible_entries(t: int, m: int, n_entries: int) -> int:
    """Entries a query at raw position t may see: min(n_entries, floor((t+1)/m)).
    A compressed entry is published once both of its tokens exist (causality)."""
    return min(int(n_entries), (int(t) + 1) // m)


def quantize_index_query(q_idx: np.ndarray) -> np.ndarray:
    """Indexer query heads (bf16 bits [..., 32, 128]) -> MXFP4 round trip, binary64.
    FP4 indexer Q and K follow the same format (zartbot §2.4.4: FP4 indexer Q/K)."""
    v = (np.ascontiguousarray(q_idx, np.uint16).astype(np.uint32) << 16).view(np.float32)
    codes, scales = mxfp4_quantize(v)
    return dequant_index(codes, scales)


def index_scores(q_idx: np.ndarray, w_head: np.ndarray, idx_codes: np.ndarray,
                 idx_scales: np.ndarray, entries: np.ndarray | None = None) -> np.ndarray:
    """Scores of one query against index-K entries.

    s(t, j) = sum_h w_h * max(0, q_h . k_j) in binary64, with q_h the MXFP4 round
    trip of the bf16 query and k_j the dequantised MXFP4 key.  ``entries`` lists
    the entry indices to score (default: all rows).  [zartbot §3.3.2 Top-K
    selection set; spec reading of the lost formula]
    """
    qd = quantize_index_query(q_idx)                     # [32, 128]
    w = np.asarray(w_head, np.float64)                   # [32]
    if entries is None:
        entries = np.arange(idx_codes.shape[0])
    out = np.empty(len(entries))
    step = 65536
    for a in range(0, len(entries), step):
        e = entries[a:a + step]
        kd = dequant_index(idx_codes[e], idx_scales[e])  # [n, 128]
        dots = kd @ qd.T                                 # [n, 32]
        out[a:a + step] = np.maximum(dots, 0.0) @ w
    return out


def block_topm(scores: np.ndarray, n_visible: int, M: int) -> np.ndarray:
    """HSI candidate blocks for one query.  [dilfish §4.7; zartbot §2.3.4]

    g_r = max of the scores in block r = [8r, 8r+8) over visible entries (the last
    block is padded with -inf), the block holding entry n_visible-1 gets +inf, and
    the M blocks with the largest g (ties: lower block id) are kept.  Returns the
    block ids sorted ascending, padded with -1 to length M.
    """
    out = np.full(M, -1, np.int32)
    nv = int(n_visible)
    if nv <= 0:
        return out
    nb = (nv + BLOCK - 1) // BLOCK
    padded = np.full(nb * BLOCK, -np.inf)
    padded[:nv] = scores[:nv]
    g = padded.reshape(nb, BLOCK).max(axis=1)
    g[(nv - 1) // BLOCK] = np.inf
    order = np.lexsort((np.arange(nb), -g))
    chosen = np.sort(order[:M])
    out[:len(chosen)] = chosen
    return out


def block_summary(idx_codes: np.ndarray, idx_scales: np.ndarray, n: int):
    """HISA block summaries of the first n index-K entries.  [zartbot §2.3.4,
    the HISA paragraph: every block of consecutive positions keeps the mean of
    its indexer keys, a decode step updating only the newest block]

    Block r covers entries [8r, min(8r + 8, n)).  Its mean key is computed in
    binary32: the dequantised keys (exact in binary32) are added in entry order
    starting from +0, and the sum is divided by the number of entries in the
    block; the mean is then stored as MXFP4 like every index key.  Returns
    (codes [nb, 64], scales [nb, 4]) with nb = ceil(n / 8).
    """
    n = int(n)
    nb = (n + BLOCK - 1) // BLOCK
    kd = np.zeros((nb * BLOCK, D_IDX), np.float32)
    kd[:n] = dequant_index(idx_codes[:n], idx_scales[:n]).astype(np.float32)   # exact
    kd = kd.reshape(nb, BLOCK, D_IDX)
    acc = np.zeros((nb, D_IDX), np.float32)
    for p in range(BLOCK):                               # entry order; absent entries add +0
        acc = acc + kd[:, p]
    count = np.minimum(BLOCK, n - BLOCK * np.arange(nb)).astype(np.float32)
    mean = acc / count[:, None]
    return mxfp4_quantize(mean)


def hisa_blocks(q_idx: np.ndarray, w_head: np.ndarray, sum_codes: np.ndarray,
                sum_scales: np.ndarray, n_visible: int, M: int) -> np.ndarray:
    """HISA first stage for one query: the indexer score of every block that
    holds a visible entry, computed on the block's mean key (the same
    s = sum_h w_h ReLU(q_h . k)), and the M best blocks by (score desc, block
    asc), returned ascending and -1 padded.  No block is forced in (the forced
    newest block is HSI's boundary rule).  The second stage scores the chosen
    blocks' visible entries, as a Reindex layer does over its pool.  [zartbot
    §2.3.4, the HISA paragraph]
    """
    nv = int(n_visible)
    nb = (nv + BLOCK - 1) // BLOCK
    if nb == 0:
        return np.full(M, -1, np.int32)
    g = index_scores(q_idx, w_head, sum_codes[:nb], sum_scales[:nb])
    return select_topk(g, np.arange(nb), M)


def pool_entries(blocks: np.ndarray, n_visible: int) -> np.ndarray:
    """Candidate pool: every visible entry of the chosen blocks (bitmap expansion
    limited to the visible width).  [zartbot §2.3.4]"""
    b = blocks[blocks >= 0].astype(np.int64)
    ent = (b[:, None] * BLOCK + np.arange(BLOCK)[None, :]).ravel()
    return np.sort(ent[ent < int(n_visible)])


def select_topk(scores: np.ndarray, domain: np.ndarray, K: int) -> np.ndarray:
    """Top-K of ``scores`` over the entry ids in ``domain`` by (score desc, id
    asc); returns the ids sorted ascending, padded with -1 to length K."""
    out = np.full(K, -1, np.int32)
    domain = np.asarray(domain, np.int64)
    if len(domain) == 0:
        return out
    s = np.asarray(scores, np.float64)[domain]
    order = np.lexsort((domain, -s))
    chosen = np.sort(domain[order[:K]])
    out[:len(chosen)] = chosen
    return out


# ------------------------------------------------------------ attention
def swa_fp8_quantize(swa_bits: np.ndarray) -> np.ndarray:
    """FP8 SWA rows: every bf16 window value rounded to E4M3 on its own (nearest,
    ties to the even code, saturating at +-448, no scale factor).  The pages say
    only that the quantisation-sensitive SWA KV keeps FP8 precision while the
    main KV drops to FP4; E4M3 covers the latent's range (RMS 1 after the norm,
    largest values near 10) without a scale.  [zartbot §2.4.4; sarnas, the FP4
    cache paragraph]  bf16 bits [..., 512] -> uint8 [..., 512]."""
    v = bf16_to_f64(np.asarray(swa_bits)).astype(np.float32)         # exact
    out = np.zeros(v.shape, np.uint8)
    v = np.ascontiguousarray(v)
    native.lib().oracle_e4m3_encode_rows(ptr(v), v.size, ptr(out))
    return out


def window_positions(t: int) -> np.ndarray:
    """Raw positions of the SWA window of a query at raw position t (self included)."""
    return np.arange(max(0, int(t) - WINDOW + 1), int(t) + 1)


def attention(q: np.ndarray, sel: np.ndarray, main_kv: np.ndarray, swa: np.ndarray,
              swa_base: int, t: int, scale: float) -> np.ndarray:
    """Joint sparse + SWA attention of one query token, binary64.

    Keys and values are the same vectors (K = V = the shared latent): the
    dequantised main-KV entries listed in ``sel`` (ids >= 0) followed by the SWA
    rows of the window [max(0, t-127), t] (row = position - swa_base): bf16 bits
    (uint16) or FP8 rows from ``swa_fp8_quantize`` (uint8, E4M3 values).  One
    softmax of scale * q_h . v_i over all of them; o_h = sum_i p_hi v_i.
    q bf16 bits [64, 512]; returns binary64 [64, 512].  [zartbot §3.3.2 readout
    of SWA and selected main KV in one sparse attention; §3.3.2.1 key = value]
    """
    ids = np.asarray(sel)
    ids = ids[ids >= 0].astype(np.int64)
    keys = [dequant_main(main_kv[ids])] if len(ids) else []
    rows = window_positions(t) - int(swa_base)
    keys.append(_E4M3[swa[rows]] if swa.dtype == np.uint8 else bf16_to_f64(swa[rows]))
    V = np.concatenate(keys, axis=0)                    # [n_keys, 512]
    qd = bf16_to_f64(q)                                 # [64, 512]
    logits = (qd @ V.T) * scale                         # [64, n_keys]
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return p @ V


# ------------------------------------------------------------ modes
FULL, REINDEX, REUSE = 0, 1, 2


def decode_query(mode: int, *, t: int, m: int, n_entries: int, main_kv, idx_codes,
                 idx_scales, q, swa, swa_base, scale, M, K, q_idx=None, w_head=None,
                 pool_blocks=None, sel=None):
    """One query token of one CSA2 layer in the given mode.  [zartbot §3.2 access
    table; dilfish §4.3]

      Full:    score every visible entry, build the candidate pool (top-M blocks)
               and its own top-K over all visible entries, attend.
      Reindex: score only the pool's visible entries with its own index query,
               top-K inside the pool, attend.
      Reuse:   attend with the given selection.
    Returns (pool_blocks, sel, out binary64 [64, 512]).
    """
    nv = visible_entries(t, m, n_entries)
    if mode == FULL:
        s = index_scores(q_idx, w_head, idx_codes[:nv], idx_scales[:nv])
        pool_blocks = block_topm(s, nv, M)
        sel = select_topk(s, np.arange(nv), K)
    elif mode == REINDEX:
        dom = pool_entries(pool_blocks, nv)
        s_dom = index_scores(q_idx, w_head, idx_codes, idx_scales, dom)
        s = np.full(max(nv, 1), -np.inf)
        s[dom] = s_dom
        sel = select_topk(s, dom, K)
    elif mode != REUSE:
        raise ValueError(mode)
    out = attention(q, sel, main_kv, swa, swa_base, t, scale)
    return pool_blocks, sel, out
