"""GPU parity of the HISA variant of the indexer's first stage: block summary
keys (bit-exact against the oracle) and the top-M blocks by summary score
(equal to the oracle's up to ties inside its 1e-4 relative window), then the
Reindex second stage over those blocks."""
import numpy as np
import pytest

import oracle
import synth
from tests import cases
from tests.test_gpu_parity import DEV, GpuLayer, dev, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_kv_cache_csa2_gb300 as m
    m.load()
    return m


class _Store:
    """A summary store with a chosen number of rows (the binding's layout)."""

    def __init__(self, B, sum_cap, fill=0xAB):
        self.B, self.sum_cap = B, sum_cap
        self.codes = torch.full((B, sum_cap, 64), fill, dtype=torch.uint8, device=DEV)
        self.scales = torch.full((B, sum_cap, 4), fill, dtype=torch.uint8, device=DEV)


def _random_cache(csa2, B, n, seed, m=1):
    """An index cache of n random MXFP4 keys per sequence (no cache write)."""
    g = synth.rng(seed)
    codes, scales = synth.index_key_bytes(g, B, n)
    cache = csa2.Cache(B, n, m, device=DEV)
    cache.idx_codes[:, :n] = dev(codes)
    cache.idx_scales[:, :n] = dev(scales)
    cache.n_entries.fill_(n)
    return cache, codes, scales, g


@pytest.mark.parametrize("n,B", [(1000, 2), (8 * 37 + 5, 1), (3, 2), (8 * 64, 1)])
def test_block_summary_bit_exact(csa2, n, B):
    """Every block of a ragged cache, and rows past the last block untouched."""
    cache, codes, scales, _ = _random_cache(csa2, B, n, seed=700 + n)
    rows = -(-cache.cap // 8)
    store = _Store(B, -(-rows // 8) * 8 + 8)
    ws = csa2.Workspace(1 << 16, device=DEV)
    nb = -(-n // 8)
    first = torch.zeros(B, dtype=torch.int64, device=DEV)
    csa2.block_summary(cache, store, first, nb + 3, ws)
    got_c, got_s = host(store.codes), host(store.scales)
    for b in range(B):
        want_c, want_s = oracle.block_summary(codes[b], scales[b], n)
        np.testing.assert_array_equal(got_c[b, :nb], want_c)
        np.testing.assert_array_equal(got_s[b, :nb], want_s)
        assert np.all(got_c[b, nb:] == 0xAB) and np.all(got_s[b, nb:] == 0xAB)
    assert ws.sync_status()[0] == 0


def test_block_summary_of_written_cache_bit_exact(csa2):
    """Summaries of keys produced by the cache write (m = 2, ragged)."""
    case = cases.make_case(B=2, T=2 * 611, m=2, Q=1, M=8, K=8, seed=711)
    L = GpuLayer(csa2, case)
    _, codes, scales = cases.oracle_cache(case)
    n = case.n_entries
    np.testing.assert_array_equal(host(L.cache.idx_codes)[:, :n], codes)   # the cache write is exact
    store = csa2.BlockSummaries(L.cache, device=DEV)
    first = torch.zeros(2, dtype=torch.int64, device=DEV)
    csa2.block_summary(L.cache, store, first, -(-n // 8), L.ws)
    for b in range(2):
        want_c, want_s = oracle.block_summary(codes[b], scales[b], n)
        np.testing.assert_array_equal(host(store.codes)[b, :len(want_c)], want_c)
        np.testing.assert_array_equal(host(store.scales)[b, :len(want_s)], want_s)
    assert L.ws.sync_status()[0] == 0


def test_block_summary_newest_block_update(csa2):
    """A decode step: entries appended to the newest block, only that block
    recomputed; the store then equals the oracle's summaries of the longer
    cache.  Sequences of different lengths, one first block per sequence."""
    n_full = np.array([8 * 50 + 5, 8 * 20 + 7])
    cache, codes, scales, _ = _random_cache(csa2, 2, int(n_full.max()), seed=720)
    cache.n_entries.copy_(torch.from_numpy((n_full - 3).astype(np.int32)))
    store = csa2.BlockSummaries(cache, device=DEV)
    ws = csa2.Workspace(1 << 16, device=DEV)
    csa2.block_summary(cache, store, torch.zeros(2, dtype=torch.int64, device=DEV), 64, ws)
    cache.n_entries.copy_(torch.from_numpy(n_full.astype(np.int32)))
    newest = torch.from_numpy((n_full - 1) // 8).to(DEV)
    csa2.block_summary(cache, store, newest, 1, ws)
    for b in range(2):
        want_c, want_s = oracle.block_summary(codes[b], scales[b], int(n_full[b]))
        np.testing.assert_array_equal(host(store.codes)[b, :len(want_c)], want_c)
        np.testing.assert_array_equal(host(store.scales)[b, :len(want_s)], want_s)
    assert ws.sync_status()[0] == 0


def test_block_summary_rows_past_the_store_report_bounds(csa2):
    cache, codes, scales, _ = _random_cache(csa2, 1, 8 * 20, seed=730)
    store = _Store(1, 8)
    ws = csa2.Workspace(1 << 16, device=DEV)
    csa2.block_summary(cache, store, torch.zeros(1, dtype=torch.int64, device=DEV), 20, ws)
    st, detail = ws.sync_status()
    assert st == 6 and 8 <= detail < 20
    want_c, want_s = oracle.block_summary(codes[0], scales[0], 64)
    np.testing.assert_array_equal(host(store.codes)[0], want_c)             # rows inside were written
    np.testing.assert_array_equal(host(store.scales)[0], want_s)


def test_block_summary_argument_errors(csa2):
    cache, _, _, _ = _random_cache(csa2, 1, 128, seed=731)                   # 16 summary rows
    ws = csa2.Workspace(1 << 16, device=DEV)
    bad = _Store(1, 12)                                                      # sum_cap % 8 != 0
    with pytest.raises(csa2.Csa2Error):
        csa2.block_summary(cache, bad, torch.zeros(1, dtype=torch.int64, device=DEV), 1, ws)
    small = _Store(1, 8)
    q_idx = torch.zeros((1, 1, 32, 128), dtype=torch.int16, device=DEV)
    w = torch.zeros((1, 1, 32), device=DEV)
    pos = torch.zeros((1, 1), dtype=torch.int64, device=DEV)
    pool = torch.empty((1, 1, 4), dtype=torch.int32, device=DEV)
    ws2 = csa2.Workspace(csa2.hisa_blocks_workspace_size(1, 1, 64), device=DEV)
    with pytest.raises(csa2.Csa2Error):                                      # store shorter than the cache
        csa2.hisa_blocks(cache, small, q_idx, w, pos, 64, 4, pool, ws2)


def _summary_scores(q_idx, w_head, sc, ss, nb):
    return oracle.index_scores(q_idx, w_head, sc[:nb], ss[:nb])


def _check_hisa(got_pool, case_q_idx, case_w, sc, ss, nv, M, what):
    nb = -(-nv // 8)
    if nb == 0:
        assert np.all(got_pool == -1), what
        return
    want = oracle.hisa_blocks(case_q_idx, case_w, sc, ss, nv, M)
    g = _summary_scores(case_q_idx, case_w, sc, ss, nb)
    cases.assert_set_within_tie_window(got_pool, want, lambda r: g[r], what=what)
    ids = got_pool[got_pool >= 0]
    assert np.all(np.diff(ids) > 0), what
    assert np.all(got_pool[len(ids):] == -1), what
    assert len(ids) == min(M, nb), what


@pytest.mark.parametrize("M", [16, 100, 2048])
def test_hisa_blocks_match_oracle(csa2, M):
    """Short summary rows (one CTA per query): queries that see nothing, one
    entry, a ragged last block and everything; M above the visible block count
    for the early queries (and for all of them at M = 2048)."""
    B, Q, n = 2, 5, 4000
    cache, codes, scales, g = _random_cache(csa2, B, n, seed=740 + M)
    q_pos = np.array([[3999, 2500, 0, 13, 1234], [-1, 3999, 3000, 7, 800]], np.int64)
    q_idx = synth.index_queries(g, B, Q)
    w_head = synth.head_weights(g, B, Q)
    store = csa2.BlockSummaries(cache, device=DEV)
    ws = csa2.Workspace(csa2.hisa_blocks_workspace_size(B, Q, n), device=DEV)
    csa2.block_summary(cache, store, torch.zeros(B, dtype=torch.int64, device=DEV), -(-n // 8), ws)
    pool = torch.empty((B, Q, M), dtype=torch.int32, device=DEV)
    csa2.hisa_blocks(cache, store, dev(q_idx), dev(w_head), dev(q_pos), n, M, pool, ws)
    got = host(pool)
    for b in range(B):
        sc, ss = oracle.block_summary(codes[b], scales[b], n)
        for qi in range(Q):
            nv = oracle.visible_entries(q_pos[b, qi], 1, n)
            _check_hisa(got[b, qi], q_idx[b, qi], w_head[b, qi], sc, ss, nv, M, f"b{b} q{qi}")
    assert ws.sync_status()[0] == 0


def test_hisa_blocks_long_rows_match_oracle(csa2):
    """Summary rows longer than 4,096 blocks (over 32,768 entries) take the
    multi-CTA row selection; m = 2 visibility, rows of 20,001 and 17,501
    blocks."""
    B, Q, n, M = 1, 3, 8 * 20000 + 3, 2048
    cache, codes, scales, g = _random_cache(csa2, B, n, seed=760, m=2)
    q_pos = np.array([[2 * n - 1, 2 * n - 6, 2 * 140000 + 1]], np.int64)
    q_idx = synth.index_queries(g, B, Q)
    w_head = synth.head_weights(g, B, Q)
    store = csa2.BlockSummaries(cache, device=DEV)
    ws = csa2.Workspace(csa2.hisa_blocks_workspace_size(B, Q, n), device=DEV)
    csa2.block_summary(cache, store, torch.zeros(B, dtype=torch.int64, device=DEV), -(-n // 8), ws)
    pool = torch.empty((B, Q, M), dtype=torch.int32, device=DEV)
    csa2.hisa_blocks(cache, store, dev(q_idx), dev(w_head), dev(q_pos), n, M, pool, ws)
    got = host(pool)
    sc, ss = oracle.block_summary(codes[0], scales[0], n)
    for qi in range(Q):
        nv = oracle.visible_entries(q_pos[0, qi], 2, n)
        _check_hisa(got[0, qi], q_idx[0, qi], w_head[0, qi], sc, ss, nv, M, f"q{qi}")
    assert ws.sync_status()[0] == 0


def test_hisa_then_reindex_selects_inside_the_blocks(csa2):
    """Both HISA stages on a written cache: the blocks of the first stage, then
    a Reindex call over them; its top-K equals the oracle's top-K of the
    entries of those blocks, and the attention output matches."""
    case = cases.make_case(B=1, T=2 * 3000, m=2, Q=2, M=64, K=128, seed=770,
                           q_pos=np.array([[5999, 4001]]))
    L = GpuLayer(csa2, case)
    main, codes, scales = cases.oracle_cache(case)
    n = case.n_entries
    store = csa2.BlockSummaries(L.cache, device=DEV)
    hws = csa2.Workspace(csa2.hisa_blocks_workspace_size(1, 2, n), device=DEV)
    csa2.block_summary(L.cache, store, torch.zeros(1, dtype=torch.int64, device=DEV), -(-n // 8), hws)
    pool = torch.empty((1, 2, case.M), dtype=torch.int32, device=DEV)
    csa2.hisa_blocks(L.cache, store, L.q_idx, L.w_head, L.q_pos, n, case.M, pool, hws)
    sc, ss = oracle.block_summary(codes[0], scales[0], n)
    got_pool = host(pool)
    for qi in range(2):
        nv = oracle.visible_entries(case.q_pos[0, qi], 2, n)
        _check_hisa(got_pool[0, qi], case.q_idx[0, qi], case.w_head[0, qi], sc, ss, nv, case.M, f"q{qi}")
    sel = torch.empty((1, 2, case.K), dtype=torch.int32, device=DEV)
    out = torch.empty((1, 2, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_REINDEX, 1, 2, n, case.M, case.K), device=DEV)
    csa2.decode(csa2.MODE_REINDEX, L.cache, q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base,
                scale=case.scale, sel=sel, out=out, ws=ws, q_idx=L.q_idx, w_head=L.w_head, pool_blocks=pool,
                M=case.M, max_n=n)
    got_sel = host(sel)
    got_out = (host(out).astype(np.uint32) << 16).view(np.float32)
    for qi in range(2):
        nv = oracle.visible_entries(case.q_pos[0, qi], 2, n)
        ent = oracle.pool_entries(got_pool[0, qi], nv)
        s_full = np.full(nv, -np.inf)
        s_full[ent] = oracle.index_scores(case.q_idx[0, qi], case.w_head[0, qi], codes[0], scales[0], ent)
        want = oracle.select_topk(s_full, ent, case.K)
        cases.assert_set_within_tie_window(got_sel[0, qi], want, lambda j: s_full[j], what=f"sel q{qi}")
        assert set(got_sel[0, qi][got_sel[0, qi] >= 0]) <= set(ent.tolist())
        want_o = oracle.attention(case.q[0, qi], got_sel[0, qi], main[0], case.swa[0], case.swa_base[0],
                                  case.q_pos[0, qi], case.scale)
        cases.check_attention(got_out[0, qi], want_o, what=f"attn q{qi}")
    assert ws.sync_status()[0] == 0
