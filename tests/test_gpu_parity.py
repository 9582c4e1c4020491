"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Sizes span several CUDA tiles and ragged tails; the oracle finishes each case in
seconds.  Quantised bytes must match bit for bit; index sets may differ only
inside the 1e-4 relative tie window of the oracle's k-th score; attention must
reach rel-L2 <= 1e-2 and max-abs <= 3e-2 against the binary64 oracle."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import cases

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_kv_cache_csa2_gb300 as m
    m.load()
    return m


def dev(a: np.ndarray):
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


def bf16_to_f32(t) -> np.ndarray:
    return (host(t).astype(np.uint32) << 16).view(np.float32)


class GpuLayer:
    """Device copies of a case plus its cache written by the CUDA cache write."""

    def __init__(self, csa2, case: cases.LayerCase, entry0: int = 0, cap: int | None = None):
        self.case = case
        n = case.n_entries
        self.cap = cap if cap is not None else entry0 + n
        self.cache = csa2.Cache(case.B, self.cap, case.m, device=DEV)
        self.ws = csa2.Workspace(1 << 20, device=DEV)
        self.rope = csa2.rope_table(entry0 + n + 8).to(DEV)
        self.entry_start = torch.full((case.B,), entry0, dtype=torch.int64, device=DEV)
        csa2.compress_quantize(self.cache, dev(case.x), self.entry_start, dev(case.w0), dev(case.w1),
                               self.rope, dev(case.w_idx), self.ws)
        self.cache.n_entries.fill_(entry0 + n)
        self.q_pos = dev(case.q_pos)
        self.q_idx = dev(case.q_idx)
        self.w_head = dev(case.w_head)
        self.q = dev(case.q)
        self.swa = dev(case.swa)
        self.swa_base = dev(case.swa_base)
        st, _ = self.ws.sync_status()
        assert st == 0


# ------------------------------------------------------------------ library
def test_library_loads_on_gpu(csa2):
    assert csa2.load().csa2_layout_version() == 1


# ------------------------------------------------------------------ cache write
@pytest.mark.parametrize("m,T,B,entry0", [(2, 2 * 100, 2, 0), (1, 77, 3, 5), (2, 2 * 33, 1, 1000),
                                          (1, 1, 1, 0), (2, 2 * 32, 2, 31)])
def test_cache_write_bit_exact(csa2, m, T, B, entry0):
    case = cases.make_case(B=B, T=T, m=m, Q=1, M=4, K=4, seed=100 + T + m)
    L = GpuLayer(csa2, case, entry0=entry0)
    main, codes, scales = cases.oracle_cache(case, entry0)
    n = case.n_entries
    np.testing.assert_array_equal(host(L.cache.main_kv)[:, entry0:entry0 + n], main)
    np.testing.assert_array_equal(host(L.cache.idx_codes)[:, entry0:entry0 + n], codes)
    np.testing.assert_array_equal(host(L.cache.idx_scales)[:, entry0:entry0 + n], scales)
    # untouched entries stay zero
    assert not host(L.cache.main_kv)[:, :entry0].any()


def test_cache_write_config1_bit_exact(csa2):
    case = cases.config1_case()
    L = GpuLayer(csa2, case)
    main, codes, scales = cases.oracle_cache(case)
    np.testing.assert_array_equal(host(L.cache.main_kv), main)
    np.testing.assert_array_equal(host(L.cache.idx_codes), codes)
    np.testing.assert_array_equal(host(L.cache.idx_scales), scales)
    # 288 + 68 bytes per entry, entries = tokens / 2
    assert main.shape[1] * (main.shape[2] + codes.shape[2] + scales.shape[2]) == 2048 * 356


def test_cache_write_out_of_range_entries_report_bounds(csa2):
    case = cases.make_case(B=1, T=40, m=1, Q=1, M=4, K=4, seed=7)
    cache = csa2.Cache(1, 32, 1, device=DEV)                     # 8 entries do not fit
    ws = csa2.Workspace(1 << 16, device=DEV)
    rope = csa2.rope_table(64).to(DEV)
    start = torch.zeros(1, dtype=torch.int64, device=DEV)
    csa2.compress_quantize(cache, dev(case.x), start, dev(case.w0), dev(case.w1), rope, dev(case.w_idx), ws)
    st, detail = ws.sync_status()
    assert st == 6 and 32 <= detail < 40
    main, _, _ = cases.oracle_cache(case)
    np.testing.assert_array_equal(host(cache.main_kv)[0], main[0, :32])
    assert ws.sync_status()[0] == 0                               # cleared after reading


# ------------------------------------------------------------------ indexer
def _oracle_scores(case, codes, scales, b, qi, entries):
    return oracle.index_scores(case.q_idx[b, qi], case.w_head[b, qi], codes[b], scales[b], entries)


def _score_bound(case, codes, scales, b, qi, entries):
    qd = oracle.quantize_index_query(case.q_idx[b, qi])
    kd = oracle.dequant_index(codes[b][entries], scales[b][entries])
    dots = kd @ qd.T
    return 1e-5 * (np.maximum(dots, 0) @ np.abs(case.w_head[b, qi].astype(np.float64))) + 1e-30


@pytest.mark.parametrize("m,T,B,Q", [(1, 1000, 2, 3), (2, 2 * 2100, 1, 2), (1, 1000, 2, 6), (2, 2 * 1500, 1, 9)])
def test_index_score_all_entries(csa2, m, T, B, Q):
    """Every visible entry of every query; Q >= 4 runs the grouped kernel (four
    queries share each key tile), with a partial last group for Q = 6 and 9."""
    case = cases.make_case(B=B, T=T, m=m, Q=Q, M=8, K=8, seed=200 + T)
    L = GpuLayer(csa2, case)
    max_n = case.n_entries + 3
    scores = torch.full((B, Q, max_n), float("nan"), device=DEV)
    csa2.index_score(L.cache, L.q_idx, L.w_head, L.q_pos, scores, max_n, L.ws)
    got = host(scores)
    _, codes, scales = cases.oracle_cache(case)
    for b in range(B):
        for qi in range(Q):
            nv = oracle.visible_entries(case.q_pos[b, qi], m, case.n_entries)
            ent = np.arange(nv)
            want = _oracle_scores(case, codes, scales, b, qi, ent)
            bound = _score_bound(case, codes, scales, b, qi, ent)
            assert np.all(np.abs(got[b, qi, :nv] - want) <= bound)
            assert np.all(np.isnan(got[b, qi, nv:]))             # invisible columns untouched
    assert L.ws.sync_status()[0] == 0


def test_index_score_grouped_equals_single_query_bit_for_bit(csa2):
    """Scoring four queries per CTA and one query per CTA runs the same head sum
    in the same order, so the scores agree bit for bit."""
    case = cases.make_case(B=1, T=3000, m=1, Q=5, M=8, K=8, seed=251)
    L = GpuLayer(csa2, case)
    max_n = case.n_entries
    grouped = torch.full((1, 5, max_n), float("nan"), device=DEV)
    csa2.index_score(L.cache, L.q_idx, L.w_head, L.q_pos, grouped, max_n, L.ws)
    single = torch.full((1, 5, max_n), float("nan"), device=DEV)
    for qi in range(5):
        csa2.index_score(L.cache, L.q_idx[:, qi:qi + 1].contiguous(), L.w_head[:, qi:qi + 1].contiguous(),
                         L.q_pos[:, qi:qi + 1].contiguous(), single[:, qi:qi + 1], max_n, L.ws)
    a, b = host(grouped), host(single)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    assert np.array_equal(a.view(np.uint32)[~np.isnan(a)], b.view(np.uint32)[~np.isnan(b)])
    assert L.ws.sync_status()[0] == 0


def test_index_score_pool_mode(csa2):
    case = cases.make_case(B=2, T=3000, m=1, Q=2, M=37, K=16, seed=301,
                           q_pos=np.array([[2999, 1500], [2000, 17]]))
    L = GpuLayer(csa2, case)
    g = np.random.default_rng(5)
    M = case.M
    pool = np.full((2, 2, M), -1, np.int32)
    for b in range(2):
        for qi in range(2):
            nb = -(-oracle.visible_entries(case.q_pos[b, qi], 1, 3000) // 8)
            k = min(M - 3, nb)
            pool[b, qi, :k] = np.sort(g.choice(nb, k, replace=False))
    scores = torch.empty((2, 2, M * 8), device=DEV)
    csa2.index_score(L.cache, L.q_idx, L.w_head, L.q_pos, scores, 0, L.ws, pool_blocks=dev(pool), M=M)
    got = host(scores)
    _, codes, scales = cases.oracle_cache(case)
    for b in range(2):
        for qi in range(2):
            nv = oracle.visible_entries(case.q_pos[b, qi], 1, 3000)
            for i in range(M):
                blk = pool[b, qi, i]
                seg = got[b, qi, 8 * i:8 * i + 8]
                if blk < 0:
                    assert np.all(seg == -np.inf)
                    continue
                ent = blk * 8 + np.arange(8)
                vis = ent < nv
                assert np.all(seg[~vis] == -np.inf)
                if vis.any():
                    want = _oracle_scores(case, codes, scales, b, qi, ent[vis])
                    bound = _score_bound(case, codes, scales, b, qi, ent[vis])
                    assert np.all(np.abs(seg[vis] - want) <= bound)


# ------------------------------------------------------------------ selection
def _check_selection_property(sel, scores_f32, domain, K):
    """GPU selection is consistent with the GPU's own scores: ascending, -1
    padded, inside the domain, and every chosen score ranks above every
    non-chosen one under (score desc, id asc)."""
    ids = sel[sel >= 0]
    assert np.all(np.diff(ids) > 0)
    assert np.all(sel[len(ids):] == -1)
    assert len(ids) == min(K, len(domain))
    dom = set(int(x) for x in domain)
    assert set(int(x) for x in ids) <= dom
    if len(ids) < len(domain):
        rest = np.array(sorted(dom - set(int(x) for x in ids)))
        worst = min(ids, key=lambda j: (scores_f32[j], -j))
        best_rest = max(rest, key=lambda j: (scores_f32[j], -j))
        assert (scores_f32[worst], -worst) > (scores_f32[best_rest], -best_rest)


@pytest.mark.parametrize("M,K", [(16, 8), (128, 256), (300, 33)])
def test_block_topk_and_select_full(csa2, M, K):
    case = cases.make_case(B=2, T=2 * 1200, m=2, Q=3, M=M, K=K, seed=400 + M,
                           q_pos=np.array([[2399, 2398, 1500], [2000, 3, 0]]))
    L = GpuLayer(csa2, case)
    max_n = case.n_entries
    scores = torch.empty((2, 3, max_n), device=DEV)
    csa2.index_score(L.cache, L.q_idx, L.w_head, L.q_pos, scores, max_n, L.ws)
    ws = csa2.Workspace(csa2.block_topk_workspace_size(2, 3, max_n), device=DEV)
    pool = torch.empty((2, 3, M), dtype=torch.int32, device=DEV)
    csa2.block_topk(L.cache, scores, L.q_pos, max_n, M, pool, ws)
    sel = torch.empty((2, 3, K), dtype=torch.int32, device=DEV)
    csa2.select_topk(L.cache, scores, L.q_pos, K, sel, max_n, L.ws)
    got_scores, got_pool, got_sel = host(scores), host(pool), host(sel)
    _, codes, scales = cases.oracle_cache(case)
    for b in range(2):
        for qi in range(3):
            nv = oracle.visible_entries(case.q_pos[b, qi], 2, case.n_entries)
            s_or = _oracle_scores(case, codes, scales, b, qi, np.arange(nv))
            want_pool = oracle.block_topm(s_or, nv, M)
            want_sel = oracle.select_topk(s_or, np.arange(nv), K)
            # block maxima of the oracle scores decide the tie window for blocks
            gmax = np.full(max(1, -(-nv // 8)), -np.inf)
            for r in range(len(gmax)):
                gmax[r] = s_or[8 * r:min(8 * r + 8, nv)].max() if nv else -np.inf
            if nv:
                gmax[(nv - 1) // 8] = np.inf
            cases.assert_set_within_tie_window(got_pool[b, qi], want_pool, lambda r: gmax[r], what="pool")
            cases.assert_set_within_tie_window(got_sel[b, qi], want_sel, lambda j: s_or[j], what="sel")
            # property checks on the GPU's own scores
            _check_selection_property(got_sel[b, qi], got_scores[b, qi], np.arange(nv), K)
            nb = -(-nv // 8)
            if nv:
                gg = np.array([got_scores[b, qi, 8 * r:min(8 * r + 8, nv)].max() for r in range(nb)], np.float32)
                gg[(nv - 1) // 8] = np.inf
                _check_selection_property(got_pool[b, qi], gg, np.arange(nb), M)
                assert (nv - 1) // 8 in got_pool[b, qi]
            else:
                assert np.all(got_pool[b, qi] == -1) and np.all(got_sel[b, qi] == -1)


def test_select_topk_pool_mode(csa2):
    case = cases.make_case(B=1, T=5000, m=1, Q=2, M=64, K=100, seed=501,
                           q_pos=np.array([[4999, 2222]]))
    L = GpuLayer(csa2, case)
    M, K = case.M, case.K
    max_n = case.n_entries
    scores = torch.empty((1, 2, max_n), device=DEV)
    csa2.index_score(L.cache, L.q_idx, L.w_head, L.q_pos, scores, max_n, L.ws)
    ws = csa2.Workspace(csa2.block_topk_workspace_size(1, 2, max_n), device=DEV)
    pool = torch.empty((1, 2, M), dtype=torch.int32, device=DEV)
    csa2.block_topk(L.cache, scores, L.q_pos, max_n, M, pool, ws)
    # Reindex-style: fresh index queries score only the pool
    q2 = dev(np.ascontiguousarray(case.q_idx[:, ::-1]))
    pscores = torch.empty((1, 2, M * 8), device=DEV)
    csa2.index_score(L.cache, q2, L.w_head, L.q_pos, pscores, 0, L.ws, pool_blocks=pool, M=M)
    sel = torch.empty((1, 2, K), dtype=torch.int32, device=DEV)
    csa2.select_topk(L.cache, pscores, L.q_pos, K, sel, 0, L.ws, pool_blocks=pool, M=M)
    got_pool, got_sel, got_ps = host(pool), host(sel), host(pscores)
    _, codes, scales = cases.oracle_cache(case)
    qi_rev = case.q_idx[:, ::-1]
    for qi in range(2):
        nv = oracle.visible_entries(case.q_pos[0, qi], 1, max_n)
        dom = oracle.pool_entries(got_pool[0, qi], nv)
        s = np.full(nv, -np.inf)
        s[dom] = oracle.index_scores(qi_rev[0, qi], case.w_head[0, qi], codes[0], scales[0], dom)
        want = oracle.select_topk(s, dom, K)
        cases.assert_set_within_tie_window(got_sel[0, qi], want, lambda j: s[j], what="reindex sel")
        slot_score = {}
        for i, blk in enumerate(got_pool[0, qi]):
            if blk >= 0:
                for r in range(8):
                    if blk * 8 + r < nv:
                        slot_score[blk * 8 + r] = got_ps[0, qi, 8 * i + r]
        arr = np.full(nv, -np.inf, np.float32)
        for j, v in slot_score.items():
            arr[j] = v
        _check_selection_property(got_sel[0, qi], arr, dom, K)


# ------------------------------------------------------------------ attention
def _oracle_attention(case, main, b, qi, sel_row):
    return oracle.attention(case.q[b, qi], sel_row, main[b], case.swa[b], case.swa_base[b],
                            case.q_pos[b, qi], case.scale)


@pytest.mark.parametrize("K,B,Q", [(256, 1, 2), (37, 2, 3), (512, 1, 1), (1, 1, 2)])
def test_sparse_swa_attention(csa2, K, B, Q):
    case = cases.make_case(B=B, T=1500, m=1, Q=Q, M=8, K=K, seed=600 + K)
    L = GpuLayer(csa2, case)
    g = np.random.default_rng(K)
    sel = np.full((B, Q, K), -1, np.int32)
    for b in range(B):
        for qi in range(Q):
            k = max(1, K - 5)
            sel[b, qi, :k] = g.choice(1500, k, replace=False)
    out = torch.empty((B, Q, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.attn_workspace_size(B, Q, K), device=DEV)
    csa2.sparse_swa_attn(L.cache, L.q, dev(sel), L.swa, L.swa_base, L.q_pos, case.scale, out, ws)
    got = bf16_to_f32(out)
    main, _, _ = cases.oracle_cache(case)
    for b in range(B):
        for qi in range(Q):
            cases.check_attention(got[b, qi], _oracle_attention(case, main, b, qi, sel[b, qi]), f"b{b} q{qi}")
    assert ws.sync_status()[0] == 0


def test_attention_window_clipped_at_start_and_no_selection(csa2):
    case = cases.make_case(B=1, T=64, m=2, Q=3, M=4, K=8, seed=700, q_pos=np.array([[0, 5, 63]]))
    L = GpuLayer(csa2, case)
    sel = np.full((1, 3, 8), -1, np.int32)
    sel[0, 2, :3] = [0, 10, 31]
    out = torch.empty((1, 3, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.attn_workspace_size(1, 3, 8), device=DEV)
    csa2.sparse_swa_attn(L.cache, L.q, dev(sel), L.swa, L.swa_base, L.q_pos, case.scale, out, ws)
    got = bf16_to_f32(out)
    main, _, _ = cases.oracle_cache(case)
    # position 0 with nothing selected attends to its own window row only
    np.testing.assert_array_equal(got[0, 0], np.broadcast_to(
        synth_bf16(case.swa[0, 0 - case.swa_base[0]]), (64, 512)))
    for qi in range(3):
        cases.check_attention(got[0, qi], _oracle_attention(case, main, 0, qi, sel[0, qi]))
    assert ws.sync_status()[0] == 0


def test_attention_running_maximum_grows_past_the_rescale_threshold(csa2):
    """Heads whose largest logit arrives in a late chunk of keys: heads 0..15
    point at a key of the last run of 128 selected slots, heads 16..23 at
    (twice) a key of the second run, heads 24..31 away from a key of the first
    run; the rest are random.  The largest logits (about 22 and 45) exceed the
    earlier chunks' maxima by far more than the kernel's rescale threshold, so
    the accumulated output of those heads is rescaled on the way; every head
    must still match the one-softmax oracle."""
    case = cases.make_case(B=1, T=1500, m=1, Q=1, M=8, K=512, seed=612)
    main, _, _ = cases.oracle_cache(case)
    g = np.random.default_rng(612)
    sel = g.choice(1500, 512, replace=False).astype(np.int32)
    q = case.q.copy()
    v_late = oracle.dequant_main(main[0, sel[400]]).astype(np.float32)
    v_mid = oracle.dequant_main(main[0, sel[200]]).astype(np.float32)
    v_early = oracle.dequant_main(main[0, sel[10]]).astype(np.float32)
    q[0, 0, 0:16] = synth.f32_to_bf16_bits(np.broadcast_to(v_late, (16, 512)).copy())
    q[0, 0, 16:24] = synth.f32_to_bf16_bits(np.broadcast_to(2 * v_mid, (8, 512)).copy())
    q[0, 0, 24:32] = synth.f32_to_bf16_bits(np.broadcast_to(-v_early, (8, 512)).copy())
    case.q = q
    L = GpuLayer(csa2, case)
    out = torch.empty((1, 1, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.attn_workspace_size(1, 1, 512), device=DEV)
    csa2.sparse_swa_attn(L.cache, L.q, dev(sel[None, None]), L.swa, L.swa_base, L.q_pos, case.scale, out, ws)
    assert ws.sync_status()[0] == 0
    got = bf16_to_f32(out)[0, 0]
    want = _oracle_attention(case, main, 0, 0, sel)
    cases.check_attention(got, want, "running maximum")
    for h in (0, 16, 24, 40):
        cases.check_attention(got[h:h + 1], want[h:h + 1], f"head {h}")


def synth_bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_attention_out_of_range_selection_reports_bounds(csa2):
    case = cases.make_case(B=1, T=100, m=1, Q=1, M=4, K=4, seed=701)
    L = GpuLayer(csa2, case)
    sel = np.array([[[3, 200, 7, -1]]], np.int32)                 # 200 >= cap (104)
    out = torch.empty((1, 1, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.attn_workspace_size(1, 1, 4), device=DEV)
    csa2.sparse_swa_attn(L.cache, L.q, dev(sel), L.swa, L.swa_base, L.q_pos, case.scale, out, ws)
    st, detail = ws.sync_status()
    assert st == 6 and detail == 200
    main, _, _ = cases.oracle_cache(case)
    cases.check_attention(bf16_to_f32(out)[0, 0],
                          _oracle_attention(case, main, 0, 0, np.array([3, -1, 7, -1])))


# ------------------------------------------------------------------ modes
def test_decode_config1_full_reindex_reuse(csa2):
    """Config 1: a tiny Full layer (m=2, 2048 entries, M=128, K=256, 4 queries at
    t = 4092..4095), then a Reindex and a Reuse layer on the same cache."""
    case = cases.config1_case()
    L = GpuLayer(csa2, case)
    B, Q, M, K, max_n = 1, 4, case.M, case.K, case.n_entries
    pool = torch.empty((B, Q, M), dtype=torch.int32, device=DEV)
    sel = torch.empty((B, Q, K), dtype=torch.int32, device=DEV)
    out = torch.empty((B, Q, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(max(csa2.decode_workspace_size(m, B, Q, max_n, M, K) for m in (0, 1, 2)), device=DEV)
    common = dict(q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base, scale=case.scale, ws=ws)
    csa2.decode(csa2.MODE_FULL, L.cache, sel=sel, out=out, M=M, max_n=max_n, q_idx=L.q_idx,
                w_head=L.w_head, pool_blocks=pool, **common)
    full_out, full_sel, full_pool = bf16_to_f32(out), host(sel), host(pool)
    main, codes, scales = cases.oracle_cache(case)
    assert [oracle.visible_entries(t, 2, 2048) for t in case.q_pos[0]] == [2046, 2047, 2047, 2048]
    for qi in range(Q):
        pb, sl, o = oracle.decode_query(oracle.FULL, t=case.q_pos[0, qi], m=2, n_entries=2048, main_kv=main[0],
                                        idx_codes=codes[0], idx_scales=scales[0], q=case.q[0, qi],
                                        swa=case.swa[0], swa_base=case.swa_base[0], scale=case.scale, M=M, K=K,
                                        q_idx=case.q_idx[0, qi], w_head=case.w_head[0, qi])
        nv = oracle.visible_entries(case.q_pos[0, qi], 2, 2048)
        s_or = _oracle_scores(case, codes, scales, 0, qi, np.arange(nv))
        cases.assert_set_within_tie_window(full_sel[0, qi], sl, lambda j: s_or[j], what="full sel")
        gmax = np.array([s_or[8 * r:min(8 * r + 8, nv)].max() for r in range(-(-nv // 8))])
        gmax[(nv - 1) // 8] = np.inf
        cases.assert_set_within_tie_window(full_pool[0, qi], pb, lambda r: gmax[r], what="full pool")
        cases.check_attention(full_out[0, qi], _oracle_attention(case, main, 0, qi, full_sel[0, qi]), "full")
        if set(full_sel[0, qi]) == set(sl):
            cases.check_attention(full_out[0, qi], o, "full e2e")
    # Reuse with the Full layer's selection: bit-identical output
    out2 = torch.empty_like(out)
    csa2.decode(csa2.MODE_REUSE, L.cache, sel=sel, out=out2, **common)
    assert torch.equal(out, out2)
    # Reindex over the Full layer's pool with new index queries
    q_idx2 = dev(np.ascontiguousarray(case.q_idx[:, ::-1]))
    sel2 = torch.empty_like(sel)
    csa2.decode(csa2.MODE_REINDEX, L.cache, sel=sel2, out=out2, M=M, max_n=max_n, q_idx=q_idx2,
                w_head=L.w_head, pool_blocks=pool, **common)
    got2, got_sel2 = bf16_to_f32(out2), host(sel2)
    qi_rev = case.q_idx[:, ::-1]
    for qi in range(Q):
        nv = oracle.visible_entries(case.q_pos[0, qi], 2, 2048)
        _, sl, _ = oracle.decode_query(oracle.REINDEX, t=case.q_pos[0, qi], m=2, n_entries=2048, main_kv=main[0],
                                       idx_codes=codes[0], idx_scales=scales[0], q=case.q[0, qi], swa=case.swa[0],
                                       swa_base=case.swa_base[0], scale=case.scale, M=M, K=K,
                                       q_idx=qi_rev[0, qi], w_head=case.w_head[0, qi], pool_blocks=full_pool[0, qi])
        dom = oracle.pool_entries(full_pool[0, qi], nv)
        s = np.full(nv, -np.inf)
        s[dom] = oracle.index_scores(qi_rev[0, qi], case.w_head[0, qi], codes[0], scales[0], dom)
        cases.assert_set_within_tie_window(got_sel2[0, qi], sl, lambda j: s[j], what="reindex sel")
        assert set(got_sel2[0, qi][got_sel2[0, qi] >= 0]) <= set(dom)
        cases.check_attention(got2[0, qi], _oracle_attention(case, main, 0, qi, got_sel2[0, qi]), "reindex")
    assert ws.sync_status()[0] == 0


def test_decode_reindex_with_all_blocks_equals_full_selection(csa2):
    case = cases.make_case(B=1, T=800, m=1, Q=2, M=100, K=20, seed=801)
    L = GpuLayer(csa2, case)
    B, Q, M, K, max_n = 1, 2, 100, 20, 800
    pool = torch.empty((B, Q, M), dtype=torch.int32, device=DEV)
    sel = torch.empty((B, Q, K), dtype=torch.int32, device=DEV)
    out = torch.empty((B, Q, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(max(csa2.decode_workspace_size(m, B, Q, max_n, M, K) for m in (0, 1)), device=DEV)
    common = dict(q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base, scale=case.scale, ws=ws, M=M,
                  max_n=max_n, q_idx=L.q_idx, w_head=L.w_head)
    csa2.decode(csa2.MODE_FULL, L.cache, sel=sel, out=out, pool_blocks=pool, **common)
    assert np.all(host(pool)[0, :, :100] == np.arange(100))      # ceil(800/8) = 100 blocks: all kept
    sel2 = torch.empty_like(sel)
    out2 = torch.empty_like(out)
    csa2.decode(csa2.MODE_REINDEX, L.cache, sel=sel2, out=out2, pool_blocks=pool, **common)
    assert torch.equal(sel, sel2)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("mode_out,K,Q,T", [(0, 200, 3, 1200), (1, 512, 2, 4096), (0, 20, 2, 300)])
def test_decode_packed_selection_roundtrip(csa2, mode_out, K, Q, T):
    """A Full or Reindex call with packed_sel copies the main-KV bytes of every
    selected entry into slot order; a Reuse call reading them gives the same
    output, bit for bit, as a Reuse call that gathers from the cache (K spans
    several 128-slot runs and a partial one)."""
    M = 150 if T >= 1200 else 40
    case = cases.make_case(B=2, T=T, m=1, Q=Q, M=M, K=K, seed=811 + K)
    L = GpuLayer(csa2, case)
    B, max_n = 2, T
    pool = torch.empty((B, Q, M), dtype=torch.int32, device=DEV)
    sel = torch.empty((B, Q, K), dtype=torch.int32, device=DEV)
    out = torch.empty((B, Q, 64, 512), dtype=torch.int16, device=DEV)
    packed = torch.full((B, Q, K, 288), 0xA5, dtype=torch.uint8, device=DEV)
    ws = csa2.Workspace(max(csa2.decode_workspace_size(m, B, Q, max_n, M, K) for m in (0, 1, 2)), device=DEV)
    common = dict(q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base, scale=case.scale, ws=ws, M=M,
                  max_n=max_n, q_idx=L.q_idx, w_head=L.w_head)
    if mode_out == 1:                       # a pool first, then the Reindex call writes the packed copy
        csa2.decode(csa2.MODE_FULL, L.cache, sel=sel, out=out, pool_blocks=pool, **common)
        csa2.decode(csa2.MODE_REINDEX, L.cache, sel=sel, out=out, pool_blocks=pool, packed_sel=packed, **common)
    else:
        csa2.decode(csa2.MODE_FULL, L.cache, sel=sel, out=out, pool_blocks=pool, packed_sel=packed, **common)
    assert ws.sync_status()[0] == 0
    s_h, p_h, main = host(sel), host(packed), host(L.cache.main_kv)
    valid = s_h >= 0
    assert valid.sum() > 0
    for b in range(B):
        for qi in range(Q):
            ids = s_h[b, qi][valid[b, qi]]
            assert np.array_equal(p_h[b, qi][valid[b, qi]], main[b, ids])
    out_gather = torch.empty_like(out)
    out_packed = torch.empty_like(out)
    csa2.decode(csa2.MODE_REUSE, L.cache, sel=sel, out=out_gather, **common)
    csa2.decode(csa2.MODE_REUSE, L.cache, sel=sel, out=out_packed, packed_sel=packed, **common)
    assert ws.sync_status()[0] == 0
    assert torch.equal(out_gather, out_packed)
    assert torch.equal(out_gather, out)     # Reuse with the same selection and queries = the writing call


@pytest.mark.parametrize("split,K,Q,T", [(2, 512, 2, 4096), (5, 512, 1, 4096), (3, 200, 3, 1200), (9, 20, 2, 300)])
def test_decode_attention_split(csa2, split, K, Q, T):
    """The attention of a query split over several CTAs (attn_split), each
    walking a contiguous range of its key chunks (the window, then the runs of
    128 selected entries) with its own softmax state, merged by the combine
    kernel.  A Full call with the split selects exactly what the call without it
    selects and writes the same packed copy; every output matches the oracle's
    attention over the selection; Reuse calls with the split, gathering and
    reading the packed copy, agree with each other and with the Full call bit
    for bit.  Split 9 exceeds the chunk count (K = 20: the window and one run)
    and is reduced to it; K = 200 ends in a partial run of 72 entries."""
    M = 150 if T >= 1200 else 40
    case = cases.make_case(B=2, T=T, m=1, Q=Q, M=M, K=K, seed=833 + K + split)
    L = GpuLayer(csa2, case)
    B, max_n = 2, T
    pool = torch.empty((B, Q, M), dtype=torch.int32, device=DEV)
    sel = torch.empty((B, Q, K), dtype=torch.int32, device=DEV)
    out1 = torch.empty((B, Q, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(max(csa2.decode_workspace_size(m, B, Q, max_n, M, K) for m in (0, 1, 2)), device=DEV)
    common = dict(q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base, scale=case.scale, ws=ws, M=M,
                  max_n=max_n, q_idx=L.q_idx, w_head=L.w_head)
    csa2.decode(csa2.MODE_FULL, L.cache, sel=sel, out=out1, pool_blocks=pool, **common)
    pool_s = torch.empty_like(pool)
    sel_s = torch.empty_like(sel)
    out_s = torch.empty_like(out1)
    packed = torch.full((B, Q, K, 288), 0xA5, dtype=torch.uint8, device=DEV)
    csa2.decode(csa2.MODE_FULL, L.cache, sel=sel_s, out=out_s, pool_blocks=pool_s, packed_sel=packed,
                attn_split=split, **common)
    assert ws.sync_status()[0] == 0
    assert torch.equal(sel, sel_s) and torch.equal(pool, pool_s)
    s_h, p_h, main_dev = host(sel_s), host(packed), host(L.cache.main_kv)
    valid = s_h >= 0
    for b in range(B):
        for qi in range(Q):
            assert np.array_equal(p_h[b, qi][valid[b, qi]], main_dev[b, s_h[b, qi][valid[b, qi]]])
    main, _, _ = cases.oracle_cache(case)
    got = bf16_to_f32(out_s)
    for b in range(B):
        for qi in range(Q):
            cases.check_attention(got[b, qi], _oracle_attention(case, main, b, qi, s_h[b, qi]),
                                  f"split {split} b{b} q{qi}")
    out_g = torch.empty_like(out1)
    out_p = torch.empty_like(out1)
    csa2.decode(csa2.MODE_REUSE, L.cache, sel=sel_s, out=out_g, attn_split=split, **common)
    csa2.decode(csa2.MODE_REUSE, L.cache, sel=sel_s, out=out_p, packed_sel=packed, attn_split=split, **common)
    assert ws.sync_status()[0] == 0
    assert torch.equal(out_g, out_p)
    assert torch.equal(out_g, out_s)
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        csa2.decode(csa2.MODE_REUSE, L.cache, sel=sel_s, out=out_g, attn_split=-1, **common)


def test_decode_packed_selection_must_be_aligned(csa2):
    case = cases.make_case(B=1, T=300, m=1, Q=1, M=40, K=20, seed=815)
    L = GpuLayer(csa2, case)
    sel = torch.zeros((1, 1, 20), dtype=torch.int32, device=DEV)
    out = torch.empty((1, 1, 64, 512), dtype=torch.int16, device=DEV)
    packed = torch.zeros(20 * 288 + 16, dtype=torch.uint8, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(2, 1, 1, 300, 40, 20), device=DEV)
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        csa2.decode(csa2.MODE_REUSE, L.cache, q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base,
                    scale=case.scale, sel=sel, out=out, ws=ws, packed_sel=packed[8:])


def test_decode_reindex_select_equal_and_two_level_scores(csa2):
    """Reindex selection where the scores leave the select little to separate.
    Query 0: every entry carries the same index-key row, so every score is the
    same: every pooled key is a candidate, the first digit pass finds all of
    them in one bin, and the lowest ids of the pool (every other block) must
    be taken.  Query 1: the pooled blocks with index 1 mod 8 (none of query
    0's) carry a second row with a higher score, so the keys take two values
    and K cuts through the lower group: all higher keys plus the lowest-id
    lower keys.  Both compared with the oracle's exact selection, and the
    attention over them."""
    T, M = 4096, 512
    case = cases.make_case(B=1, T=T, m=1, Q=2, M=M, K=1, seed=913)
    L = GpuLayer(csa2, case)
    main, codes, scales = cases.oracle_cache(case)
    codes, scales = codes.copy(), scales.copy()
    s_all = _oracle_scores(case, codes, scales, 0, 1, np.arange(T))
    order = np.argsort(-s_all, kind="stable")
    hi_row, lo_row = int(order[10]), int(order[2000])
    assert s_all[hi_row] > s_all[lo_row]
    hi_c, hi_s = codes[0, hi_row].copy(), scales[0, hi_row].copy()
    codes[0, :] = codes[0, lo_row].copy()
    scales[0, :] = scales[0, lo_row].copy()
    hi_blocks = np.arange(1, 200, 8)                               # odd blocks only
    for blk in hi_blocks:
        codes[0, 8 * blk:8 * blk + 8] = hi_c
        scales[0, 8 * blk:8 * blk + 8] = hi_s
    L.cache.idx_codes[0, :T].copy_(torch.from_numpy(codes[0]))
    L.cache.idx_scales[0, :T].copy_(torch.from_numpy(scales[0]))

    K = 300
    pool = np.full((1, 2, M), -1, np.int32)
    pool[0, 0, :256] = np.arange(0, M, 2)                          # every other block
    pool[0, 1, :200] = np.arange(200)
    sel = torch.empty((1, 2, K), dtype=torch.int32, device=DEV)
    out = torch.empty((1, 2, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(1, 1, 2, T, M, K), device=DEV)
    csa2.decode(csa2.MODE_REINDEX, L.cache, q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base,
                scale=case.scale, sel=sel, out=out, ws=ws, M=M, max_n=T, q_idx=L.q_idx, w_head=L.w_head,
                pool_blocks=dev(pool))
    assert ws.sync_status()[0] == 0
    got, got_out = host(sel), bf16_to_f32(out)
    for qi in range(2):
        nv = oracle.visible_entries(case.q_pos[0, qi], 1, T)
        s = np.full(T, -np.inf)
        s[:nv] = _oracle_scores(case, codes, scales, 0, qi, np.arange(nv))
        dom = oracle.pool_entries(pool[0, qi], nv)
        want = oracle.select_topk(s, dom, K)
        if qi == 0:
            assert len(np.unique(s[dom])) == 1                     # one score for the whole pool
        else:
            hi = np.isin(dom // 8, hi_blocks)
            assert len(np.unique(s[dom])) == 2 and 0 < hi.sum() < K
        np.testing.assert_array_equal(got[0, qi], want)
        cases.check_attention(got_out[0, qi], _oracle_attention(case, main, 0, qi, got[0, qi]),
                              f"reindex equal scores q{qi}")


def test_decode_reindex_select_ties_and_short_pool(csa2):
    """Reindex selection is one radix select over the keys of the whole pool
    (512 blocks = 32 tiles, scored in several rounds; each select thread owns
    64 consecutive slots).  Query 0: every block in the pool, and eight blocks
    spread over the pool carry copies of one index-key row, so 65 entries have
    bit-identical scores in different rounds and different threads' key rows,
    and K cuts through them: the lowest ids must win (score desc, id asc).  Its
    last pooled entry is not yet visible.  Query 1: a pool of 30 blocks (240
    entries) padded with -1 and K > 240, so every pooled entry is chosen in
    ascending order and the tail of sel is -1."""
    T, M = 4096, 512
    case = cases.make_case(B=1, T=T, m=1, Q=2, M=M, K=1, seed=911)
    L = GpuLayer(csa2, case)
    main, codes, scales = cases.oracle_cache(case)
    codes, scales = codes.copy(), scales.copy()
    s0 = _oracle_scores(case, codes, scales, 0, 0, np.arange(T))
    X = int(np.argsort(-s0, kind="stable")[350])
    tie_blocks = [5, 70, 140, 200, 260, 330, 400, 470]          # one in each CTA's eighth (64 blocks)
    for blk in tie_blocks:
        codes[0, 8 * blk:8 * blk + 8] = codes[0, X]
        scales[0, 8 * blk:8 * blk + 8] = scales[0, X]
    L.cache.idx_codes[0, :T].copy_(torch.from_numpy(codes[0]))
    L.cache.idx_scales[0, :T].copy_(torch.from_numpy(scales[0]))
    tied = np.sort(np.concatenate([[X], *[np.arange(8 * b, 8 * b + 8) for b in tie_blocks]]))
    nv0 = oracle.visible_entries(case.q_pos[0, 0], 1, T)
    assert nv0 == T - 1
    s0 = np.full(T, -np.inf)
    s0[:nv0] = _oracle_scores(case, codes, scales, 0, 0, np.arange(nv0))
    v = s0[X]
    n_greater = int(np.sum(s0 > v))
    K = n_greater + 32
    assert 240 < K <= 512 and n_greater + len(tied) > K

    g = np.random.default_rng(5)
    pool = np.full((1, 2, M), -1, np.int32)
    pool[0, 0] = np.arange(M)
    pool[0, 1, :30] = np.sort(g.choice(M, 30, replace=False))
    sel = torch.empty((1, 2, K), dtype=torch.int32, device=DEV)
    out = torch.empty((1, 2, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(1, 1, 2, T, M, K), device=DEV)
    csa2.decode(csa2.MODE_REINDEX, L.cache, q_pos=L.q_pos, q=L.q, swa=L.swa, swa_base_pos=L.swa_base,
                scale=case.scale, sel=sel, out=out, ws=ws, M=M, max_n=T, q_idx=L.q_idx, w_head=L.w_head,
                pool_blocks=dev(pool))
    assert ws.sync_status()[0] == 0
    got, got_out = host(sel), bf16_to_f32(out)

    # query 0: exact top-K by (score desc, id asc); ties inside the tie group go to the lowest ids
    want0 = oracle.select_topk(s0, oracle.pool_entries(pool[0, 0], nv0), K)
    cases.assert_set_within_tie_window(got[0, 0], want0, lambda j: s0[j], what="reindex ties")
    assert np.all(np.diff(got[0, 0]) > 0) and got[0, 0].max() < nv0
    taken = np.isin(tied, got[0, 0])
    assert 0 < taken.sum() < len(tied)
    assert np.all(taken[:taken.sum()]), "tied entries must be taken in ascending id order"
    cases.check_attention(got_out[0, 0], _oracle_attention(case, main, 0, 0, got[0, 0]), "reindex ties")

    # query 1: fewer pooled entries than K
    nv1 = oracle.visible_entries(case.q_pos[0, 1], 1, T)
    dom1 = oracle.pool_entries(pool[0, 1], nv1)
    assert len(dom1) == 240
    want1 = np.full(K, -1, np.int32)
    want1[:240] = dom1
    np.testing.assert_array_equal(got[0, 1], want1)
    cases.check_attention(got_out[0, 1], _oracle_attention(case, main, 0, 1, got[0, 1]), "reindex short pool")
