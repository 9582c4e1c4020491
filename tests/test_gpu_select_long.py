"""Full-row selection on long rows (more than 16,384 visible entries): the
multi-CTA histogram / filter / resolve path behind csa2_block_topk,
csa2_select_topk and the Full decode.

The scores are seeded synthetic inputs handed to the library and to the oracle
alike, so both rank the same binary32 values: the chosen entry and block ids
must equal the oracle's exactly, ties included (score desc, id asc).  The
distributions cover the spread case (normal scores), heavy ties (scores on a
1/8 grid), scores bunched far from zero (threshold bins too full for the
candidate lists, which sends rows to the exact single-CTA select) and a row
of equal scores, with rows of different visible lengths in one call (causal
queries, n_visible <= K, n_visible = 0)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
K_SEL, M_BLK = 512, 2048


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_kv_cache_csa2_gb300 as m
    m.load()
    return m


def _scores(kind: str, seed: int, shape) -> np.ndarray:
    g = synth.rng(seed)
    x = g.standard_normal(shape)
    if kind == "normal":
        return x.astype(np.float32)
    if kind == "grid":                       # many exact ties
        return (np.round(x * 8) / 8).astype(np.float32)
    if kind == "bunched":                    # all keys in one or two 12-bit bins
        return (1000.0 + 1e-3 * x).astype(np.float32)
    if kind == "equal":
        return np.ones(shape, np.float32)
    raise ValueError(kind)


def _run(csa2, kind, seed, m, max_n, n_entries, q_pos, K=K_SEL, M=M_BLK):
    B, Q = q_pos.shape
    cache = csa2.Cache(B, max_n, m)
    cache.n_entries.copy_(torch.tensor(n_entries, dtype=torch.int32))
    s = _scores(kind, seed, (B, Q, max_n))
    scores = torch.from_numpy(s).to(DEV)
    d_pos = torch.from_numpy(q_pos.astype(np.int64)).to(DEV)
    ws_b = csa2.Workspace(csa2.block_topk_workspace_size(B, Q, max_n))
    ws_s = csa2.Workspace(csa2.select_topk_workspace_size(B, Q, max_n))
    pool = torch.full((B, Q, M), 7, dtype=torch.int32, device=DEV)
    sel = torch.full((B, Q, K), 7, dtype=torch.int32, device=DEV)
    csa2.block_topk(cache, scores, d_pos, max_n, M, pool, ws_b)
    csa2.select_topk(cache, scores, d_pos, K, sel, max_n, ws_s)
    assert ws_b.sync_status() == (0, 0)
    assert ws_s.sync_status() == (0, 0)
    got_pool, got_sel = pool.cpu().numpy(), sel.cpu().numpy()
    for b in range(B):
        for qi in range(Q):
            nv = min(oracle.visible_entries(int(q_pos[b, qi]), m, int(n_entries[b])), max_n)
            row = s[b, qi].astype(np.float64)
            want_sel = oracle.select_topk(row, np.arange(nv), K)
            want_pool = oracle.block_topm(row, nv, M)
            np.testing.assert_array_equal(got_sel[b, qi], want_sel, err_msg=f"{kind} sel b={b} q={qi} nv={nv}")
            np.testing.assert_array_equal(got_pool[b, qi], want_pool, err_msg=f"{kind} pool b={b} q={qi} nv={nv}")


@pytest.mark.parametrize("kind", ["normal", "grid"])
def test_long_rows_match_oracle_exactly(csa2, kind):
    """200,003-entry rows (a stride that is no multiple of 4), four causal
    queries of different visible lengths, m = 1."""
    max_n = 200_003
    q_pos = np.array([[200_002, 100_000], [149_999, 1_000_000]])
    _run(csa2, kind, 7100 + len(kind), 1, max_n, [max_n, 150_000], q_pos)


@pytest.mark.parametrize("kind", ["normal", "grid"])
def test_rows_past_the_bitmap_limit_match_oracle_exactly(csa2, kind):
    """Rows of more than 524,288 visible entries, where the resolve step puts
    the chosen ids in order with a bitonic sort instead of the row bitmap:
    600,011-entry rows, with causal queries of 555,556 and 580,000 visible
    entries beside one of exactly 524,288 (the last row length that takes the
    bitmap) in the same call."""
    max_n = 600_011
    q_pos = np.array([[600_010, 524_287], [555_555, 2_000_000]])
    _run(csa2, kind, 7500 + len(kind), 1, max_n, [max_n, 580_000], q_pos)


def test_long_rows_with_short_and_empty_queries(csa2):
    """m = 2 rows where some queries see fewer than K entries or fewer than M
    blocks (all of them are chosen), and one sees nothing."""
    max_n = 40_000
    q_pos = np.array([[79_999, 600, 0, 20_001, 5_000]])
    _run(csa2, "normal", 7200, 2, max_n, [max_n], q_pos)


@pytest.mark.parametrize("kind", ["bunched", "equal"])
def test_full_threshold_bins_fall_back_exactly(csa2, kind):
    """Scores packed into one or two histogram bins overflow the candidate
    lists; the rows go to the single-CTA radix select and stay exact."""
    max_n = 40_000
    q_pos = np.array([[39_999, 30_000], [25_000, 39_999]])
    _run(csa2, kind, 7300 + len(kind), 1, max_n, [max_n, max_n], q_pos)


def test_small_k_and_m(csa2):
    """K and M far below the row length: the threshold sits deep in the tail."""
    max_n = 70_000
    q_pos = np.array([[69_999, 50_000, 33_333]])
    _run(csa2, "normal", 7400, 1, max_n, [max_n], q_pos, K=1, M=3)
    _run(csa2, "grid", 7401, 1, max_n, [max_n], q_pos, K=17, M=1)
