"""The allocation-free candidate-block call, checked against the regular one.

csa2_block_topk_static serves callers that may not allocate device memory (a
plugin inside an engine that owns the whole GPU through its own allocator, or a
latency-critical path that must not hit cudaMalloc).  It keeps its scratch in
a fixed array inside the library.  This file is collected last so that a
failure here never hides the other tests; it also passes on its own."""
import numpy as np
import pytest

import oracle
import synth
from tests import cases

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_kv_cache_csa2_gb300 as m
    m.load()
    return m


def _dev(a):
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def test_static_block_topk_matches_workspace_version_twice(csa2):
    case = cases.make_case(B=2, T=2 * 1500, m=2, Q=3, M=40, K=16, seed=901,
                           q_pos=np.array([[2999, 2000, 700], [2998, 5, 1]]))
    n = case.n_entries
    cache = csa2.Cache(case.B, n, case.m, device="cuda")
    ws = csa2.Workspace(csa2.block_topk_workspace_size(case.B, case.Q, n), device="cuda")
    rope = csa2.rope_table(n).to("cuda")
    csa2.compress_quantize(cache, _dev(case.x), torch.zeros(case.B, dtype=torch.int64, device="cuda"),
                           _dev(case.w0), _dev(case.w1), rope, _dev(case.w_idx), ws)
    cache.n_entries.fill_(n)
    q_pos = _dev(case.q_pos)
    scores = torch.empty((case.B, case.Q, n), device="cuda")
    csa2.index_score(cache, _dev(case.q_idx), _dev(case.w_head), q_pos, scores, n, ws)
    want = torch.full((case.B, case.Q, case.M), -7, dtype=torch.int32, device="cuda")
    csa2.block_topk(cache, scores, q_pos, n, case.M, want, ws)
    assert ws.sync_status()[0] == 0
    for _ in range(2):                                    # two calls in a row share the array
        got = torch.full_like(want, -7)
        assert csa2.block_topk_static(cache, scores, q_pos, n, case.M, got) == 0
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    # a second, smaller request right after a larger one sees no stale keys
    got1 = torch.full((1, 1, case.M), -7, dtype=torch.int32, device="cuda")
    want1 = torch.full_like(got1, -7)
    csa2.block_topk(cache, scores[1:, 1:2].contiguous(), q_pos[1:, 1:2].contiguous(), n, case.M, want1, ws)
    assert csa2.block_topk_static(cache, scores[1:, 1:2].contiguous(), q_pos[1:, 1:2].contiguous(), n,
                                  case.M, got1) == 0
    torch.cuda.synchronize()
    assert torch.equal(got1, want1)


def test_static_block_topk_rejects_requests_beyond_the_scratch(csa2):
    cache = csa2.Cache(1, 8, 1, device="cuda")
    q_pos = torch.zeros((1, 1), dtype=torch.int64, device="cuda")
    out = torch.empty((1, 1, 4), dtype=torch.int32, device="cuda")
    scores = torch.empty((1, 1, 8), device="cuda")
    # 2 * 1 * ceil(8_388_616 / 8) = 2,097,154 keys > 1,048,576
    st = csa2.block_topk_static(cache, scores, torch.zeros((2, 1), dtype=torch.int64, device="cuda"),
                                8_388_616, 4, out)
    assert st == 3                                        # CSA2_ERR_WORKSPACE, nothing enqueued
    assert csa2.block_topk_static(cache, scores, q_pos, 8, 4, out) == 0


@pytest.mark.parametrize("max_n,n_entries,q_pos", [
    (131_072, [131_072], [[131_071, 131_064, 70_000, 5]]),
    (200_003, [200_003], [[200_002, 150_000, 131_073, 9]]),
])
def test_static_block_topk_long_rows_match_regular_call_and_oracle(csa2, max_n, n_entries, q_pos):
    """Rows long enough that the two calls take different routes: the regular
    call hands rows over 16,384 entries to the multi-CTA row selection, the
    allocation-free call keeps its block maxima in the fixed array and selects
    past 131,072 entries with the single-CTA radix select.  Both must give the
    oracle's blocks exactly, the forced newest block and the order of equal
    maxima included; q_pos makes the queries see different prefixes."""
    q_pos = np.array(q_pos, np.int64)
    B, Q = q_pos.shape
    M = 2048
    cache = csa2.Cache(B, max_n + (-max_n) % 8, 1, device="cuda")
    cache.n_entries.copy_(torch.tensor(n_entries, dtype=torch.int32))
    g = synth.rng(990 + max_n % 97)
    s = (np.round(g.standard_normal((B, Q, max_n)) * 16) / 16).astype(np.float32)   # many equal maxima
    scores = torch.from_numpy(s).to("cuda")
    d_pos = torch.from_numpy(q_pos).to("cuda")
    ws = csa2.Workspace(csa2.block_topk_workspace_size(B, Q, max_n), device="cuda")
    want = torch.full((B, Q, M), -7, dtype=torch.int32, device="cuda")
    csa2.block_topk(cache, scores, d_pos, max_n, M, want, ws)
    assert ws.sync_status()[0] == 0
    for _ in range(2):
        got = torch.full_like(want, -7)
        assert csa2.block_topk_static(cache, scores, d_pos, max_n, M, got) == 0
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    got_h = got.cpu().numpy()
    for b in range(B):
        for qi in range(Q):
            nv = min(oracle.visible_entries(int(q_pos[b, qi]), 1, n_entries[b]), max_n)
            np.testing.assert_array_equal(got_h[b, qi], oracle.block_topm(s[b, qi].astype(np.float64), nv, M),
                                          err_msg=f"b={b} q={qi} nv={nv}")

