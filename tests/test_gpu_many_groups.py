"""Index scan over more query groups than one launch's grid holds.

The scan issues at most 65,535 query groups per launch (the grid's y extent)
and splits larger calls into several launches with a group offset.  Both
variants are run across that boundary: one query per sequence (65,540
sequences, one group each) and the grouped path (13,108 sequences x 25
queries = 65,540 groups of five).  The caches hold random MXFP4 bytes; the
oracle scores sampled sequences on each side of the boundary from the same
bytes, within 1e-5 of sum_h |w_h| ReLU(q_h . k_j)."""
import numpy as np
import pytest

import oracle
import synth

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


def _host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("B,Q", [(65540, 1), (13108, 25)])
def test_index_scan_across_launch_boundary(csa2, B, Q):
    cap = 16
    g = torch.Generator(device=DEV)
    g.manual_seed(9100 + Q)
    cache = csa2.Cache(B, cap, 1, device=DEV)
    cache.idx_codes.random_(0, 256, generator=g)
    cache.idx_scales.random_(120, 135, generator=g)          # E8M0 2^-7 .. 2^7
    cache.n_entries.fill_(cap)
    q_idx = synth.torch_normal(9200 + Q, (B, Q, 32, 128), torch.bfloat16, DEV)
    w_head = torch.randn((B, Q, 32), generator=g, device=DEV, dtype=torch.float32)
    q_pos = torch.full((B, Q), cap - 1, dtype=torch.int64, device=DEV)
    scores = torch.full((B, Q, cap), -123.0, device=DEV)
    ws = csa2.Workspace(1 << 16, device=DEV)
    csa2.index_score(cache, q_idx.view(torch.int16), w_head, q_pos, scores, cap, ws)
    assert ws.sync_status() == (0, 0)
    groups_per_seq = -(-Q // 5) if Q >= 5 else Q
    boundary_seq = 65535 // groups_per_seq                     # the sequence holding group 65,535
    for b in sorted(x for x in {0, 1, boundary_seq - 1, boundary_seq, boundary_seq + 1, B - 1} if x < B):
        codes = cache.idx_codes[b].cpu().numpy()
        scales = cache.idx_scales[b].cpu().numpy()
        qb = _host_bits(q_idx[b])
        wb = w_head[b].cpu().numpy()
        got = scores[b].cpu().numpy()
        kd = oracle.dequant_index(codes, scales)
        for qi in range(Q):
            want = oracle.index_scores(qb[qi], wb[qi], codes, scales)
            dots = kd @ oracle.quantize_index_query(qb[qi]).T
            bound = 1e-5 * (np.maximum(dots, 0) @ np.abs(wb[qi].astype(np.float64))) + 1e-30
            assert np.all(np.abs(got[qi] - want) <= bound), (b, qi)
