"""Host-side paths on the GPU: the bounded-wait timeout path of a kernel, and
first calls made by several host threads at once.

Timeout: the library's test hook (csa2_test_withhold_arrival) makes the index
scan's producer wait on an mbarrier that nothing arrives on, before the kernel
has issued any copy or MMA.  The wait gives up after a short bound, the kernel
records CSA2_ERR_TIMEOUT in the workspace status word and returns; no GPU
fault or hang is involved, and the next call on the same context is correct.

Threads: a fresh process (so that no launch attribute is set yet) starts eight
host threads that make their first library calls at the same moment, each on
its own stream and workspace; every thread's result must equal the one the
process computes afterwards on one thread."""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle
from tests import cases

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def test_withheld_arrival_times_out_and_the_context_stays_usable(csa2):
    case = cases.make_case(B=1, T=600, m=1, Q=1, M=8, K=8, seed=4401)
    n = case.n_entries
    cache = csa2.Cache(1, n, 1, device=DEV)
    ws = csa2.Workspace(1 << 16, device=DEV)
    rope = csa2.rope_table(n).to(DEV)
    csa2.compress_quantize(cache, _dev(case.x), torch.zeros(1, dtype=torch.int64, device=DEV), _dev(case.w0),
                           _dev(case.w1), rope, _dev(case.w_idx), ws)
    cache.n_entries.fill_(n)
    assert ws.sync_status() == (0, 0)
    q_pos, q_idx, w_head = _dev(case.q_pos), _dev(case.q_idx), _dev(case.w_head)
    scores = torch.full((1, 1, n), -123.0, device=DEV)
    lib = csa2.load()
    assert lib.csa2_test_withhold_arrival(1) == 0
    try:
        csa2.index_score(cache, q_idx, w_head, q_pos, scores, n, ws)      # enqueued: returns OK
        st, detail = ws.sync_status()
    finally:
        assert lib.csa2_test_withhold_arrival(0) == 0
    assert (st, detail) == (5, 2)                                        # CSA2_ERR_TIMEOUT at the hook's wait
    assert bool((scores == -123.0).all())                                # nothing was scored
    assert ws.sync_status() == (0, 0)                                    # the status word was cleared
    csa2.index_score(cache, q_idx, w_head, q_pos, scores, n, ws)
    assert ws.sync_status() == (0, 0)
    _, codes, scales = cases.oracle_cache(case)
    want = oracle.index_scores(case.q_idx[0, 0], case.w_head[0, 0], codes[0], scales[0])
    got = scores.cpu().numpy()[0, 0]
    # fp32 accumulation of exact products: within 1e-5 of sum_h |w_h| ReLU(q_h . k_j)
    qd = oracle.quantize_index_query(case.q_idx[0, 0])
    dots = oracle.dequant_index(codes[0], scales[0]) @ qd.T
    bound = 1e-5 * (np.maximum(dots, 0) @ np.abs(case.w_head[0, 0].astype(np.float64))) + 1e-30
    assert np.all(np.abs(got - want) <= bound)
    assert lib.csa2_test_withhold_arrival(2) == 1                       # only 0 and 1


_THREADS_SCRIPT = textwrap.dedent("""
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    import fp4_kv_cache_csa2_gb300 as csa2
    import synth
    csa2.load()
    B, Q, N, M, K = 2, 3, 5000, 64, 100
    g = synth.rng(4402)
    s = torch.from_numpy(g.standard_normal((B, Q, N)).astype(np.float32)).cuda()
    q_pos = torch.tensor([[4999, 3000, 20], [4000, 4999, 7]], dtype=torch.int64, device="cuda")
    cache = csa2.Cache(B, N, 1)
    cache.n_entries.fill_(N)
    torch.cuda.synchronize()
    T = 8
    outs = [None] * T
    barrier = threading.Barrier(T)
    def work(i):
        st = torch.cuda.Stream()
        ws_b = csa2.Workspace(csa2.block_topk_workspace_size(B, Q, N), stream=st)
        ws_s = csa2.Workspace(csa2.select_topk_workspace_size(B, Q, N), stream=st)
        pool = torch.empty((B, Q, M), dtype=torch.int32, device="cuda")
        sel = torch.empty((B, Q, K), dtype=torch.int32, device="cuda")
        st.synchronize()
        barrier.wait()                     # first library launches of the process, all at once
        csa2.block_topk(cache, s, q_pos, N, M, pool, ws_b, stream=st)
        csa2.select_topk(cache, s, q_pos, K, sel, N, ws_s, stream=st)
        assert ws_b.sync_status(stream=st)[0] == 0 and ws_s.sync_status(stream=st)[0] == 0
        outs[i] = (pool.cpu(), sel.cpu())
    th = [threading.Thread(target=work, args=(i,)) for i in range(T)]
    for t in th: t.start()
    for t in th: t.join()
    ws = csa2.Workspace(csa2.block_topk_workspace_size(B, Q, N))
    pool = torch.empty((B, Q, M), dtype=torch.int32, device="cuda")
    sel = torch.empty((B, Q, K), dtype=torch.int32, device="cuda")
    csa2.block_topk(cache, s, q_pos, N, M, pool, ws)
    csa2.select_topk(cache, s, q_pos, K, sel, N, ws)
    assert ws.sync_status()[0] == 0
    for i in range(T):
        assert outs[i] is not None, i
        assert torch.equal(outs[i][0], pool.cpu()) and torch.equal(outs[i][1], sel.cpu()), i
    print("THREADS_OK")
""")


def test_concurrent_first_calls_from_host_threads(csa2):
    r = subprocess.run([sys.executable, "-c", _THREADS_SCRIPT, ROOT], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0 and "THREADS_OK" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
