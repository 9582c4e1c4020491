"""Parity at the full sizes of the workload configurations, on sampled outputs.

The GPU runs each configuration whole, through the same library calls the
benchmark makes.  The oracle then recomputes a sample: it rebuilds the sampled
sequences' caches itself from the same seeded latents (regenerated chunk by
chunk, copied to the host) and recomputes the sampled queries.  Quantised
bytes must match bit for bit; index sets may differ only inside the 1e-4
relative tie window of the oracle's k-th score; attention outputs must reach
rel-L2 <= 1e-2 and max-abs <= 3e-2.  Stages are checked in order, each one on
the previous stage's GPU result once that has passed (a tie-window swap then
cannot cascade), and end to end wherever the selections agree."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import cases

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
CHUNK = 1 << 17            # tokens per cache-write call (even, so m = 2 pairs never straddle chunks)
M_BLK, K_SEL, WIN = 2048, 512, 128


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_kv_cache_csa2_gb300 as m
    m.load()
    return m


def host(t) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


def bf16_to_f32(t) -> np.ndarray:
    return (host(t).astype(np.uint32) << 16).view(np.float32)


def chunk_seed(seed: int, b: int, c: int) -> int:
    return (seed * 100_003 + b) * 1_009 + c


def chunk_latents(seed: int, b: int, c: int, T: int):
    """Latents of tokens [c*CHUNK, min((c+1)*CHUNK, T)) of sequence b, on the GPU."""
    return synth.torch_latents(chunk_seed(seed, b, c), (min(CHUNK, T - c * CHUNK),), DEV)


class Weights:
    def __init__(self, seed: int):
        g = synth.rng(seed)
        self.w0, self.w1 = synth.compressor_weights(g)
        self.w_idx = synth.index_projection(g)
        self.d_w0 = torch.from_numpy(self.w0).to(DEV)
        self.d_w1 = torch.from_numpy(self.w1).to(DEV)
        self.d_w_idx = torch.from_numpy(self.w_idx.view(np.int16)).to(DEV)


def write_sequence(csa2, cache, b: int, T: int, w: Weights, rope, ws, seed: int):
    """Cache write of sequence b's T tokens, chunk by chunk, at entries 0.."""
    view = cache.sequence(b)
    for c in range(-(-T // CHUNK)):
        x = chunk_latents(seed, b, c, T)
        start = torch.tensor([c * CHUNK // cache.m], dtype=torch.int64, device=DEV)
        csa2.compress_quantize(view, x.view(torch.int16)[None], start, w.d_w0, w.d_w1, rope, w.d_w_idx, ws)


def host_rows(seed: int, b: int, T: int, tokens) -> np.ndarray:
    """bf16 bits of the given token rows of sequence b (regenerated seeded inputs)."""
    tokens = np.asarray(tokens, np.int64)
    out = np.empty((len(tokens), 512), np.uint16)
    for c in np.unique(tokens // CHUNK):
        pick = np.nonzero(tokens // CHUNK == c)[0]
        x = chunk_latents(seed, b, int(c), T)
        rows = torch.from_numpy(tokens[pick] - int(c) * CHUNK).to(DEV)
        out[pick] = host(x[rows])
    return out


def oracle_sequence_cache(seed: int, b: int, T: int, m: int, w: Weights, cs):
    x = host_rows(seed, b, T, np.arange(T))
    return oracle.compress_quantize(x, m, w.w0, w.w1, w.w_idx, 0, cs=cs)


def check_pool(got, want, scores, nv: int, what: str):
    """Candidate blocks: tie window on the oracle's block maxima (+inf for the forced block)."""
    nb = -(-nv // 8)
    pad = np.full(nb * 8, -np.inf)
    pad[:nv] = scores[:nv]
    gmax = pad.reshape(nb, 8).max(axis=1)
    gmax[(nv - 1) // 8] = np.inf
    cases.assert_set_within_tie_window(got, want, lambda r: gmax[r], what=what)


# ------------------------------------------------------------------ config 2
def test_config2_cache_write_four_layers_of_1m_tokens(csa2):
    """Cache write of 4 source layers (3 at m=2, 1 at m=1) over 1,048,576 tokens:
    890 bytes per token in total, and 256 sampled entries per layer (first,
    last, chunk edges, random) bit-exact against the oracle."""
    T = 1 << 20
    w = Weights(1)
    rope = csa2.rope_table(T).to(DEV)
    cs = oracle.rope_table(T)
    ws = csa2.Workspace(1 << 16)
    total = 0
    for layer, m in enumerate((2, 2, 2, 1)):
        n = T // m
        cache = csa2.Cache(1, n, m)
        seed = 10 + layer
        write_sequence(csa2, cache, 0, T, w, rope, ws, seed)
        st, detail = ws.sync_status()
        assert st == 0, (st, detail)
        total += sum(int(t[0, :n].numel()) for t in (cache.main_kv, cache.idx_codes, cache.idx_scales))
        g = np.random.default_rng(100 + layer)
        edge = CHUNK // m
        ent = np.unique(np.concatenate([[0, 1, edge - 1, edge, n - 1], g.integers(0, n, 251)]))
        tokens = (ent[:, None] * m + np.arange(m)[None, :]).ravel()
        x = host_rows(seed, 0, T, tokens).reshape(len(ent), m, 512)
        main, codes, scales = host(cache.main_kv[0]), host(cache.idx_codes[0]), host(cache.idx_scales[0])
        for i, e in enumerate(ent):
            mk, c, s = oracle.compress_quantize(x[i], m, w.w0, w.w1, w.w_idx, 0, cs=cs[e:e + 1])
            assert np.array_equal(main[e], mk[0]), f"layer {layer} entry {e}: main KV bytes"
            assert np.array_equal(codes[e], c[0]), f"layer {layer} entry {e}: index codes"
            assert np.array_equal(scales[e], s[0]), f"layer {layer} entry {e}: index scales"
    assert total == 890 * T


# ------------------------------------------------------------------ config 3
def test_config3_full_decode_64_sequences_of_131072_entries(csa2):
    """Full mode at m=1: 64 sequences x 131,072 entries, one query per sequence at
    t = N-1, M = 2048, K = 512.  Three sequences are recomputed by the oracle."""
    B, N = 64, 1 << 17
    w = Weights(2)
    rope = csa2.rope_table(N).to(DEV)
    cache = csa2.Cache(B, N, 1)
    ws_cw = csa2.Workspace(1 << 16)
    for b in range(B):
        write_sequence(csa2, cache, b, N, w, rope, ws_cw, seed=2)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    q_idx = synth.torch_normal(21, (B, 1, 32, 128), torch.bfloat16, DEV)
    w_head = synth.torch_normal(22, (B, 1, 32), torch.float32, DEV)
    q = synth.torch_normal(23, (B, 1, 64, 512), torch.bfloat16, DEV)
    swa = synth.torch_swa_rows(24, (B, WIN), DEV)
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=DEV)
    swa_base = torch.full((B,), N - WIN, dtype=torch.int64, device=DEV)
    pool = torch.empty((B, 1, M_BLK), dtype=torch.int32, device=DEV)
    sel = torch.empty((B, 1, K_SEL), dtype=torch.int32, device=DEV)
    out = torch.empty((B, 1, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, B, 1, N, M_BLK, K_SEL))
    scale = 1 / math.sqrt(512)
    csa2.decode(csa2.MODE_FULL, cache, q_pos=q_pos, q=q.view(torch.int16), swa=swa.view(torch.int16),
                swa_base_pos=swa_base, scale=scale, sel=sel, out=out.view(torch.int16), ws=ws, M=M_BLK,
                max_n=N, q_idx=q_idx.view(torch.int16), w_head=w_head, pool_blocks=pool)
    st, detail = ws.sync_status()
    assert st == 0, (st, detail)
    cs = oracle.rope_table(N)
    got_pool, got_sel, got_out = host(pool), host(sel), bf16_to_f32(out)
    h_qidx, h_w, h_q, h_swa = host(q_idx), host(w_head), host(q), host(swa)
    for b in (0, 37, B - 1):
        main, codes, scales = oracle_sequence_cache(2, b, N, 1, w, cs)
        pb, sl, o = oracle.decode_query(oracle.FULL, t=N - 1, m=1, n_entries=N, main_kv=main, idx_codes=codes,
                                        idx_scales=scales, q=h_q[b, 0], swa=h_swa[b], swa_base=N - WIN,
                                        scale=scale, M=M_BLK, K=K_SEL, q_idx=h_qidx[b, 0], w_head=h_w[b, 0])
        scores = oracle.index_scores(h_qidx[b, 0], h_w[b, 0], codes, scales)
        check_pool(got_pool[b, 0], pb, scores, N, f"seq {b} pool")
        cases.assert_set_within_tie_window(got_sel[b, 0], sl, lambda j: scores[j], what=f"seq {b} sel")
        cases.check_attention(got_out[b, 0], oracle.attention(h_q[b, 0], got_sel[b, 0], main, h_swa[b], N - WIN,
                                                              N - 1, scale), f"seq {b} attention")
        if set(got_sel[b, 0]) == set(sl):
            cases.check_attention(got_out[b, 0], o, f"seq {b} end to end")


# ------------------------------------------------------------------ config 4
def test_config4_reindex_and_reuse_at_1m_entries(csa2):
    """The benchmark's chain at full size: 16 sequences x 1,048,576 entries (m=1),
    a pool from a Full source-layer scan, a Reindex layer with its own index
    queries, then a Reuse layer on the Reindex selection.  One sequence is
    recomputed by the oracle (its 1M-entry cache included)."""
    B, N = 16, 1 << 20
    w = Weights(3)
    rope = csa2.rope_table(N).to(DEV)
    cache = csa2.Cache(B, N, 1)
    ws_cw = csa2.Workspace(1 << 16)
    for b in range(B):
        write_sequence(csa2, cache, b, N, w, rope, ws_cw, seed=3)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    del rope
    scale = 1 / math.sqrt(512)
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=DEV)
    swa_base = torch.full((B,), N - WIN, dtype=torch.int64, device=DEV)
    layers = []
    for l in range(3):
        layers.append(dict(q_idx=synth.torch_normal(31 + 10 * l, (B, 1, 32, 128), torch.bfloat16, DEV),
                           w_head=synth.torch_normal(32 + 10 * l, (B, 1, 32), torch.float32, DEV),
                           q=synth.torch_normal(33 + 10 * l, (B, 1, 64, 512), torch.bfloat16, DEV),
                           swa=synth.torch_swa_rows(34 + 10 * l, (B, WIN), DEV),
                           sel=torch.empty((B, 1, K_SEL), dtype=torch.int32, device=DEV),
                           out=torch.empty((B, 1, 64, 512), dtype=torch.bfloat16, device=DEV)))
    pool = torch.empty((B, 1, M_BLK), dtype=torch.int32, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, B, 1, N, M_BLK, K_SEL))
    for l, mode in enumerate((csa2.MODE_FULL, csa2.MODE_REINDEX, csa2.MODE_REUSE)):
        L = layers[l]
        csa2.decode(mode, cache, q_pos=q_pos, q=L["q"].view(torch.int16), swa=L["swa"].view(torch.int16),
                    swa_base_pos=swa_base, scale=scale, sel=L["sel"] if l < 2 else layers[1]["sel"],
                    out=L["out"].view(torch.int16), ws=ws, M=M_BLK, max_n=N, q_idx=L["q_idx"].view(torch.int16),
                    w_head=L["w_head"], pool_blocks=pool)
    st, detail = ws.sync_status()
    assert st == 0, (st, detail)
    b = 5
    main, codes, scales = oracle_sequence_cache(3, b, N, 1, w, oracle.rope_table(N))
    h = [{k: host(v) for k, v in L.items() if k != "out"} for L in layers]
    got_pool = host(pool)[b, 0]
    # source layer: the pool
    s0 = oracle.index_scores(h[0]["q_idx"][b, 0], h[0]["w_head"][b, 0], codes, scales)
    check_pool(got_pool, oracle.block_topm(s0, N, M_BLK), s0, N, "source-layer pool")
    # source layer: its own top-512 over all 1M visible entries (a row this long
    # has its chosen ids put in order by the bitonic sort of the resolve step)
    got0 = h[0]["sel"][b, 0]
    want0 = oracle.select_topk(s0, np.arange(N), K_SEL)
    cases.assert_set_within_tie_window(got0, want0, lambda j: s0[j], what="Full sel at 1M")
    assert np.all(np.diff(got0) > 0) and got0.min() >= 0 and got0.max() < N, "Full sel ascending, in range"
    # Reindex: the layer's own scores over the pool, top-512
    dom = oracle.pool_entries(got_pool, N)
    s1 = np.full(N, -np.inf)
    s1[dom] = oracle.index_scores(h[1]["q_idx"][b, 0], h[1]["w_head"][b, 0], codes, scales, dom)
    want1 = oracle.select_topk(s1, dom, K_SEL)
    got1 = h[1]["sel"][b, 0]
    cases.assert_set_within_tie_window(got1, want1, lambda j: s1[j], what="reindex sel")
    assert set(got1[got1 >= 0]) <= set(dom)
    for l in (1, 2):
        cases.check_attention(bf16_to_f32(layers[l]["out"])[b, 0],
                              oracle.attention(h[l]["q"][b, 0], got1, main, h[l]["swa"][b], N - WIN, N - 1, scale),
                              f"layer {l} attention")


# ------------------------------------------------------------------ config 5
def test_config5_prefill_chunk_of_8192_tokens(csa2):
    """Encoder source layer (m=2): a 131,072-token prefix plus an 8192-token chunk
    (69,632 entries), 8192 causal queries in one Full call, each with its own
    top-512 over the entries visible to it plus its 128-row window.  18 queries
    (first, last, 16 evenly spaced) are recomputed by the oracle."""
    m, P, C = 2, 131072, 8192
    T = P + C
    N = T // m
    w = Weights(4)
    rope = csa2.rope_table(N).to(DEV)
    cache = csa2.Cache(1, N, m)
    ws_cw = csa2.Workspace(1 << 16)
    write_sequence(csa2, cache, 0, T, w, rope, ws_cw, seed=4)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    Q, S = C, C + WIN - 1
    q_pos = torch.arange(P, T, dtype=torch.int64, device=DEV)[None]
    swa_base = torch.full((1,), P - (WIN - 1), dtype=torch.int64, device=DEV)
    q_idx = synth.torch_normal(41, (1, Q, 32, 128), torch.bfloat16, DEV)
    w_head = synth.torch_normal(42, (1, Q, 32), torch.float32, DEV)
    q = synth.torch_normal(43, (1, Q, 64, 512), torch.bfloat16, DEV)
    swa = synth.torch_swa_rows(44, (1, S), DEV)
    pool = torch.empty((1, Q, M_BLK), dtype=torch.int32, device=DEV)
    sel = torch.empty((1, Q, K_SEL), dtype=torch.int32, device=DEV)
    out = torch.empty((1, Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, 1, Q, N, M_BLK, K_SEL))
    scale = 1 / math.sqrt(512)
    csa2.decode(csa2.MODE_FULL, cache, q_pos=q_pos, q=q.view(torch.int16), swa=swa.view(torch.int16),
                swa_base_pos=swa_base, scale=scale, sel=sel, out=out.view(torch.int16), ws=ws, M=M_BLK,
                max_n=N, q_idx=q_idx.view(torch.int16), w_head=w_head, pool_blocks=pool)
    st, detail = ws.sync_status()
    assert st == 0, (st, detail)
    main, codes, scales = oracle_sequence_cache(4, 0, T, m, w, oracle.rope_table(N))
    got_pool, got_sel = host(pool)[0], host(sel)[0]
    h_qidx, h_w, h_q, h_swa = host(q_idx)[0], host(w_head)[0], host(q)[0], host(swa)[0]
    picks = np.unique(np.concatenate([[0, Q - 1], np.linspace(0, Q - 1, 16).astype(np.int64)]))
    for qi in picks:
        t = P + int(qi)
        nv = oracle.visible_entries(t, m, N)
        s = oracle.index_scores(h_qidx[qi], h_w[qi], codes, scales, np.arange(nv))
        pb = oracle.block_topm(s, nv, M_BLK)
        check_pool(got_pool[qi], pb, s, nv, f"query {qi} pool")
        sl = oracle.select_topk(s, np.arange(nv), K_SEL)
        cases.assert_set_within_tie_window(got_sel[qi], sl, lambda j: s[j], what=f"query {qi} sel")
        got_o = bf16_to_f32(out[0, int(qi)])
        cases.check_attention(got_o, oracle.attention(h_q[qi], got_sel[qi], main, h_swa, P - (WIN - 1), t, scale),
                              f"query {qi} attention")
        if set(got_sel[qi]) == set(sl):
            cases.check_attention(got_o, oracle.attention(h_q[qi], sl, main, h_swa, P - (WIN - 1), t, scale),
                                  f"query {qi} end to end")
