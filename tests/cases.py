"""Seeded test cases (host numpy) and the parity comparators used by the tests.

Inputs come from ``synth``; expected values come from ``oracle``.  Nothing here
imports the CUDA binding."""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

import oracle
import synth


@dataclass
class LayerCase:
    """One sequence batch of a CSA2 source layer plus its decode queries."""
    B: int
    T: int                      # raw tokens written per sequence
    m: int
    Q: int
    M: int
    K: int
    S: int                      # SWA rows supplied per sequence
    seed: int
    q_pos: np.ndarray           # [B, Q] raw positions
    swa_base: np.ndarray        # [B]
    x: np.ndarray               # bf16 bits [B, T, 512]
    w0: np.ndarray
    w1: np.ndarray
    w_idx: np.ndarray           # bf16 bits [128, 512]
    q_idx: np.ndarray           # bf16 bits [B, Q, 32, 128]
    w_head: np.ndarray          # [B, Q, 32]
    q: np.ndarray               # bf16 bits [B, Q, 64, 512]
    swa: np.ndarray             # bf16 bits [B, S, 512]
    scale: float = 1 / math.sqrt(512)

    @property
    def n_entries(self) -> int:
        return self.T // self.m


def make_case(B, T, m, Q, M, K, seed, q_pos=None, S=None) -> LayerCase:
    g = synth.rng(seed)
    x = synth.latents(g, B, T)
    w0, w1 = synth.compressor_weights(g)
    w_idx = synth.index_projection(g)
    if q_pos is None:
        q_pos = np.tile(np.arange(T - Q, T), (B, 1))
    q_pos = np.asarray(q_pos, np.int64).reshape(B, Q)
    lo = max(0, int(q_pos.min()) - (oracle.WINDOW - 1))
    hi = int(q_pos.max()) + 1
    if S is None:
        S = hi - lo
    swa_base = np.full(B, lo, np.int64)
    q_idx = synth.index_queries(g, B, Q)
    w_head = synth.head_weights(g, B, Q)
    q = synth.main_queries(g, B, Q)
    swa = synth.swa_rows(g, B, S)
    return LayerCase(B, T, m, Q, M, K, S, seed, q_pos, swa_base, x, w0, w1, w_idx, q_idx, w_head, q, swa)


def config1_case() -> LayerCase:
    """Tiny Full layer (m = 2): 1 sequence, 4096 tokens -> 2048 entries, M = 128,
    K = 256, 4 queries at raw positions 4092..4095 (they see 2046, 2047, 2047 and
    2048 entries), 128-row bf16 window, seed 0."""
    return make_case(B=1, T=4096, m=2, Q=4, M=128, K=256, seed=0,
                     q_pos=np.array([[4092, 4093, 4094, 4095]]))


def oracle_cache(case: LayerCase, entry0: int = 0):
    """Oracle cache write of every sequence: (main [B,n,288], codes [B,n,64], scales [B,n,4])."""
    mains, codes, scales = [], [], []
    cs = oracle.rope_table(entry0 + case.n_entries)
    for b in range(case.B):
        mk, c, s = oracle.compress_quantize(case.x[b], case.m, case.w0, case.w1, case.w_idx, entry0, cs=cs)
        mains.append(mk)
        codes.append(c)
        scales.append(s)
    return np.stack(mains), np.stack(codes), np.stack(scales)


# ---------------------------------------------------------------- comparators
def assert_set_within_tie_window(got: np.ndarray, want: np.ndarray, score_of, rel: float = 1e-4, what=""):
    """Index sets may differ only where the oracle score of the differing ids lies
    within ``rel`` (relative) of the oracle's k-th score."""
    g = set(int(v) for v in got if v >= 0)
    w = set(int(v) for v in want if v >= 0)
    assert len(g) == len(w), f"{what}: sizes differ {len(g)} vs {len(w)}"
    diff = g ^ w
    if not diff:
        return
    kth = min(score_of(j) for j in w)
    for j in diff:
        s = score_of(j)
        assert abs(s - kth) <= rel * abs(kth) or (math.isinf(s) and math.isinf(kth)), \
            f"{what}: id {j} score {s} outside the tie window of k-th {kth}"


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_attention(got_bf16_as_f32: np.ndarray, want: np.ndarray, what=""):
    e = rel_l2(got_bf16_as_f32.astype(np.float64), want)
    mx = float(np.max(np.abs(got_bf16_as_f32.astype(np.float64) - want)))
    assert e <= 1e-2 and mx <= 3e-2, f"{what}: rel-L2 {e:.3e} max-abs {mx:.3e}"
    return e, mx
