"""GPU parity of the FP8 sliding-window variant: the E4M3 window quantiser
(bit-exact against the oracle) and the attention reading E4M3 window rows
(against the oracle's attention over those rows, and bit-identical to the
attention over bf16 rows that hold the same values)."""
import numpy as np
import pytest

import oracle
import synth
from tests import cases
from tests.test_gpu_parity import DEV, GpuLayer, bf16_to_f32, dev, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp4_kv_cache_csa2_gb300 as m
    m.load()
    return m


def test_swa_quantize_fp8_bit_exact(csa2):
    """Window rows plus values that tie, saturate, underflow or are subnormal in E4M3."""
    g = synth.rng(900)
    rows = synth.swa_rows(g, 37)
    extra = np.concatenate([np.array([448, 449, 464, 500, 1e4, -1e4, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -9,
                                      1.0625, -1.1875, 0.0, -0.0, 2.0 ** -12], np.float32),
                            g.standard_normal(498).astype(np.float32) * 50.0])
    rows = np.concatenate([rows, synth.f32_to_bf16_bits(extra).reshape(1, 512)])
    out = torch.empty((38, 512), dtype=torch.uint8, device=DEV)
    csa2.swa_quantize_fp8(dev(rows), out)
    np.testing.assert_array_equal(host(out), oracle.swa_fp8_quantize(rows))


def _reuse(csa2, L, case, sel, swa, fp8):
    out = torch.empty((case.B, case.Q, 64, 512), dtype=torch.int16, device=DEV)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_REUSE, case.B, case.Q, case.n_entries, 8,
                                                   sel.shape[-1]), device=DEV)
    csa2.decode(csa2.MODE_REUSE, L.cache, q_pos=L.q_pos, q=L.q, swa=swa, swa_base_pos=L.swa_base,
                scale=case.scale, sel=sel, out=out, ws=ws, swa_fp8=fp8)
    assert ws.sync_status()[0] == 0
    return out


@pytest.mark.parametrize("K,q_pos", [(256, [[1499, 1000, 60]]), (37, [[0, 700, 1499]])])
def test_decode_fp8_window_matches_oracle(csa2, K, q_pos):
    """Reuse layers over a given selection with E4M3 window rows, including
    queries whose window is clipped at position 0."""
    case = cases.make_case(B=1, T=1500, m=1, Q=3, M=8, K=K, seed=910 + K, q_pos=np.array(q_pos))
    L = GpuLayer(csa2, case)
    g = np.random.default_rng(K)
    sel = np.full((1, 3, K), -1, np.int32)
    for qi in range(3):
        k = max(1, K - 3)
        sel[0, qi, :k] = g.choice(1500, k, replace=False)
    swa8 = torch.empty((1, case.S, 512), dtype=torch.uint8, device=DEV)
    csa2.swa_quantize_fp8(L.swa, swa8)
    fp8_or = oracle.swa_fp8_quantize(case.swa)
    np.testing.assert_array_equal(host(swa8), fp8_or)
    got = bf16_to_f32(_reuse(csa2, L, case, dev(sel), swa8, True))
    main, _, _ = cases.oracle_cache(case)
    for qi in range(3):
        want = oracle.attention(case.q[0, qi], sel[0, qi], main[0], fp8_or[0], case.swa_base[0], case.q_pos[0, qi],
                                case.scale)
        cases.check_attention(got[0, qi], want, f"q{qi}")


def test_decode_fp8_window_equals_bf16_rows_of_its_values(csa2):
    """Full mode: the FP8 window path and the bf16 path given rows holding the
    E4M3 values produce the same selection and bit-identical outputs."""
    case = cases.make_case(B=2, T=2 * 900, m=2, Q=2, M=32, K=128, seed=930)
    L = GpuLayer(csa2, case)
    swa8 = torch.empty((2, case.S, 512), dtype=torch.uint8, device=DEV)
    csa2.swa_quantize_fp8(L.swa, swa8)
    as_bf16 = dev(synth.f32_to_bf16_bits(oracle.e4m3_values()[host(swa8)].astype(np.float32)))
    outs = []
    for swa, fp8 in ((swa8, True), (as_bf16, False)):
        sel = torch.empty((2, 2, case.K), dtype=torch.int32, device=DEV)
        pool = torch.empty((2, 2, case.M), dtype=torch.int32, device=DEV)
        out = torch.empty((2, 2, 64, 512), dtype=torch.int16, device=DEV)
        ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, 2, 2, case.n_entries, case.M, case.K),
                            device=DEV)
        csa2.decode(csa2.MODE_FULL, L.cache, q_pos=L.q_pos, q=L.q, swa=swa, swa_base_pos=L.swa_base,
                    scale=case.scale, sel=sel, out=out, ws=ws, M=case.M, max_n=case.n_entries, q_idx=L.q_idx,
                    w_head=L.w_head, pool_blocks=pool, swa_fp8=fp8)
        assert ws.sync_status()[0] == 0
        outs.append((host(sel), host(out)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_swa_fp8_argument_errors(csa2):
    x = torch.zeros((4, 512), dtype=torch.int16, device=DEV)
    out = torch.empty((4, 512), dtype=torch.uint8, device=DEV)
    lib = csa2.load()
    assert lib.csa2_swa_quantize_fp8(x.data_ptr(), 2, out.data_ptr() + 1, None) == 1      # misaligned output
    assert lib.csa2_swa_quantize_fp8(x.data_ptr(), -1, out.data_ptr(), None) == 1         # negative count
    assert lib.csa2_swa_quantize_fp8(None, 2, out.data_ptr(), None) == 1                  # null input
    csa2.swa_quantize_fp8(x[:0], out[:0])                      # no rows: nothing to do
