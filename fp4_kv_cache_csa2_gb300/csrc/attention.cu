// (c) Joint sparse + SWA attention over the shared 512-d latent (K = V), on
// the 5th-generation tensor cores.
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §3.3.2 (the readout
// concatenates the SWA KV with the selected main-KV entries into one sparse
// attention), §3.3.2.1 (key = value = the compressed content vector; the output
// is a convex combination of them), §2.4.4 (the FP4 cache is dequantised to a
// more precise format before attention: FP4 saves storage, it does not feed
// the matrix multiply); "4. 层维度(下):CSA2 与每 token 890 字节" §4.5.
//
// One thread-block cluster of C CTAs per query token, 128 keys per CTA: CTAs
// 0..C-2 take the K selected slots in runs of 128, CTA C-1 the 128 window
// positions.  In every CTA:
//   * keys land in shared memory as bf16 [128 keys][512] in 8 SW128 column
//     chunks of 64 dims: window rows by 2-D TMA straight from the bf16 window,
//     selected FP4 entries by bulk copies into a staging buffer followed by an
//     exact dequantisation (E2M1 x E4M3 has at most 6 significant bits);
//   * Q (64 heads x 512) streams through a 4-stage TMA ring;
//   * S^T = K Q^T is one M=128 (keys) x N=64 (heads) x K=512 tcgen05 bf16 MMA
//     chain into TMEM;
//   * row maxima are exchanged over distributed shared memory, P = exp(S - max)
//     is written as the K-major bf16 B operand of the second product;
//   * O^T = V^T P^T reuses the same key buffer as an MN-major A operand:
//     4 tiles of M=128 dims x N=64 heads x K=128 keys;
//   * row sums are exchanged; every CTA writes its share O_c / L of each 128-dim
//     tile as fp16 (relative rounding 2^-11, four times finer than the bf16
//     output) and bulk-copies the tiles it does not own into the owner's
//     receive slots over DSMEM; the owner adds the C shares in fp32, rounds to
//     bf16 and stores.
// All mbarrier waits are bounded; a timeout reports CSA2_ERR_TIMEOUT.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "params.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

constexpr int AT_THREADS = 256;
constexpr int AT_KEYS = 128;                  // keys per CTA (one M = 128 tile)
constexpr int AT_QSTAGES = 6;
constexpr int AT_CHUNK_BYTES = AT_KEYS * 128;            // [128 keys][64 dims] bf16 = 16 KB
constexpr int AT_OFF_K = 0;                              // 8 chunks, 128 KB
constexpr int AT_OFF_Q = 8 * AT_CHUNK_BYTES;             // 6 stages x 8 KB
constexpr int AT_OFF_SCR = AT_OFF_Q + AT_QSTAGES * 8192; // FP4 staging | S^T transposed | P
constexpr int AT_SCR_BYTES = AT_KEYS * MAIN_BYTES;       // 36,864
constexpr int AT_ST_ROW = AT_KEYS + 1;                   // padded fp32 row of S^T transposed
constexpr int AT_OFF_SMALL = AT_OFF_SCR + AT_SCR_BYTES;
constexpr int AT_SHARE_BYTES = 128 * H * 2;             // one O^T tile share in fp16: 16 KB
constexpr int AT_OFF_RECV = AT_OFF_Q;                    // 4 receive slots over the dead Q ring + scratch
// Shares are O_c / 128 (exact power-of-two scaling): |share| <= the largest |key|
// value, far inside the fp16 range.
constexpr float AT_SHARE_DIV = 128.0f;
constexpr int AT_TMEM_COLS = 512;                        // S^T: 64 cols, O^T: 4 x 64 cols

struct AtSmall {
  int kvalid[AT_KEYS];
  float loc_max[H];
  float loc_sum[H];
  float inv_l[H];
  float gmax[H];
  uint32_t lut[256];
  uint64_t bar_kv, bar_s, bar_o, bar_red;
  uint64_t bar_q[AT_QSTAGES], bar_qe[AT_QSTAGES];
  uint64_t bar_chunk[8];                 // chunk c of the keys is in shared memory (bf16, SW128)
  uint32_t tmem_base;
  int err;
};
constexpr int AT_SMEM = AT_OFF_SMALL + (int)sizeof(AtSmall) + 1024;
static_assert(AT_ST_ROW * H * 4 <= AT_SCR_BYTES, "S^T scratch must fit");
static_assert(4 * AT_SHARE_BYTES <= 8 * AT_CHUNK_BYTES, "O^T shares must fit over the keys");
static_assert(4 * AT_SHARE_BYTES <= AT_QSTAGES * 8192 + AT_SCR_BYTES, "receive slots must fit");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// byte offset of (row, byte) in a 1 KB-aligned SW128 region of 128-byte rows
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte) {
  return row * 128u + ((((byte >> 4) ^ (row & 7u)) << 4) | (byte & 15u));
}

__device__ __forceinline__ bool at_wait(uint64_t* bar, uint32_t parity, AtSmall& sm, WsHeader* hdr, int where) {
  if (tc::bar_wait(bar, parity)) return true;
  if (atomicExch(&sm.err, 1) == 0) report(hdr, CSA2_ERR_TIMEOUT, where);
  return false;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
attn_tc_kernel(AttnParams p, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_swa,
               int C) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* kbuf = smem + AT_OFF_K;
  unsigned char* qbuf = smem + AT_OFF_Q;
  unsigned char* scr = smem + AT_OFF_SCR;
  AtSmall& sm = *reinterpret_cast<AtSmall*>(smem + AT_OFF_SMALL);
  float* st = reinterpret_cast<float*>(scr);                 // S^T transposed: [64 heads][129] fp32
  __half* ostage = reinterpret_cast<__half*>(kbuf);          // 4 tiles x [128 dims][64 heads] fp16 shares
  __half* orecv = reinterpret_cast<__half*>(smem + AT_OFF_RECV); // up to 4 received shares

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int bq = blockIdx.x / C;
  const int b = bq / p.Q;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t = p.q_pos[bq];
  const bool window_cta = rank == C - 1;
  const int slot0 = rank * AT_KEYS;

  // ---------------- set-up
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, AT_TMEM_COLS);
  if (tid == 0) {
    tc::bar_init(&sm.bar_kv, 1);
    tc::bar_init(&sm.bar_s, 1);
    tc::bar_init(&sm.bar_o, 1);
    tc::bar_init(&sm.bar_red, 1);
    for (int i = 0; i < AT_QSTAGES; i++) {
      tc::bar_init(&sm.bar_q[i], 1);
      tc::bar_init(&sm.bar_qe[i], 1);
    }
    for (int i = 0; i < 8; i++) tc::bar_init(&sm.bar_chunk[i], 1);
    sm.err = 0;
    tc::bar_init_fence();
  }
  sm.lut[tid] = pack_bf16x2(e2m1_value(tid & 15u), e2m1_value((uint32_t)tid >> 4));
  if (tid < AT_KEYS) {                       // which keys of this CTA exist
    int kind = 0;
    if (!window_cta) {
      const int gs = slot0 + tid;
      if (gs < p.K) {
        const int32_t id = p.sel[(int64_t)bq * p.K + gs];
        if (id >= 0 && id < p.cap) kind = 1;
        else if (id >= p.cap) report(p.hdr, CSA2_ERR_BOUNDS, id);
      }
    } else {
      const int64_t pos = t - (WIN - 1) + tid;
      if (pos >= 0) {
        const int64_t row = pos - p.swa_base[b];
        if (row >= 0 && row < p.S) kind = 2;
        else report(p.hdr, CSA2_ERR_BOUNDS, pos);
      }
    }
    sm.kvalid[tid] = kind;
  }
  tc::fence_before_sync();
  __syncthreads();                       // local barriers and key flags visible (no remote access yet)
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  // ---------------- initial copies: window rows (window CTA) and Q chunks 0..5
  if (tid == 0) {
    if (window_cta) {
      if (p.S > 0) {         // rows outside this sequence's window are masked (kvalid == 0) but finite
        tc::bar_arrive_expect_tx(&sm.bar_kv, 8u * AT_CHUNK_BYTES);
        const int32_t row0 = (int32_t)((int64_t)b * p.S + (t - (WIN - 1) - p.swa_base[b]));
        for (int c = 0; c < 8; c++) tc::tma_load_2d(kbuf + c * AT_CHUNK_BYTES, &map_swa, c * 64, row0, &sm.bar_kv);
      } else {
        tc::bar_arrive_expect_tx(&sm.bar_kv, 0u);
      }
    }
    for (int c = 0; c < AT_QSTAGES; c++) {
      tc::bar_arrive_expect_tx(&sm.bar_q[c], 8192u);
      tc::tma_load_2d(qbuf + c * 8192, &map_q, c * 64, bq * H, &sm.bar_q[c]);
    }
  }

  // ---------------- keys: FP4 entries by 16-byte asynchronous copies, then warp w
  // dequantises 64-dim chunk w and publishes it on its own mbarrier
  if (!window_cta) {
    for (int i = tid; i < AT_KEYS * (MAIN_BYTES / 16); i += AT_THREADS) {
      const int s = i / (MAIN_BYTES / 16), part = i % (MAIN_BYTES / 16);
      if (sm.kvalid[s] == 1) {
        const int32_t id = p.sel[(int64_t)bq * p.K + slot0 + s];
        const unsigned char* src = p.main_kv + ((int64_t)b * p.cap + id) * MAIN_BYTES + part * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                     :: "r"(tc::smem_u32(scr + s * MAIN_BYTES + part * 16)), "l"(src) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int c = warp;
    unsigned char* rowp = kbuf + c * AT_CHUNK_BYTES;
    for (int s = lane; s < AT_KEYS; s += 32) {
      if (sm.kvalid[s] == 1) {
        const unsigned char* ent = scr + s * MAIN_BYTES;
        const uint4 c0 = *reinterpret_cast<const uint4*>(ent + c * 32);
        const uint4 c1 = *reinterpret_cast<const uint4*>(ent + c * 32 + 16);
        const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(ent + 256 + c * 4);
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int g = 0; g < 4; g++) {                      // 16 channels per E4M3 scale
          const float sc = e4m3_value((sc4 >> (8 * g)) & 255u);
          const uint32_t sc2 = pack_bf16x2(sc, sc);
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 8; k++) {
            const uint32_t byte = (cw[2 * g + (k >> 2)] >> (8 * (k & 3))) & 255u;
            asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[k]) : "r"(sm.lut[byte]), "r"(sc2));
          }
          *reinterpret_cast<uint4*>(rowp + sw128((uint32_t)s, (uint32_t)g * 32u)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(rowp + sw128((uint32_t)s, (uint32_t)g * 32u + 16u)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 8; u++)
          *reinterpret_cast<uint4*>(rowp + sw128((uint32_t)s, (uint32_t)u * 16u)) = make_uint4(0, 0, 0, 0);
      }
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::bar_arrive(&sm.bar_chunk[c]);
  } else if (p.S == 0) {                                   // no window rows supplied: zero keys
    for (int i = tid; i < 8 * AT_CHUNK_BYTES / 16; i += AT_THREADS)
      reinterpret_cast<uint4*>(kbuf)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    __syncthreads();
  }

  // ---------------- S^T = K Q^T  (M = 128 keys, N = 64 heads, K = 512 dims); the
  // issuing thread also refills Q stages 0 and 1 with chunks 6 and 7
  if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc_s = tc::idesc_bf16(AT_KEYS, H, 0, 0);
    if (window_cta) at_wait(&sm.bar_kv, 0, sm, p.hdr, 11);
    for (int c = 0; c < 8; c++) {
      const int s = c % AT_QSTAGES;
      if (!window_cta && !at_wait(&sm.bar_chunk[c], 0, sm, p.hdr, 16)) break;
      if (!at_wait(&sm.bar_q[s], (c / AT_QSTAGES) & 1, sm, p.hdr, 12)) break;
      tc::fence_after_sync();
      const uint32_t a0 = tc::smem_u32(kbuf + c * AT_CHUNK_BYTES), b0 = tc::smem_u32(qbuf + s * 8192);
#pragma unroll
      for (int ks = 0; ks < 4; ks++)
        tc::mma_bf16(tmem, tc::smem_desc(a0 + ks * 32, 16, 1024, tc::SW_128B),
                     tc::smem_desc(b0 + ks * 32, 16, 1024, tc::SW_128B), idesc_s, (c | ks) ? 1u : 0u);
      tc::commit(&sm.bar_qe[s]);
      if (c == 2 || c == 3) {              // stage c-2 is free once chunk c-2's MMAs finished
        const int r = c - 2;
        if (!at_wait(&sm.bar_qe[r], 0, sm, p.hdr, 10)) break;
        tc::bar_arrive_expect_tx(&sm.bar_q[r], 8192u);
        tc::tma_load_2d(qbuf + r * 8192, &map_q, (r + AT_QSTAGES) * 64, bq * H, &sm.bar_q[r]);
      }
    }
    tc::commit(&sm.bar_s);
  }
  __syncwarp();

  // ---------------- S^T from TMEM -> scaled, masked, transposed into smem
  at_wait(&sm.bar_s, 0, sm, p.hdr, 13);
  tc::fence_after_sync();
  {
    const int q4 = warp & 3, half = warp >> 2;
    const int m = q4 * 32 + lane;                   // key row
    float v[32];
    tc::tmem_ld_x32(tmem + ((uint32_t)(q4 * 32) << 16) + half * 32, v);
    const bool valid = sm.kvalid[m] != 0;
#pragma unroll
    for (int j = 0; j < 32; j++) st[(half * 32 + j) * AT_ST_ROW + m] = valid ? v[j] * p.scale : -INFINITY;
  }
  __syncthreads();
  // row maxima of this CTA (warp w: heads 8w .. 8w+7)
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int h = warp * 8 + i;
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; j++) mx = fmaxf(mx, st[h * AT_ST_ROW + lane + 32 * j]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    if (lane == 0) sm.loc_max[h] = mx;
  }
  cluster.sync();                                          // #1: maxima visible
  if (tid < H) {
    float gm = -INFINITY;
    for (int c = 0; c < C; c++) gm = fmaxf(gm, cluster.map_shared_rank(sm.loc_max, c)[tid]);
    sm.gmax[tid] = (gm == -INFINITY) ? 0.f : gm;
  }
  __syncthreads();
  float pv[8][4];
  float lsum[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int h = warp * 8 + i;
    const float gm = sm.gmax[h];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 4; j++) {                 // keys 2*lane, 2*lane+1, 64+2*lane, 65+2*lane
      const int k = (j >> 1) * 64 + 2 * lane + (j & 1);
      const float s_ = st[h * AT_ST_ROW + k];
      const float e = (s_ == -INFINITY) ? 0.f : __expf(s_ - gm);
      pv[i][j] = e;
      sum += e;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    lsum[i] = sum;
  }
  __syncthreads();                                         // every read of S^T is done: P overwrites it
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int h = warp * 8 + i;
    if (lane == 0) sm.loc_sum[h] = lsum[i];
#pragma unroll
    for (int blk = 0; blk < 2; blk++)
      *reinterpret_cast<uint32_t*>(scr + blk * 8192 + sw128((uint32_t)h, (uint32_t)(4 * lane))) =
          pack_bf16x2(pv[i][2 * blk], pv[i][2 * blk + 1]);
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // ---------------- O^T = V^T P^T  (4 tiles of M = 128 dims, N = 64 heads, K = 128 keys)
  if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc_o = tc::idesc_bf16(128, H, 1, 0);
    const uint32_t kb = tc::smem_u32(kbuf), pb = tc::smem_u32(scr);
    for (int tile = 0; tile < 4; tile++) {
#pragma unroll
      for (int ks = 0; ks < AT_KEYS / 16; ks++) {
        const uint64_t ad = tc::smem_desc(kb + (2 * tile) * AT_CHUNK_BYTES + ks * 2048, AT_CHUNK_BYTES, 1024,
                                          tc::SW_128B);
        const uint64_t bd = tc::smem_desc(pb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, tc::SW_128B);
        tc::mma_bf16(tmem + 64 + tile * 64, ad, bd, idesc_o, ks ? 1u : 0u);
      }
    }
    tc::commit(&sm.bar_o);
  }
  __syncwarp();
  at_wait(&sm.bar_o, 0, sm, p.hdr, 14);
  tc::fence_after_sync();
  // this CTA's share O_c / L per tile as fp16 [dim][head], 16-byte units swizzled by dim
  {
    const int q4 = warp & 3, half = warp >> 2;
    uint32_t ta[4][32];
#pragma unroll
    for (int tile = 0; tile < 4; tile++) {       // issue all four TMEM loads, then wait once
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                   "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                   : "=r"(ta[tile][0]), "=r"(ta[tile][1]), "=r"(ta[tile][2]), "=r"(ta[tile][3]), "=r"(ta[tile][4]),
                     "=r"(ta[tile][5]), "=r"(ta[tile][6]), "=r"(ta[tile][7]), "=r"(ta[tile][8]), "=r"(ta[tile][9]),
                     "=r"(ta[tile][10]), "=r"(ta[tile][11]), "=r"(ta[tile][12]), "=r"(ta[tile][13]), "=r"(ta[tile][14]),
                     "=r"(ta[tile][15]), "=r"(ta[tile][16]), "=r"(ta[tile][17]), "=r"(ta[tile][18]), "=r"(ta[tile][19]),
                     "=r"(ta[tile][20]), "=r"(ta[tile][21]), "=r"(ta[tile][22]), "=r"(ta[tile][23]), "=r"(ta[tile][24]),
                     "=r"(ta[tile][25]), "=r"(ta[tile][26]), "=r"(ta[tile][27]), "=r"(ta[tile][28]), "=r"(ta[tile][29]),
                     "=r"(ta[tile][30]), "=r"(ta[tile][31])
                   : "r"(tmem + ((uint32_t)(q4 * 32) << 16) + 64 + tile * 64 + half * 32) : "memory");
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    const int d = q4 * 32 + lane;                 // dim row inside a tile
#pragma unroll
    for (int tile = 0; tile < 4; tile++) {
      __half* row = ostage + tile * (128 * H) + d * H;
#pragma unroll
      for (int u = 0; u < 4; u++) {               // 16-byte units = 8 heads: half*32 + 8u .. +7
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int j = 8 * u + 2 * e;
          const __half2 h2 = __floats2half2_rn(__uint_as_float(ta[tile][j]) * (1.0f / AT_SHARE_DIV),
                                               __uint_as_float(ta[tile][j + 1]) * (1.0f / AT_SHARE_DIV));
          w[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        const int unit = (half * 4 + u) ^ (d & 7);
        *reinterpret_cast<uint4*>(row + unit * 8) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  tc::fence_proxy_async_smem();
  cluster.sync();                                          // #2: shares staged, receive slots free, sums visible
  if (tid < H) {
    float L = 0.f;
    for (int c = 0; c < C; c++) L += cluster.map_shared_rank(sm.loc_sum, c)[tid];
    sm.inv_l[tid] = (L > 0.f) ? AT_SHARE_DIV / L : 0.f;
  }
  __syncthreads();
  // no remote shared-memory reads after this point: let the cluster go ahead
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // ---------------- cluster reduction: tile t is owned by CTA t % C; the others send
  // their fp16 share into the owner's slot (j * (C - 1) + sender index)
  int owned = 0;
  for (int tile = rank; tile < 4; tile += C) owned++;
  if (tid == 0) {
    if (owned) tc::bar_arrive_expect_tx(&sm.bar_red, (uint32_t)(owned * (C - 1) * AT_SHARE_BYTES));
    for (int tile = 0; tile < 4; tile++) {
      const int owner = tile % C;
      if (owner == rank) continue;
      const int j = tile / C;
      const int slot = j * (C - 1) + (rank < owner ? rank : rank - 1);
      const uint32_t src = tc::smem_u32(ostage + tile * (128 * H));
      uint32_t dst, rbar;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(tc::smem_u32(orecv + slot * (128 * H))), "r"(owner));
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(tc::smem_u32(&sm.bar_red)), "r"(owner));
      asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                   :: "r"(dst), "r"(src), "r"(AT_SHARE_BYTES), "r"(rbar) : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  if (owned) {
    at_wait(&sm.bar_red, 0, sm, p.hdr, 15);
    uint16_t* out = p.out + (int64_t)bq * H * D;
    int j = 0;
    for (int tile = rank; tile < 4; tile += C, j++) {
      // thread: dim d (consecutive lanes -> coalesced bf16 stores per head row), 8-head unit u
      for (int task = tid; task < 128 * 8; task += AT_THREADS) {
        const int d = task & 127, u = task >> 7;
        const int off = d * H + ((u ^ (d & 7)) << 3);
        float acc[8];
        {
          const uint4 v = *reinterpret_cast<const uint4*>(ostage + tile * (128 * H) + off);
          const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const float2 f = __half22float2(h2[e]);
            acc[2 * e] = f.x;
            acc[2 * e + 1] = f.y;
          }
        }
        for (int r = 0; r < C - 1; r++) {
          const uint4 v = *reinterpret_cast<const uint4*>(orecv + (j * (C - 1) + r) * (128 * H) + off);
          const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const float2 f = __half22float2(h2[e]);
            acc[2 * e] += f.x;
            acc[2 * e + 1] += f.y;
          }
        }
        uint16_t* o = out + (u * 8) * D + tile * 128 + d;
#pragma unroll
        for (int e = 0; e < 8; e++)
          o[e * D] = (uint16_t)(pack_bf16x2(acc[e] * sm.inv_l[u * 8 + e], 0.f) & 0xFFFFu);
      }
    }
  }
  if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  tc::fence_before_sync();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // every CTA done reading ours
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 at_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// bf16 matrix [rows][512] with SW128 boxes of 64 columns x box_rows rows.
static bool encode_bf16_rows512(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = at_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t attn_partials_bytes(int64_t, int) { return 0; }

cudaError_t launch_attention(AttnParams p, int B, float*, cudaStream_t stream) {
  const int64_t BQ = (int64_t)B * p.Q;
  if (BQ == 0) return cudaSuccess;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  CUtensorMap map_q, map_swa;
  if (!encode_bf16_rows512(&map_q, p.q, (uint64_t)BQ * H, 64)) return cudaErrorInvalidValue;
  const uint64_t swa_rows = (uint64_t)B * (uint64_t)(p.S > 0 ? p.S : 1);
  if (!encode_bf16_rows512(&map_swa, p.swa, swa_rows, AT_KEYS)) return cudaErrorInvalidValue;
  const int C = (p.K + AT_KEYS - 1) / AT_KEYS + 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(BQ * C));
  cfg.blockDim = dim3(AT_THREADS);
  cfg.dynamicSmemBytes = AT_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel, p, map_q, map_swa, C);
}

}  // namespace csa2
