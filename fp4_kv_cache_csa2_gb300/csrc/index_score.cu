// (b) Lightning-indexer scores  s(t,j) = sum_h w_h * ReLU(q_h . k_j)
// over 32 index heads x 128 dims, with MXFP4 queries and keys, on the
// 5th-generation tensor cores (tcgen05, kind::mxf4 block-scaled MMA).
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4 (the Full layer
// scores every causally visible main-KV position; Reindex layers score only the
// candidate pool), §2.4.4 (FP4 indexer Q and K); "4. 层维度(下):CSA2 与每 token
// 890 字节" §4.4 (index K is OCP MXFP4: E2M1 + one E8M0 scale per 32), §4.7.
//
// One CTA scores a run of 128-entry tiles for a group of NQ queries of one
// sequence (NQ = 1 for decode and pool scans; NQ = 5 when a sequence brings many
// queries, as a prefill chunk does, so that every tile of keys loaded feeds a
// 160-column MMA instead of a 32-column one; three 160-column accumulators and
// the scale-word columns fill the 512 TMEM columns):
//   warp 0      producer: full scans load 128-entry tiles of index-K codes
//               (SW64 K-major, 64 B per entry) with a 3-D tensor map that puts
//               slot 4g + q of the tile in row 32q + g, and the 4-byte E8M0
//               words with 1-D bulk copies (mbarrier expect-tx); pool scans
//               gather the 16 candidate blocks of a tile with cp.async, one
//               512-byte block per warp instruction, into the same rows.
//               6-stage ring.
//   warp 1..I   MMA issuers (I = 2 for NQ = 1, 3 for NQ = 5; warp 1 owns
//               TMEM): issuer k takes every I-th tile into its own TMEM
//               accumulator: one tcgen05.cp of the tile's 512 bytes of scale
//               words into TMEM (with that row order, 16 contiguous bytes per
//               lane of every lane quarter: row 32q + g reads word q), then two
//               M=128 N=32*NQ K=64 block-scaled MMAs.  A single issuer is bound
//               by its own wait latencies, not by the tensor core.
//   warp I+1    publisher: turns the TMA completions (mbarriers) into shared
//               words the issuers poll.
//   the rest    4*NQ epilogue warps, one per (TMEM lane quarter, query): 32 head
//               dot products from TMEM -> ReLU -> weighted sum -> score.
// The queries are quantised once per CTA (the B operand, 2 KB per query, and
// its scale words: head n of query j -> lane n of every lane quarter, column
// base + j).
// Products of E2M1 values scaled by powers of two are exact; the accumulation
// is fp32.  Every mbarrier wait is bounded and reports CSA2_ERR_TIMEOUT.
#include <cstddef>
#include <cudaTypedefs.h>

#include "host_once.cuh"
#include "index_query.cuh"
#include "params.cuh"
#include "tc.cuh"


namespace csa2 {

constexpr int IS_STAGES = 6;
constexpr int IS_TILE = 128;
constexpr int IS_CODES = IS_TILE * IDX_CODE_BYTES;         // 8192
constexpr int IS_STAGE_BYTES = IS_CODES + 1024;            // codes + 512 B scales, 1 KB aligned stride
constexpr int IS_POOL_MAX = CSA2_MAX_M;
constexpr int IS_GROUP = 5;                                 // queries per CTA for many-query sequences

// Warp roles: 0 producer; 1..ISSUERS MMA issuers (issuer k takes tiles
// i = k mod ISSUERS into accumulator k); ISSUERS+1 publisher; then 4*NQ
// epilogue warps, one per (TMEM lane quarter, query).
template <int NQ>
struct IsCfg {
  static constexpr int N = NQ * HI;                         // MMA N: query heads
  static constexpr int ISSUERS = NQ == 1 ? 2 : 3;           // = accumulators
  static constexpr int PUB_WARP = 1 + ISSUERS;
  static constexpr int EPI0 = PUB_WARP + 1;                 // first epilogue warp
  static constexpr int EPI_WARPS = 4 * NQ;
  static constexpr int THREADS = 32 * (EPI0 + EPI_WARPS);
  static constexpr int ACC_COL = 0;                         // ISSUERS accumulators of N columns
  static constexpr int SFA_COL = ISSUERS * N;               // 4 columns per stage
  static constexpr int SFB_COL = SFA_COL + 4 * IS_STAGES;   // NQ columns
  static constexpr int TMEM_COLS = NQ == 1 ? 128 : 512;
  static constexpr int MIN_CTAS = NQ == 1 ? 3 : 1;         // resident CTAs per SM (one issue chain each)
  static_assert(SFB_COL % 8 == 0 && SFB_COL + NQ <= TMEM_COLS, "TMEM columns");
};

template <int NQ>
struct IsSmem {
  uint8_t stage[IS_STAGES][IS_STAGE_BYTES];
  uint8_t qcodes[NQ * HI * IDX_CODE_BYTES];  // 2 KB per query, SW64
  int32_t pool[IS_POOL_MAX];
  float w[NQ * HI];
  uint32_t sfb[NQ * HI];                     // query scale words
  uint64_t full[IS_STAGES], empty[IS_STAGES];
  uint64_t acc_full[4];
  uint64_t test_bar;                         // test hook only: nothing ever arrives on it
  uint32_t ready[IS_STAGES];                 // tile i + 1 once tile i sits in stage i % IS_STAGES
  uint32_t acc_free[4];                      // epilogue warps done reading accumulator k, cumulative
  uint32_t tmem_base;
  volatile int abort_flag;
};
template <int NQ>
constexpr size_t is_smem_bytes() { return sizeof(IsSmem<NQ>) + 1024; }

// Shared-memory row of tile slot u: slot 4g + q sits in row 32q + g, so that
// the 16 bytes of scale words of slots 4g..4g+3 (contiguous as they arrive) are
// the words lane g of every TMEM lane quarter needs: row 32q + g takes word q.
__device__ __forceinline__ int is_tile_row(int u) { return 32 * (u & 3) + (u >> 2); }

// Bounded spin until the shared word reaches `target` (acquire); false on
// abort or timeout (which sets the abort flag and reports CSA2_ERR_TIMEOUT).
// The issuers poll plain words: after a thread has MMAs in flight, its
// mbarrier waits return markedly later than the barrier completes.
template <class Sm>
__device__ __forceinline__ bool poll_at_least(const uint32_t* word, uint32_t target, Sm& sm, WsHeader* hdr) {
  for (uint32_t it = 0; it < (1u << 26); it++) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(tc::smem_u32(word)) : "memory");
    if ((int32_t)(v - target) >= 0) return true;
    if (sm.abort_flag) return false;
    __nanosleep(32);          // leave the issue slots to the epilogue warps of this SM sub-partition
  }
  sm.abort_flag = 1;
  report(hdr, CSA2_ERR_TIMEOUT, 1);
  return false;
}

__device__ __forceinline__ void publish_word(uint32_t* word, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" :: "r"(tc::smem_u32(word)), "r"(v) : "memory");
}

template <class Sm>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Sm& sm, WsHeader* hdr) {
  if (sm.abort_flag) return false;
  for (int round = 0; round < 64; round++) {
    if (tc::bar_wait(bar, parity, 1u << 16)) return true;
    if (sm.abort_flag) return false;
  }
  sm.abort_flag = 1;
  report(hdr, CSA2_ERR_TIMEOUT, 1);
  return false;
}

template <int NQ, bool OFFSET>
__global__ void __launch_bounds__(IsCfg<NQ>::THREADS, IsCfg<NQ>::MIN_CTAS)
index_score_tc_kernel(IsParams p, const __grid_constant__ CUtensorMap map_tile) {
  using C = IsCfg<NQ>;
  extern __shared__ unsigned char smem_raw[];
  IsSmem<NQ>& sm = *reinterpret_cast<IsSmem<NQ>*>(tc::align_smem_1k(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int groups = (p.Q + NQ - 1) / NQ;    // query groups per sequence
  // grid: x = slice of the group's tiles, y = (sequence, query group), counted
  // from p.group0 when a call has more groups than one grid holds (OFFSET: the
  // launcher issues at most 65535 groups per launch).  Any arithmetic on the
  // block index here (a division of a linear index, a padded z plane, even the
  // offset) kept more values live and made the grouped scan 5-20 % slower, so
  // calls that fit one grid use the block index as it is.
  const int64_t group = OFFSET ? p.group0 + blockIdx.y : (int64_t)blockIdx.y;
  const int crank = (int)blockIdx.x;
  const int b = (int)(group / groups);
  const int qf = (int)(group % groups) * NQ;
  const int nq = p.Q - qf < NQ ? p.Q - qf : NQ;   // queries in this group
  const int64_t bq0 = (int64_t)b * p.Q + qf;
  const bool pool_mode = p.pool != nullptr;  // (NQ == 1 only)

  // ---- visible entries of each query; this CTA's tile range
  int64_t nvq[NQ];
  int64_t n_units = 0;                       // entries (full) or pool slots (pool)
#pragma unroll
  for (int j = 0; j < NQ; j++) {
    int64_t v = 0;
    if (j < nq) {
      v = visible_entries(p.q_pos[bq0 + j], p.m, p.n_entries[b]);
      if (v > p.cap) {
        if (tid == 0 && crank == 0) report(p.hdr, CSA2_ERR_BOUNDS, v);
        v = p.cap;
      }
      if (!pool_mode && v > p.max_n) {
        if (tid == 0 && crank == 0) report(p.hdr, CSA2_ERR_BOUNDS, v);
        v = p.max_n;
      }
    }
    nvq[j] = v;
    if (v > n_units) n_units = v;
  }
  if (pool_mode) n_units = (int64_t)p.M * BLK;
  const int64_t nv = nvq[0];
  const int64_t n_tiles = ceil_div(n_units, IS_TILE);
  const int64_t t0 = (int64_t)crank * p.entries_per_cta;
  int64_t t1 = t0 + p.entries_per_cta;
  if (t1 > n_tiles) t1 = n_tiles;
  const int n = (int)(t1 > t0 ? t1 - t0 : 0);
  if (n == 0) return;

  // ---- set-up
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, C::TMEM_COLS);
  if (tid == 0) {
    for (int s = 0; s < IS_STAGES; s++) {
      tc::bar_init(&sm.full[s], 1);
      tc::bar_init(&sm.empty[s], 1);
    }
    for (int k = 0; k < 4; k++) {
      tc::bar_init(&sm.acc_full[k], 1);
      sm.acc_free[k] = 0;
    }
    for (int s = 0; s < IS_STAGES; s++) sm.ready[s] = 0;
    tc::bar_init(&sm.test_bar, 1);
    sm.abort_flag = 0;
    tc::bar_init_fence();
  }
  for (int i = tid; i < NQ * HI; i += C::THREADS)
    sm.w[i] = i < nq * HI ? p.w_head[bq0 * HI + i] : 0.0f;
  if (pool_mode) {
    const int32_t* pool = p.pool + bq0 * p.M;
    for (int i = tid; i < p.M; i += C::THREADS) sm.pool[i] = pool[i];
  }
  if (warp == 0 && lane == 0) tc::prefetch_tensormap(&map_tile);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  // ---- quantise the queries (B operand); the scale word of head n of query j
  // goes to TMEM lane 32q + n, column SFB_COL + j, of every lane quarter q (the
  // MMA reads B scales from the quarter of the A row it is computing)
  if (warp >= C::EPI0 && warp < C::EPI0 + NQ) {
    const int j = warp - C::EPI0;
    if (j < nq) {
      quantize_index_query_warp(p.q_idx + (bq0 + j) * HI * DI, sm.qcodes + j * HI * IDX_CODE_BYTES,
                                sm.sfb + j * HI);
    } else {                                  // missing query of a partial group: zero codes, scores unused
      for (int i = lane; i < HI * IDX_CODE_BYTES / 16; i += 32)
        reinterpret_cast<uint4*>(sm.qcodes + j * HI * IDX_CODE_BYTES)[i] = make_uint4(0u, 0u, 0u, 0u);
      sm.sfb[j * HI + lane] = 0u;
    }
  }
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (warp >= C::EPI0 && warp < C::EPI0 + 4) {
#pragma unroll
    for (int j = 0; j < NQ; j++)
      tc::tmem_st_x1(tmem + ((uint32_t)((warp & 3) * 32) << 16) + C::SFB_COL + j, sm.sfb[j * HI + lane]);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  const int64_t row_base = (int64_t)b * p.cap;
  const int64_t rows_total = (int64_t)p.B * p.cap;

  if (warp == 0) {
    // ================= producer
    int issued = 0;
    if (p.test_withhold) {
      // test hook: a bounded wait on a barrier that no thread, copy or MMA
      // arrives on, before anything is issued; it gives up, and the abort
      // stops every role with nothing in flight
      if (lane == 0 && !tc::bar_wait(&sm.test_bar, 0, 1024u)) {
        sm.abort_flag = 1;
        report(p.hdr, CSA2_ERR_TIMEOUT, 2);
      }
      __syncwarp();
    }
    if (!pool_mode) {
      if (lane == 0) {
        for (int i = 0; i < n; i++) {
          const int s = i % IS_STAGES;
          if (sm.abort_flag) break;
          if (i >= IS_STAGES && !wait_or_abort(&sm.empty[s], ((i / IS_STAGES) - 1) & 1, sm, p.hdr)) break;
          const int64_t row0 = row_base + (t0 + i) * IS_TILE;
          int64_t rows = rows_total - row0;
          if (rows > IS_TILE) rows = IS_TILE;
          const uint32_t sbytes = (uint32_t)rows * IDX_SCALE_BYTES;     // cap % 8 == 0 -> multiple of 16
          tc::bar_arrive_expect_tx(&sm.full[s], IS_CODES + sbytes);
          tc::tma_load_3d(sm.stage[s], &map_tile, 0, (int32_t)(row0 / 4), 0, &sm.full[s]);
          tc::bulk_load(sm.stage[s] + IS_CODES, p.idx_scales + row0 * IDX_SCALE_BYTES, sbytes, &sm.full[s]);
          issued = i + 1;
        }
        if (sm.abort_flag) {
          // drain copies still in flight before the CTA exits
          for (int i = issued - 1; i >= 0 && i >= issued - IS_STAGES; i--)
            tc::bar_wait(&sm.full[i % IS_STAGES], (i / IS_STAGES) & 1, 1u << 20);
        }
      }
    } else {
      // 16 candidate blocks of 8 entries per tile.  One warp instruction copies
      // one whole block (512 contiguous code bytes, 16 per lane: entry l/4,
      // 16-byte chunk l%4) to the tile rows of its entries; lanes 2b and 2b+1
      // copy block b's 32 bytes of scale words.  A tile is published two tiles
      // later, once its copies have retired and been fenced for the tensor core.
      constexpr int LAG = 2;
      auto publish = [&](int i) {
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) publish_word(&sm.ready[i % IS_STAGES], (uint32_t)(i + 1));
      };
      for (int i = 0; i < n; i++) {
        const int s = i % IS_STAGES;
        if (sm.abort_flag) break;
        if (i >= IS_STAGES && !wait_or_abort(&sm.empty[s], ((i / IS_STAGES) - 1) & 1, sm, p.hdr)) break;
        uint8_t* codes = sm.stage[s];
        uint8_t* scl = sm.stage[s] + IS_CODES;
        const int64_t pl = (t0 + i) * 16 + (lane & 15);
        int32_t my_blk = (pl < p.M) ? sm.pool[pl] : -1;
        if (my_blk >= 0 && (int64_t)my_blk * BLK >= p.cap) my_blk = -1;   // reported by the epilogue
        const int r = lane >> 2, c = lane & 3;
#pragma unroll 4
        for (int sb = 0; sb < 16; sb++) {
          const int32_t blk = __shfl_sync(0xFFFFFFFFu, my_blk, sb);
          if (blk < 0) continue;
          const int u = sb * BLK + r;                       // slot of the tile
          const int trow = is_tile_row(u);
          const uint8_t* src = p.idx_codes + (row_base + (int64_t)blk * BLK) * IDX_CODE_BYTES + lane * 16;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                       :: "r"(tc::smem_u32(codes + trow * 64 + ((c ^ ((trow >> 1) & 3)) * 16))), "l"(src) : "memory");
        }
        {
          const int sb = lane >> 1, half = lane & 1;
          const int32_t blk = __shfl_sync(0xFFFFFFFFu, my_blk, sb);
          if (blk >= 0)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                         :: "r"(tc::smem_u32(scl + sb * 32 + half * 16)),
                            "l"(p.idx_scales + (row_base + (int64_t)blk * BLK) * IDX_SCALE_BYTES + half * 16) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (i >= LAG) {
          asm volatile("cp.async.wait_group %0;" :: "n"(LAG) : "memory");
          publish(i - LAG);
        }
        issued = i + 1;
      }
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      for (int i = issued - LAG < 0 ? 0 : issued - LAG; i < issued; i++) publish(i);
    }
  } else if (warp <= C::ISSUERS) {
    // ================= MMA issuer k: tiles k, k + ISSUERS, ... into accumulator k
    const int k = warp - 1;
    if (lane == 0) {
      const uint64_t bdesc = tc::smem_desc(tc::smem_u32(sm.qcodes), 16, 512, tc::SW_64B);
      constexpr uint32_t id0 = tc::idesc_mxf4(IS_TILE, C::N, 0, 0);
      constexpr uint32_t id1 = tc::idesc_mxf4(IS_TILE, C::N, 2, 2);
      const uint32_t d = tmem + C::ACC_COL + k * C::N;
      int use = 0;
      for (int i = k; i < n; i += C::ISSUERS, use++) {
        const int s = i % IS_STAGES;
        if (!poll_at_least(&sm.ready[s], (uint32_t)(i + 1), sm, p.hdr)) break;
        if (use > 0 && !poll_at_least(&sm.acc_free[k], (uint32_t)(C::EPI_WARPS * use), sm, p.hdr)) break;
        tc::fence_after_sync();
        const uint32_t sfa = tmem + C::SFA_COL + s * 4;
        // 32 rows x 16 bytes (scale words 4g..4g+3) to lanes 32q + g of every quarter q
        tc::tmem_cp_32x128b_warpx4(sfa, tc::smem_desc(tc::smem_u32(sm.stage[s] + IS_CODES), 128, 128, tc::SW_NONE));
        const uint64_t adesc = tc::smem_desc(tc::smem_u32(sm.stage[s]), 16, 512, tc::SW_64B);
        tc::mma_mxf4(d, adesc, bdesc, id0, sfa, tmem + C::SFB_COL, 0);
        tc::mma_mxf4(d, adesc + 2, bdesc + 2, id1, sfa, tmem + C::SFB_COL, 1);   // next 32 bytes of K
        tc::commit(&sm.empty[s]);
        tc::commit(&sm.acc_full[k]);
      }
      // after an abort the epilogue may stop reading: the MMAs already issued
      // must finish before the accumulators' TMEM is released
      if (sm.abort_flag && use > 0) tc::bar_wait(&sm.acc_full[k], (uint32_t)(use - 1) & 1u, 1u << 20);
    }
    __syncwarp();
  } else if (warp == C::PUB_WARP) {
    // ================= publisher: TMA completions -> ready words for the issuers
    if (!pool_mode && lane == 0) {
      for (int i = 0; i < n; i++) {
        if (!wait_or_abort(&sm.full[i % IS_STAGES], (i / IS_STAGES) & 1, sm, p.hdr)) break;
        publish_word(&sm.ready[i % IS_STAGES], (uint32_t)(i + 1));
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue: warp (lane quarter q, query jq); lane r of
    // quarter q holds tile row 32q + r = slot 4r + q of the tile
    const int q = warp & 3;
    const int jq = (warp - C::EPI0) >> 2;
    const int slot = 4 * lane + q;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int64_t nv_mine = nvq[0];
#pragma unroll
    for (int j = 1; j < NQ; j++)
      if (jq == j) nv_mine = nvq[j];
    float* out_row = p.scores + (pool_mode ? bq0 * p.M * BLK : (bq0 + jq) * p.max_n);
    unsigned long long w2[HI / 2];
    pack_head_weights(sm.w + jq * HI, w2);
    for (int j = 0; j < n; j++) {
      const int k = j % C::ISSUERS;
      const bool ok_tile = __all_sync(0xFFFFFFFFu, wait_or_abort(&sm.acc_full[k], (j / C::ISSUERS) & 1, sm, p.hdr));
      if (!ok_tile) break;                                        // (the warp leaves together)
      tc::fence_after_sync();
      float v[32];
      tc::tmem_ld_x32(tmem + lane_off + C::ACC_COL + k * C::N + jq * HI, v);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0)
        asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" :: "r"(tc::smem_u32(&sm.acc_free[k])) : "memory");
      const float sc = index_head_sum(v, w2);
      const int64_t u = (t0 + j) * IS_TILE + slot;
      if (!pool_mode) {
        if (u < nv_mine && jq < nq) out_row[u] = sc;
      } else {
        bool ok = false;
        if (u < n_units) {
          const int32_t blk = sm.pool[u / BLK];
          const int64_t e = (int64_t)blk * BLK + (u % BLK);
          if (blk >= 0) {
            if ((int64_t)blk * BLK >= p.cap) {
              if ((u % BLK) == 0) report(p.hdr, CSA2_ERR_BOUNDS, blk);
            } else if (e < nv) {
              ok = true;
            }
          }
        }
        if (u < n_units) out_row[u] = ok ? sc : -INFINITY;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
// Index-code rows [rows][64 B] seen as [rows/4 groups g][4 members q][64 B], so
// that one box of 32 groups x 4 members lands member-major: shared row 32q + g
// holds entry 4g + q of the tile (the row order the scale-word copy needs), in
// the SW64 layout.
static bool encode_tile_rows(CUtensorMap* map, const void* base, uint64_t rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows / 4, 4};
  cuuint64_t strides[2] = {4 * 64, 64};
  cuuint32_t box[3] = {64, IS_TILE / 4, 4};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static cudaError_t set_is_attrs() {
  static_assert(IsCfg<1>::MIN_CTAS * (is_smem_bytes<1>() + 1024) <= 228 * 1024, "resident CTAs");
  static PerDeviceOnce attrs;
  return attrs.ensure([](int) {
    cudaError_t e = cudaSuccess;
    for (auto k : {index_score_tc_kernel<1, false>, index_score_tc_kernel<1, true>}) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)is_smem_bytes<1>());
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    }
    for (auto k : {index_score_tc_kernel<IS_GROUP, false>, index_score_tc_kernel<IS_GROUP, true>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)is_smem_bytes<IS_GROUP>());
    return e;
  });
}

// test hook of the calling host thread (csa2_test_withhold_arrival)
static thread_local bool g_test_withhold = false;
static void set_test_withhold(bool on) { g_test_withhold = on; }

cudaError_t launch_index_score(IsParams p, cudaStream_t stream) {
  if (p.B == 0 || p.Q == 0) return cudaSuccess;
  p.test_withhold = g_test_withhold ? 1 : 0;
  cudaError_t ae = set_is_attrs();
  if (ae != cudaSuccess) return ae;
  int num_sms = 0;
  if ((ae = device_sms(&num_sms)) != cudaSuccess) return ae;
  const uint64_t rows = (uint64_t)p.B * (uint64_t)p.cap;
  if (rows == 0) return cudaSuccess;
  CUtensorMap map_tile;
  if (!encode_tile_rows(&map_tile, p.idx_codes, rows)) return cudaErrorInvalidValue;
  const int64_t units = p.pool ? (int64_t)p.M * BLK : p.max_n;
  const int64_t tiles = ceil_div(units, IS_TILE);
  if (tiles == 0) return cudaSuccess;
  // many queries per sequence (and no pool): groups of IS_GROUP queries share each key tile
  const bool grouped = p.pool == nullptr && p.Q >= IS_GROUP;
  const int nq = grouped ? IS_GROUP : 1;
  const int64_t groups = (int64_t)p.B * ceil_div(p.Q, nq);
  // one wave: as many CTAs as are resident at once (the launch bounds and the
  // shared-memory carveout guarantee MIN_CTAS per SM), at least 2 tiles per CTA
  const int64_t resident = (int64_t)(grouped ? IsCfg<IS_GROUP>::MIN_CTAS : IsCfg<1>::MIN_CTAS) * num_sms;
  int64_t split = resident / groups;
  if (split > ceil_div(tiles, 2)) split = ceil_div(tiles, 2);
  if (split < 1) split = 1;
  const int64_t per = ceil_div(tiles, split);
  p.entries_per_cta = per;     // tiles per CTA
  const int64_t split_ctas = ceil_div(tiles, per);
  if (split_ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
  // at most 65535 query groups per launch (the grid's y limit); the launches of
  // one call are independent (disjoint queries, shared read-only inputs)
  for (int64_t g0 = 0; g0 < groups; g0 += 65535) {
    p.group0 = g0;
    const dim3 grid((unsigned)split_ctas, (unsigned)(groups - g0 < 65535 ? groups - g0 : 65535));
    const bool offset = groups > 65535;
    if (grouped && offset)
      index_score_tc_kernel<IS_GROUP, true><<<grid, IsCfg<IS_GROUP>::THREADS, is_smem_bytes<IS_GROUP>(), stream>>>(
          p, map_tile);
    else if (grouped)
      index_score_tc_kernel<IS_GROUP, false><<<grid, IsCfg<IS_GROUP>::THREADS, is_smem_bytes<IS_GROUP>(), stream>>>(
          p, map_tile);
    else if (offset)
      index_score_tc_kernel<1, true><<<grid, IsCfg<1>::THREADS, is_smem_bytes<1>(), stream>>>(p, map_tile);
    else
      index_score_tc_kernel<1, false><<<grid, IsCfg<1>::THREADS, is_smem_bytes<1>(), stream>>>(p, map_tile);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa2

extern "C" csa2_status csa2_test_withhold_arrival(int enable) {
  if (enable != 0 && enable != 1) return CSA2_ERR_INVALID_ARG;
  csa2::set_test_withhold(enable != 0);
  return CSA2_OK;
}
