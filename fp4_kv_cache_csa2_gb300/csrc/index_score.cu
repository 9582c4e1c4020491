// (b) Lightning-indexer scores  s(t,j) = sum_h w_h * ReLU(q_h . k_j)
// over 32 index heads x 128 dims, with MXFP4 queries and keys, on the
// 5th-generation tensor cores (tcgen05, kind::mxf4 block-scaled MMA).
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4 (the Full layer
// scores every causally visible main-KV position; Reindex layers score only the
// candidate pool), §2.4.4 (FP4 indexer Q and K); "4. 层维度(下):CSA2 与每 token
// 890 字节" §4.4 (index K is OCP MXFP4: E2M1 + one E8M0 scale per 32), §4.7.
//
// One CTA scores a run of 128-entry tiles of one query:
//   warp 0      producer: full scans load 128-entry tiles of index-K codes
//               (SW64 K-major, 64 B per entry) with a 2-D tensor map and the
//               4-byte E8M0 words with 1-D bulk copies (mbarrier expect-tx); pool
//               scans gather the 16 candidate blocks of a tile with cp.async,
//               one 512-byte block per warp instruction, into the same layout.
//               6-stage ring.
//   warp 1      TMEM owner and MMA issuer: per tile two M=128 N=32 K=64
//               block-scaled MMAs into one of two TMEM accumulators.
//   warps 2..5  per tile: copy the 128 scale words into TMEM (row m -> lane m,
//               column base + m/32), then the epilogue of the previous tile:
//               32 head dot products from TMEM -> ReLU -> weighted sum -> score.
// The query is quantised once per CTA (the B operand, 2 KB, and its scales).
// Products of E2M1 values scaled by powers of two are exact; the accumulation
// is fp32.  Every mbarrier wait is bounded and reports CSA2_ERR_TIMEOUT.
#include <cstddef>
#include <cudaTypedefs.h>

#include "index_query.cuh"
#include "params.cuh"
#include "tc.cuh"


namespace csa2 {

constexpr int IS_THREADS = 192;
constexpr int IS_STAGES = 6;
constexpr int IS_TILE = 128;
constexpr int IS_CODES = IS_TILE * IDX_CODE_BYTES;         // 8192
constexpr int IS_STAGE_BYTES = IS_CODES + 1024;            // codes + 512 B scales, 1 KB aligned stride
constexpr int IS_POOL_MAX = CSA2_MAX_M;
constexpr int IS_TMEM_COLS = 128;
constexpr int IS_ACC_COL = 0;                               // two accumulators of 32 columns
constexpr int IS_SFA_COL = 64;                              // 4 columns per stage
constexpr int IS_SFB_COL = 96;

struct IsSmem {
  uint8_t stage[IS_STAGES][IS_STAGE_BYTES];
  uint8_t qcodes[HI * IDX_CODE_BYTES];      // 2 KB, SW64
  int32_t pool[IS_POOL_MAX];
  float w[HI];
  uint32_t sfb[HI];                          // query scale words (head n -> lane n of every quarter)
  uint64_t full[IS_STAGES], empty[IS_STAGES], sf_full[IS_STAGES];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  volatile int abort_flag;
};
constexpr size_t IS_SMEM = sizeof(IsSmem) + 1024;

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, IsSmem& sm, WsHeader* hdr) {
  if (sm.abort_flag) return false;
  for (int round = 0; round < 64; round++) {
    if (tc::bar_wait(bar, parity, 1u << 16)) return true;
    if (sm.abort_flag) return false;
  }
  sm.abort_flag = 1;
  report(hdr, CSA2_ERR_TIMEOUT, 1);
  return false;
}

__global__ void __launch_bounds__(IS_THREADS, 1)
index_score_tc_kernel(IsParams p, const __grid_constant__ CUtensorMap map_tile,
                      const __grid_constant__ CUtensorMap map_block) {
  extern __shared__ unsigned char smem_raw[];
  IsSmem& sm = *reinterpret_cast<IsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bq = (int)blockIdx.y;
  const int crank = (int)blockIdx.x;         // slice of the query
  const int b = bq / p.Q;
  const bool pool_mode = p.pool != nullptr;

  // ---- this CTA's tile range
  int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[b]);
  if (nv > p.cap) {
    if (tid == 0 && blockIdx.x == 0) report(p.hdr, CSA2_ERR_BOUNDS, nv);
    nv = p.cap;
  }
  int64_t n_units;                         // entries (full) or pool slots (pool)
  if (pool_mode) {
    n_units = (int64_t)p.M * BLK;
  } else {
    if (nv > p.max_n) {
      if (tid == 0 && blockIdx.x == 0) report(p.hdr, CSA2_ERR_BOUNDS, nv);
      nv = p.max_n;
    }
    n_units = nv;
  }
  const int64_t n_tiles = ceil_div(n_units, IS_TILE);
  const int64_t t0 = (int64_t)crank * p.entries_per_cta;
  int64_t t1 = t0 + p.entries_per_cta;
  if (t1 > n_tiles) t1 = n_tiles;
  const int n = (int)(t1 > t0 ? t1 - t0 : 0);
  if (n == 0) return;

  // ---- set-up
  if (warp == 1) tc::tmem_alloc(&sm.tmem_base, IS_TMEM_COLS);
  if (tid == 0) {
    for (int s = 0; s < IS_STAGES; s++) {
      tc::bar_init(&sm.full[s], pool_mode ? 32 : 1);
      tc::bar_init(&sm.empty[s], 1);
      tc::bar_init(&sm.sf_full[s], 4);
    }
    for (int i = 0; i < 2; i++) {
      tc::bar_init(&sm.acc_full[i], 1);
      tc::bar_init(&sm.acc_empty[i], 4);
    }
    sm.abort_flag = 0;
    tc::bar_init_fence();
  }
  if (tid < HI) sm.w[tid] = p.w_head[(int64_t)bq * HI + tid];
  if (pool_mode) {
    const int32_t* pool = p.pool + (int64_t)bq * p.M;
    for (int i = tid; i < p.M; i += IS_THREADS) sm.pool[i] = pool[i];
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensormap(&map_tile);
    tc::prefetch_tensormap(&map_block);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  // ---- quantise the query (B operand); its scale words go to TMEM lanes
  // 32q + n of every lane quarter q (the MMA reads B scales from the quarter of
  // the A row it is computing)
  if (warp == 4) quantize_index_query_warp(p.q_idx + (int64_t)bq * HI * DI, sm.qcodes, sm.sfb);
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (warp >= 2) {
    tc::tmem_st_x1(tmem + ((uint32_t)((warp & 3) * 32) << 16) + IS_SFB_COL, sm.sfb[lane]);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  const int64_t row_base = (int64_t)b * p.cap;
  const int64_t rows_total = (int64_t)p.B * p.cap;

  if (warp == 0) {
    // ================= TMA producer
    int issued = 0;
    for (int i = 0; i < n; i++) {
      const int s = i % IS_STAGES;
      if (i >= IS_STAGES && !wait_or_abort(&sm.empty[s], ((i / IS_STAGES) - 1) & 1, sm, p.hdr)) break;
      uint8_t* codes = sm.stage[s];
      uint8_t* scl = sm.stage[s] + IS_CODES;
      const int64_t t = t0 + i;
      if (!pool_mode) {
        if (lane == 0) {
          const int64_t row0 = row_base + t * IS_TILE;
          int64_t rows = rows_total - row0;
          if (rows > IS_TILE) rows = IS_TILE;
          const uint32_t sbytes = (uint32_t)rows * IDX_SCALE_BYTES;     // cap % 8 == 0 -> multiple of 16
          tc::bar_arrive_expect_tx(&sm.full[s], IS_CODES + sbytes);
          tc::tma_load_2d(codes, &map_tile, 0, (int32_t)row0, &sm.full[s]);
          tc::bulk_load(scl, p.idx_scales + row0 * IDX_SCALE_BYTES, sbytes, &sm.full[s]);
        }
      } else {
        // 16 candidate blocks of 8 entries.  One warp instruction copies one whole
        // block (512 contiguous code bytes, 16 per lane: entry l/4, 16-byte chunk
        // l%4) into the SW64 layout, so each instruction touches 4 cache lines;
        // lanes 2b and 2b+1 then copy block b's 32 bytes of scale words.  Each
        // lane's arrival fires once its own copies have landed.
        const int64_t pl = t * 16 + (lane & 15);
        int32_t my_blk = (pl < p.M) ? sm.pool[pl] : -1;
        if (my_blk >= 0 && (int64_t)my_blk * BLK >= p.cap) my_blk = -1;   // reported by the epilogue
        const int r = lane >> 2, c = lane & 3;
#pragma unroll 4
        for (int sb = 0; sb < 16; sb++) {
          const int32_t blk = __shfl_sync(0xFFFFFFFFu, my_blk, sb);
          if (blk < 0) continue;
          const int trow = sb * BLK + r;
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
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(tc::smem_u32(&sm.full[s])) : "memory");
      }
      issued = i + 1;
    }
    if (sm.abort_flag && lane == 0) {
      // drain copies still in flight before the CTA exits
      for (int i = issued - 1; i >= 0 && i >= issued - IS_STAGES; i--)
        tc::bar_wait(&sm.full[i % IS_STAGES], (i / IS_STAGES) & 1, 1u << 20);
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      const uint64_t bdesc = tc::smem_desc(tc::smem_u32(sm.qcodes), 16, 512, tc::SW_64B);
      constexpr uint32_t id0 = tc::idesc_mxf4(IS_TILE, HI, 0, 0);
      constexpr uint32_t id1 = tc::idesc_mxf4(IS_TILE, HI, 2, 2);
      for (int i = 0; i < n; i++) {
        const int s = i % IS_STAGES, buf = i & 1;
        if (!wait_or_abort(&sm.sf_full[s], (i / IS_STAGES) & 1, sm, p.hdr)) break;
        if (i >= 2 && !wait_or_abort(&sm.acc_empty[buf], ((i >> 1) - 1) & 1, sm, p.hdr)) break;
        tc::fence_after_sync();
        const uint64_t adesc = tc::smem_desc(tc::smem_u32(sm.stage[s]), 16, 512, tc::SW_64B);
        const uint32_t d = tmem + IS_ACC_COL + buf * 32;
        const uint32_t sfa = tmem + IS_SFA_COL + s * 4;
        tc::mma_mxf4(d, adesc, bdesc, id0, sfa, tmem + IS_SFB_COL, 0);
        tc::mma_mxf4(d, adesc + 2, bdesc + 2, id1, sfa, tmem + IS_SFB_COL, 1);   // next 32 bytes of K
        tc::commit(&sm.empty[s]);
        tc::commit(&sm.acc_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // ================= scale copy into TMEM + epilogue (warps 2..5)
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    const int m = q * 32 + lane;              // tile row owned by this thread
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float* out_row = p.scores + (pool_mode ? (int64_t)bq * p.M * BLK : (int64_t)bq * p.max_n);
    for (int i = 0; i <= n; i++) {
      if (i < n) {
        const int s = i % IS_STAGES;
        if (!wait_or_abort(&sm.full[s], (i / IS_STAGES) & 1, sm, p.hdr)) break;
        const uint32_t word = *reinterpret_cast<const uint32_t*>(sm.stage[s] + IS_CODES + m * 4);
        tc::tmem_st_x1(tmem + lane_off + IS_SFA_COL + s * 4 + q, word);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::bar_arrive(&sm.sf_full[s]);
      }
      if (i >= 1) {
        const int j = i - 1, buf = j & 1;
        if (!wait_or_abort(&sm.acc_full[buf], (j >> 1) & 1, sm, p.hdr)) break;
        tc::fence_after_sync();
        float v[32];
        tc::tmem_ld_x32(tmem + lane_off + IS_ACC_COL + buf * 32, v);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::bar_arrive(&sm.acc_empty[buf]);
        float sc = 0.0f;
#pragma unroll
        for (int h = 0; h < HI; h++) sc = fmaf(sm.w[h], fmaxf(v[h], 0.0f), sc);
        const int64_t u = (t0 + j) * IS_TILE + m;
        if (!pool_mode) {
          if (u < n_units) out_row[u] = sc;
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
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, IS_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D byte tensor [rows][64] with SW64 boxes of `box_rows` rows.
static bool encode_rows64(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static cudaError_t set_is_attrs() {
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(index_score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)IS_SMEM);
  if (e == cudaSuccess) attr_dev = dev;
  return e;
}

cudaError_t launch_index_score(IsParams p, cudaStream_t stream) {
  if (p.B == 0 || p.Q == 0) return cudaSuccess;
  cudaError_t ae = set_is_attrs();
  if (ae != cudaSuccess) return ae;
  int dev = 0;
  cudaGetDevice(&dev);
  int num_sms = 148;
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  const uint64_t rows = (uint64_t)p.B * (uint64_t)p.cap;
  if (rows == 0) return cudaSuccess;
  CUtensorMap map_tile, map_block;
  if (!encode_rows64(&map_tile, p.idx_codes, rows, IS_TILE) || !encode_rows64(&map_block, p.idx_codes, rows, BLK))
    return cudaErrorInvalidValue;
  const int64_t units = p.pool ? (int64_t)p.M * BLK : p.max_n;
  const int64_t tiles = ceil_div(units, IS_TILE);
  if (tiles == 0) return cudaSuccess;
  const int64_t BQ = (int64_t)p.B * p.Q;
  // aim at ~3 CTAs per SM over the whole launch, at least 2 tiles per CTA
  int64_t split = ceil_div(3 * (int64_t)num_sms, BQ);
  if (split > ceil_div(tiles, 2)) split = ceil_div(tiles, 2);
  if (split < 1) split = 1;
  const int64_t per = ceil_div(tiles, split);
  p.entries_per_cta = per;     // tiles per CTA
  dim3 grid((unsigned)ceil_div(tiles, per), (unsigned)BQ);
  index_score_tc_kernel<<<grid, IS_THREADS, IS_SMEM, stream>>>(p, map_tile, map_block);
  return cudaGetLastError();
}

// Reindex: score the pool of every query and publish its top-K in one launch.
}  // namespace csa2
