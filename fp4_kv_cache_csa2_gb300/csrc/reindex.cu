// (b) Fused Reindex layer: the lightning-indexer scores of the candidate pool
// and the exact top-K over them, in one kernel with one CTA per query token.
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4 (a Reindex layer
// scores only the entries of the candidate blocks its source layer chose and
// keeps its own top-512), §2.4.4 (FP4 indexer Q and K); "4. 层维度(下):CSA2 与
// 每 token 890 字节" §4.4 (index K is OCP MXFP4), §4.7 (hierarchical sparse
// indexing).
//
// One CTA (256 threads, one per SM) takes one query and scores its whole pool
// (up to 2048 blocks = 128 tiles of 128 slots) in bulk-synchronous rounds of
// RX_ROUND tiles, with no per-tile hand-offs.  Tiles and TMEM accumulators are
// double-buffered, so that one CTA barrier per round separates three stages of
// three consecutive rounds:
//   1. warps 0..6 copy the next round's tiles, one tile each (one 512-byte block
//      of index codes per warp instruction, into the SW64 K-major layout, plus
//      the blocks' scale words) with cp.async;
//   2. meanwhile one thread of warp 7 issues this round's block-scaled MMAs
//      (M = 128 entries, N = 32 heads, K = 128 as two K = 64 halves; the tile's
//      E8M0 words go to TMEM by tcgen05.cp just before), one accumulator per tile;
//   3. then all warps read the previous round's accumulators back (lane = entry,
//      column = head) and form s = sum_h w_h ReLU(q_h . k), kept as an
//      order-preserving key per pool slot (0 for slots outside the search
//      domain).
// The query is quantised to MXFP4 and its scale words stored in TMEM once.
// Then one exact radix select over all slot keys in shared memory takes the
// top K by (score desc, slot asc) and writes the entries in slot order.
// Products of E2M1 values scaled by powers of two are exact; the accumulation
// is fp32.  Ties go to the lower pool slot (= lower entry for an ascending
// pool).  The MMA wait is bounded and reports CSA2_ERR_TIMEOUT.
//
// The query is quantised by warp 7 while warps 0..6 issue round 0's copies.
//
// (A cluster of six CTAs per query, each scoring a sixth of the pool and
// exchanging digit histograms for the select, decoded 2.42M query-token-layers
// per second at 1M entries and batch 16, against 2.63M with the first version
// of this one-CTA kernel and 3.36M with the current one: a cluster holds its
// six SMs for its slowest member's whole run, and the select's exchange rounds
// were most of that run.)
#include <cstddef>

#include "index_query.cuh"
#include "host_once.cuh"
#include "params.cuh"
#include "tc.cuh"

namespace csa2 {

constexpr int RX_THREADS = 256;
constexpr int RX_WARPS = RX_THREADS / 32;
constexpr int RX_TILE = 128;                                    // pool slots per tile
constexpr int RX_SLOTS = CSA2_MAX_M * BLK;                      // 16,384
constexpr int RX_ROUND = 7;                                     // tiles (and TMEM accumulators) per round
constexpr int RX_BUFS = 2;                                      // rounds whose tiles / accumulators are live
constexpr int RX_CODES = RX_TILE * IDX_CODE_BYTES;              // 8192
constexpr int RX_TILE_BYTES = RX_CODES + 512;                   // codes + 512 B scale words (SW64 atoms: 512 B aligned)
constexpr int RX_TMEM_COLS = 512;
constexpr int RX_ACC_COL = 0;                                   // tile j of buffer b: 32 columns at 32 (RX_ROUND b + j)
constexpr int RX_SFA_COL = RX_BUFS * RX_ROUND * HI;             // its scale words: 4 columns at RX_SFA_COL + 4 (RX_ROUND b + j)
constexpr int RX_SFB_COL = RX_SFA_COL + 4 * RX_BUFS * RX_ROUND;
static_assert(RX_SFB_COL + 4 <= RX_TMEM_COLS, "TMEM columns");

struct RxSmem {
  uint8_t tile[RX_BUFS][RX_ROUND][RX_TILE_BYTES];   // SW64 codes, then 128 scale words
  uint8_t qcodes[HI * IDX_CODE_BYTES];          // 2 KB, SW64
  int32_t pool[CSA2_MAX_M];                     // the query's blocks (-1: none)
  float w[HI];
  uint32_t sfb[HI];
  alignas(16) uint32_t keys[RX_SLOTS / 64 * 68];   // slot keys, rows of 64 (+ 4 pad words); 0 = outside the search domain
  alignas(16) uint32_t hist[4096];              // digit histogram of the current select pass
  int32_t wsum[RX_WARPS];
  uint32_t wmax[RX_WARPS];
  int32_t bcast[4];
  uint64_t mma_done[RX_BUFS];
  uint32_t tmem_base;
};
constexpr size_t RX_SMEM = sizeof(RxSmem) + 1024;

// Shared-memory index of slot u's key: rows of 64 keys padded to 68 words, so
// that the select's threads, which own one row each and read it as 16-byte
// vectors, hit distinct banks in every quarter-warp phase.
constexpr int RX_KROW = 68;
__device__ __forceinline__ int key_index(int u) { return (u >> 6) * RX_KROW + (u & 63); }
static_assert(RX_SMEM <= 227 * 1024, "shared memory");

// 16-byte shared-memory load at a shared-window address (kept in order with
// the surrounding shared-memory atomics).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}

// Exclusive prefix sum over the CTA (RX_THREADS threads); *total receives the sum.
template <class Sm>
__device__ int cta_exclusive_scan(int v, Sm& fs, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) fs.wsum[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < RX_WARPS; w++) {
    const int ws = fs.wsum[w];
    base += (w < warp) ? ws : 0;
    tot += ws;
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

// Top-K of n keys (n a multiple of 64; key 0 = not a candidate; key of index i
// at keys[key_index(i)]) by (key desc, index asc), within the CTA: exact radix
// select.
//   * Every thread brings the largest and the second largest of the keys it
//     formed (first, second).  Those 2 x 256 >= K distinct keys are all at
//     least the smallest second, lo, so no key below lo can be among the top K:
//     the candidates are the keys >= lo (all nonzero keys when a thread formed
//     fewer than two), typically a small fraction.
//   * The select runs on kp = key - lo, which orders the candidates as the keys
//     do, over digits of kp: the first 12 bits just below the span of the
//     candidates (max key - lo), so that they spread over all 4096 bins (few
//     share one, few shared-memory atomics collide, and the threshold bin
//     usually holds just the keys still to take), then 8 bits at a time.
//   * Each pass builds the shared histogram of the digit over the candidates
//     that match the digits chosen so far; a scan of the bins from the top (each
//     thread sums a run of bins) gives the threshold digit and the number of
//     ties still to take; a threshold bin taken whole ends the passes early.
//   * Thread t owns keys 64 t .. 64 t + 63.  The first pass walks them two
//     16-byte vectors at a time in a short rolled loop and records the
//     candidates among them as a bit mask; the later passes and the final
//     walk visit only the candidates, and the final walk records its keys
//     above and at the threshold as bit masks, so the output visits the
//     chosen keys only.
// out(i, r) is called for the chosen keys in index order (r = 0, 1, ...); the
// function returns their number.
template <class Sm, class Out>
__device__ int cta_select(const uint32_t* keys, int n, int K, uint32_t first, uint32_t second, Sm& fs, Out out) {
  static_assert(RX_THREADS == 256 && 2 * RX_THREADS >= CSA2_MAX_K, "bin runs per thread; the candidate floor");
  if (K <= 0) return 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool mine = 64 * tid < n;
  // row t: 64 keys (16 vectors of 16 bytes) and 4 pad words
  const uint32_t row = tc::smem_u32(keys + tid * RX_KROW);
  const uint32_t hist_base = tc::smem_u32(fs.hist);
  {
    const uint32_t wlo = __reduce_min_sync(0xFFFFFFFFu, second), whi = __reduce_max_sync(0xFFFFFFFFu, first);
    if (lane == 0) {
      fs.wsum[warp] = (int)wlo;
      fs.wmax[warp] = whi;
    }
  }
  __syncthreads();
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
  for (int w = 0; w < RX_WARPS; w++) {
    lo = min(lo, (uint32_t)fs.wsum[w]);
    hi = max(hi, fs.wmax[w]);
  }
  lo = max(lo, 1u);                                        // key 0 is never a candidate
  const uint32_t span = hi >= lo ? hi - lo : 0u;           // every candidate's kp is at most span
  const int span_bits = span ? 32 - __clz(span) : 0;
  uint32_t prefix = 0, mask = 0;                           // digits of kp fixed so far
  uint64_t cand = 0;                                       // this thread's candidates (set by the first pass)
  int remaining = K;
  bool take_all = false;                                   // at most K candidates
  int shift = max(0, span_bits - 12), width = 12;
#pragma unroll 1
  for (int pass = 0;; pass++) {
    const int nbins = 1 << width;
    const uint32_t dmask = (uint32_t)nbins - 1u;
    for (int b = tid; b < nbins; b += RX_THREADS) fs.hist[b] = 0;
    __syncthreads();
    if (mine && pass == 0) {                               // every key: the candidates, their first digit
      uint4 nx0 = lds128(row), nx1 = lds128(row + 16u);
#pragma unroll 1
      for (int v = 0; v < 16; v += 2) {                    // two vectors (eight keys) per iteration
        const uint4 q0 = nx0, q1 = nx1;
        if (v + 2 < 16) {                                  // the next pair
          nx0 = lds128(row + 16u * (v + 2));
          nx1 = lds128(row + 16u * (v + 3));
        }
        const uint32_t kk[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint32_t nib = 0;
#pragma unroll
        for (int e = 0; e < 8; e++) {
          if (kk[e] >= lo) {
            nib |= 1u << e;
            asm volatile("red.shared.add.u32 [%0], 1;" :: "r"(hist_base + 4u * (((kk[e] - lo) >> shift) & dmask)));
          }
        }
        cand |= (uint64_t)nib << (4 * v);
      }
    } else if (mine) {                                     // the candidates only
#pragma unroll 1
      for (uint64_t cm = cand; cm != 0ull; cm &= cm - 1ull) {
        const int bit = __ffsll((long long)cm) - 1;
        const uint32_t kp = lds32(row + 4u * bit) - lo;
        if ((kp & mask) == prefix)
          asm volatile("red.shared.add.u32 [%0], 1;" :: "r"(hist_base + 4u * ((kp >> shift) & dmask)));
      }
    }
    __syncthreads();
    // thread t sums the run of bpt bins below nbins - bpt t (larger digits go to
    // lower threads), each lane starting at its own bin of the run (no two lanes
    // of a warp on one bank)
    const int bpt = nbins >= RX_THREADS ? nbins / RX_THREADS : 1;
    const int top = nbins - bpt * tid;                     // bins [top - bpt, top) when top > 0
    int c = 0;
    if (top > 0)
      for (int q = 0; q < bpt; q++) c += (int)fs.hist[top - 1 - ((q + lane) & (bpt - 1))];
    int tot;
    const int above = cta_exclusive_scan(c, fs, &tot);     // keys with a larger digit than this run
    if (pass == 0 && tot <= remaining) {
      if (tid == 0) fs.bcast[0] = -1;                      // at most K candidates: take them all
    } else if (above < remaining && above + c >= remaining) {
      int run = above, d = top - 1;                        // walk the run from its largest digit
      for (;; d--) {
        const int h = (int)fs.hist[d];
        if (run + h >= remaining) {
          fs.bcast[0] = d;                                 // the digit of the K-th largest key
          fs.bcast[1] = remaining - run;
          fs.bcast[2] = h;
          break;
        }
        run += h;
      }
    }
    __syncthreads();
    const int d = fs.bcast[0];
    if (d < 0) {
      take_all = true;
      remaining = 0;
      break;
    }
    // the rest of the threshold bin is taken whole: the keys' remaining bits
    // need not be looked at
    const bool whole = fs.bcast[2] == fs.bcast[1];
    prefix |= (uint32_t)d << shift;
    // every bit at and above the digit is fixed now (those above the first
    // digit are zero for every candidate)
    mask = ~((1u << shift) - 1u);
    remaining = fs.bcast[1];
    __syncthreads();                                       // bcast and hist read before the next pass writes them
    if (whole || shift == 0) break;
    width = min(8, shift);
    shift -= width;
  }
  const uint32_t thr = prefix;
  const int take_eq = remaining;                           // keys equal to thr still to take, in index order
  uint64_t gtm = 0, eqm = 0;                               // this thread's keys above / at the threshold
  if (take_all) {
    gtm = cand;
  } else {
#pragma unroll 1
    for (uint64_t cm = cand; cm != 0ull; cm &= cm - 1ull) {
      const int bit = __ffsll((long long)cm) - 1;
      const uint32_t km = (lds32(row + 4u * bit) - lo) & mask;   // digits fixed so far
      if (km > thr) gtm |= 1ull << bit;
      else if (km == thr) eqm |= 1ull << bit;
    }
  }
  const int gt = __popcll(gtm), eq = __popcll(eqm);
  // one scan of (gt, eq) packed in 16-bit halves (fewer than 2^16 keys)
  int both_tot;
  const int both_before = cta_exclusive_scan((gt << 16) | eq, fs, &both_tot);
  const int gt_before = both_before >> 16, eq_before = both_before & 0xFFFF;
  const int mine_eq = max(0, min(eq, take_eq - eq_before));
  uint64_t take = gtm;
  for (int q = 0; q < mine_eq; q++) {                      // the first mine_eq ties, in index order
    const uint64_t low = eqm & (~eqm + 1ull);
    take |= low;
    eqm ^= low;
  }
  int r = gt_before + min(eq_before, take_eq);
  while (take != 0ull) {
    const int bit = __ffsll((long long)take) - 1;
    take &= take - 1ull;
    out(64 * tid + bit, r++);
  }
  return (both_tot >> 16) + min(both_tot & 0xFFFF, take_eq);
}

__global__ void __launch_bounds__(RX_THREADS, 1) reindex_select_kernel(IsParams p) {
  extern __shared__ unsigned char smem_raw[];
  RxSmem& sm = *reinterpret_cast<RxSmem*>(tc::align_smem_1k(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bq = (int)blockIdx.x;
  const int b = bq / p.Q;

  // ---- set-up: TMEM, barrier, head weights, the pool, the query
  if (warp == 0) tc::tmem_alloc(&sm.tmem_base, RX_TMEM_COLS);
  if (tid == 0) {
    for (int b = 0; b < RX_BUFS; b++) tc::bar_init(&sm.mma_done[b], 1);
    tc::bar_init_fence();
  }
  // everything above reads no input: with programmatic dependent launch it
  // overlaps the previous kernel, which may have produced the pool or the queries
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[b]);
  if (nv > p.cap) {
    if (tid == 0) report(p.hdr, CSA2_ERR_BOUNDS, nv);
    nv = p.cap;
  }
  const int n_slots = p.M * BLK;
  const int n_tiles = (n_slots + RX_TILE - 1) / RX_TILE;
  const int64_t row_base = (int64_t)b * p.cap;
  if (tid < HI) sm.w[tid] = p.w_head[(int64_t)bq * HI + tid];
  for (int i = tid; i < n_tiles * 16; i += RX_THREADS) {
    int32_t blk = i < p.M ? p.pool[(int64_t)bq * p.M + i] : -1;
    if (blk >= 0 && (int64_t)blk * BLK >= p.cap) {
      report(p.hdr, CSA2_ERR_BOUNDS, blk);
      blk = -1;
    }
    sm.pool[i] = blk;
  }
  __syncthreads();                                              // the pool, for round 0's copies
  // ---- 1. copies of the round of tiles r0 .. into buffer b: warp w < 7 takes
  // tile w; one warp instruction per block
  auto issue_copies = [&](int r0, int b) {
    const int rn = min(RX_ROUND, n_tiles - r0);
    static_assert(RX_ROUND <= RX_WARPS - 1, "one tile per copying warp");
    if (warp < rn) {
      uint8_t* codes = sm.tile[b][warp];
      const int32_t my_blk = sm.pool[(r0 + warp) * 16 + (lane & 15)];
      const int r = lane >> 2, c = lane & 3;                    // entry of the block, 16-byte chunk
#pragma unroll 4
      for (int sb = 0; sb < 16; sb++) {
        const int32_t blk = __shfl_sync(0xFFFFFFFFu, my_blk, sb);
        if (blk < 0) continue;
        const int trow = sb * BLK + r;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                     :: "r"(tc::smem_u32(codes + trow * 64 + ((c ^ ((trow >> 1) & 3)) * 16))),
                        "l"(p.idx_codes + (row_base + (int64_t)blk * BLK) * IDX_CODE_BYTES + lane * 16) : "memory");
      }
      // scale words, 4 blocks per instruction: the word of slot s lands in row
      // s % 32, word s / 32 of the tile's 512-byte scale area, the order in which
      // a 32x128b.warpx4 copy hands row m's word to TMEM lane m, column base + m / 32
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const int sb = 4 * q + (lane >> 3), r = lane & 7, slot = sb * BLK + r;
        const int32_t blk = __shfl_sync(0xFFFFFFFFu, my_blk, sb);
        if (blk >= 0)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                       :: "r"(tc::smem_u32(codes + RX_CODES + (slot & 31) * 16 + (slot >> 5) * 4)),
                          "l"(p.idx_scales + (row_base + (int64_t)blk * BLK + r) * IDX_SCALE_BYTES) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // round 0's copies fly while warp 7 quantises the query
  issue_copies(0, 0);
  if (warp == RX_WARPS - 1) quantize_index_query_warp_loads_first(p.q_idx + (int64_t)bq * HI * DI, sm.qcodes, sm.sfb);
  tc::fence_proxy_async_smem();                                 // the query codes feed the tensor cores
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  // the query's scale words to TMEM lane 32 q + head of every quarter q
  if (warp < 4) {
    tc::tmem_st_x1(tmem + ((uint32_t)(warp * 32) << 16) + RX_SFB_COL, sm.sfb[lane]);
    tc::tmem_wait_st();
  }

  const int q4 = warp & 3;                                      // TMEM lane quarter of this warp
  const int m = q4 * 32 + lane;                                 // tile row = slot within the tile
  const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
  unsigned long long w2[HI / 2];
  pack_head_weights(sm.w, w2);
  bool ok_all = true;
  uint32_t first = 0u, second = 0u;
  // ---- 3. keys of the round of tiles r0 .. from accumulator buffer b: warps
  // 0..3 take the even tiles and warps 4..7 the odd ones, all TMEM loads in flight
  auto form_keys = [&](int r0, int b) {
    const int rn = min(RX_ROUND, n_tiles - r0);
    if (ok_all) {
      static_assert(RX_ROUND <= 8, "one batch of TMEM loads per round");
      uint32_t acc[4][32];
#pragma unroll
      for (int jj = 0; jj < 4; jj++) {
        const int j = (warp >> 2) + 2 * jj;
        if (j < rn) tc::tmem_ld_x32_nowait(tmem + lane_off + RX_ACC_COL + (b * RX_ROUND + j) * HI, acc[jj]);
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int jj = 0; jj < 4; jj++) {
        const int j = (warp >> 2) + 2 * jj;
        if (j >= rn) break;
        float v[32];
#pragma unroll
        for (int h = 0; h < HI; h++) v[h] = __uint_as_float(acc[jj][h]);
        const float sc = index_head_sum(v, w2);
        const int u = (r0 + j) * RX_TILE + m;                   // pool slot
        const int32_t blk = sm.pool[u / BLK];
        const int64_t e = (int64_t)blk * BLK + (u % BLK);
        const bool ok = blk >= 0 && e < nv && u < n_slots;
        const uint32_t key = ok ? float_key(sc) : 0u;
        sm.keys[key_index(u)] = key;
        second = max(second, min(first, key));                  // the two largest keys this thread formed
        first = max(first, key);
      }
    } else {
      for (int j = warp >> 2; j < rn; j += 2) sm.keys[key_index((r0 + j) * RX_TILE + m)] = 0u;
    }
  };
  const int n_rounds = (n_tiles + RX_ROUND - 1) / RX_ROUND;
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc::fence_proxy_async_smem();                                 // the copies feed the tensor cores
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  for (int round = 0; round <= n_rounds; round++) {
    const int b = round & 1;
    // ---- 2. this round's MMAs: its tiles landed before the barrier above, and
    // its accumulators were last read by the keys of round - 2, also before it
    if (round < n_rounds && warp == RX_WARPS - 1 && lane == 0) {
      const int r0 = round * RX_ROUND, rn = min(RX_ROUND, n_tiles - r0);
      const uint64_t bdesc = tc::smem_desc(tc::smem_u32(sm.qcodes), 16, 512, tc::SW_64B);
      constexpr uint32_t id0 = tc::idesc_mxf4(RX_TILE, HI, 0, 0);
      constexpr uint32_t id1 = tc::idesc_mxf4(RX_TILE, HI, 2, 2);
      if (ok_all) {
        for (int j = 0; j < rn; j++) {
          const uint64_t adesc = tc::smem_desc(tc::smem_u32(sm.tile[b][j]), 16, 512, tc::SW_64B);
          const uint32_t d = tmem + RX_ACC_COL + (b * RX_ROUND + j) * HI;
          const uint32_t sfa = tmem + RX_SFA_COL + (b * RX_ROUND + j) * 4;
          tc::tmem_cp_32x128b_warpx4(sfa, tc::smem_desc(tc::smem_u32(sm.tile[b][j] + RX_CODES), 128, 128, tc::SW_NONE));
          tc::mma_mxf4(d, adesc, bdesc, id0, sfa, tmem + RX_SFB_COL, 0);
          tc::mma_mxf4(d, adesc + 2, bdesc + 2, id1, sfa, tmem + RX_SFB_COL, 1);   // next 32 bytes of K
        }
      }
      tc::commit(&sm.mma_done[b]);
    }
    __syncwarp();
    // ---- the previous round's products are complete: its tiles may be
    // overwritten by the next round's copies, its accumulators hold its scores
    if (round >= 1) {
      if (!tc::bar_wait(&sm.mma_done[b ^ 1], (uint32_t)((round - 1) >> 1) & 1u)) {
        if (tid == 0) report(p.hdr, CSA2_ERR_TIMEOUT, 2);
        ok_all = false;
      }
      tc::fence_after_sync();
    }
    if (round + 1 < n_rounds) issue_copies((round + 1) * RX_ROUND, b ^ 1);
    if (round >= 1) form_keys((round - 1) * RX_ROUND, b ^ 1);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();                                    // accumulators read before they are written again
    __syncthreads();
    tc::fence_after_sync();
  }
  if (warp == 0) tc::tmem_dealloc(tmem, RX_TMEM_COLS);

  // ---- 4. exact top-K over the pool's slot keys, written in slot order
  int32_t* sel = p.sel + (int64_t)bq * p.K;
  static_assert(RX_TILE % 64 == 0 && RX_SLOTS / 64 == RX_THREADS, "one key row per select thread");
  const int ns = cta_select(sm.keys, n_tiles * RX_TILE, p.K, first, second, sm,
                                                  [&](int u, int r) {
    sel[r] = sm.pool[u / BLK] * BLK + (u % BLK);
  });
  // the attention may be scheduled now (it reads sel after its own wait, which
  // returns once this grid has completed and its writes are visible)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = ns + tid; i < p.K; i += RX_THREADS) sel[i] = -1;
}

cudaError_t launch_reindex_select(IsParams p, cudaStream_t stream) {
  if (p.B == 0 || p.Q == 0) return cudaSuccess;
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.ensure([](int) {
    return cudaFuncSetAttribute(reindex_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RX_SMEM);
  });
  if (e != cudaSuccess) return e;
  if (p.M < 1 || p.M > CSA2_MAX_M) return cudaErrorInvalidValue;
  const int64_t BQ = (int64_t)p.B * p.Q;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)BQ);
  cfg.blockDim = dim3(RX_THREADS);
  cfg.dynamicSmemBytes = RX_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // set-up overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reindex_select_kernel, p);
}

}  // namespace csa2
