// (b) Fused Reindex layer: the lightning-indexer scores of the candidate pool
// and the exact top-K over them, in one kernel with one thread-block cluster
// per query token.
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4 (a Reindex layer
// scores only the entries of the candidate blocks its source layer chose and
// keeps its own top-512), §2.4.4 (FP4 indexer Q and K); "4. 层维度(下):CSA2 与
// 每 token 890 字节" §4.4 (index K is OCP MXFP4), §4.7 (hierarchical sparse
// indexing).
//
// A cluster of 6 CTAs (256 threads each, one per SM) takes one query: six is
// the largest cluster size for which 16 such clusters are resident at once on
// 152 SMs.  CTA r scores a contiguous sixth of the pool slots (at most 22
// tiles of 128 = 16 blocks of 8 entries each) in bulk-synchronous phases, with
// no per-tile hand-offs:
//   1. every warp copies whole tiles (one 512-byte block of index codes per
//      warp instruction, into the SW64 K-major layout, plus the blocks' scale
//      words) with cp.async; one warp also quantises the query to MXFP4;
//   2. warps 0..3 store the E8M0 scale words of every tile (A operand) and of
//      the query (B operand, replicated to every lane quarter) in TMEM;
//   3. one thread issues the block-scaled MMAs (M = 128 entries, N = 32 heads,
//      K = 128 as two K = 64 halves) for up to 13 tiles at a time into 13
//      TMEM accumulators; all warps then read them back (lane = entry, column =
//      head) and form s = sum_h w_h ReLU(q_h . k), kept as an order-preserving
//      key per pool slot (0 for slots outside the search domain);
//   4. the cluster runs one exact radix select over all slot keys: four 8-bit
//      digit passes, each CTA pushing its digit histogram into every CTA's
//      shared memory before one cluster barrier, so that all derive the same
//      threshold digit from the same data; the same histograms give every
//      CTA's count above and at the threshold, which places every CTA's
//      chosen entries in pool-slot order without a further exchange.
// Products of E2M1 values scaled by powers of two are exact; the accumulation
// is fp32.  Ties go to the lower pool slot (= lower entry for an ascending
// pool).  The MMA wait is bounded and reports CSA2_ERR_TIMEOUT.
#include <cstddef>

#include "index_query.cuh"
#include "host_once.cuh"
#include "params.cuh"
#include "tc.cuh"

namespace csa2 {

constexpr int RX_THREADS = 256;
constexpr int RX_WARPS = RX_THREADS / 32;
constexpr int RX_CL = 6;                                        // CTAs per query
constexpr int RX_TILE = 128;                                    // pool slots per tile
constexpr int RX_MAX_TILES = (CSA2_MAX_M * BLK / RX_TILE + RX_CL - 1) / RX_CL;   // 22
constexpr int RX_ROUND = 13;                                    // TMEM accumulators per MMA round
constexpr int RX_ROUNDS = (RX_MAX_TILES + RX_ROUND - 1) / RX_ROUND;
constexpr int RX_CODES = RX_TILE * IDX_CODE_BYTES;              // 8192
constexpr int RX_TILE_BYTES = RX_CODES + 512;                   // codes + 512 B scale words (SW64 atoms: 512 B aligned)
constexpr int RX_TMEM_COLS = 512;
constexpr int RX_ACC_COL = 0;                                   // RX_ROUND accumulators of 32 columns
constexpr int RX_SFA_COL = RX_ROUND * HI;                       // 4 columns per tile
constexpr int RX_SFB_COL = RX_SFA_COL + 4 * RX_MAX_TILES;
static_assert(RX_SFB_COL + 4 <= RX_TMEM_COLS, "TMEM columns");

struct RxSmem {
  uint8_t tile[RX_MAX_TILES][RX_TILE_BYTES];   // SW64 codes, then 128 scale words
  uint8_t qcodes[HI * IDX_CODE_BYTES];          // 2 KB, SW64
  int32_t pool[RX_MAX_TILES * 16];              // this CTA's blocks (-1: none)
  float w[HI];
  uint32_t sfb[HI];
  uint32_t keys[RX_MAX_TILES * RX_TILE];        // slot keys; 0 = outside the search domain
  alignas(16) uint32_t hist[256];               // this CTA's digit histogram of the current pass
  alignas(16) uint32_t rows[2][RX_CL][256];     // every CTA's histogram, pushed by its owner (double buffered)
  int32_t gt_all[RX_CL];                       // every CTA's keys above the threshold (same in all CTAs)
  int32_t eq_all[RX_CL];                       // every CTA's keys equal to it
  int32_t wsum[RX_WARPS];
  int32_t bcast[4];
  uint32_t suf[257];                            // cluster-wide suffix sums of the current histogram
  uint64_t mma_done[RX_ROUNDS];
  uint64_t bar_rows[2];                         // rows[buf] holds every CTA's histogram of the pass
  uint32_t tmem_base;
};
constexpr size_t RX_SMEM = sizeof(RxSmem) + 1024;
static_assert(RX_SMEM <= 227 * 1024, "shared memory");

// Exclusive prefix sum over the CTA (RX_THREADS threads); *total receives the sum.
__device__ int cta_exclusive_scan(int v, RxSmem& fs, int* total) {
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

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Top-K over the keys of every CTA of the cluster (key 0 = not a candidate) by
// (key desc, slot asc), where CTA r's keys[0..n) are slots that follow those of
// CTAs 0..r-1.  Exact radix select over four 8-bit digits.  In every pass each
// CTA builds the histogram of the digit over its keys that match the prefix
// chosen so far (warp-aggregated with match_any in the first pass, where most
// keys share a digit) and stores it into row crank of every CTA's row array
// by asynchronous remote stores, which an mbarrier per row buffer counts in
// bytes (no cluster barrier, no releasing fence); then every CTA holds all
// histograms, turns each row into suffix sums (keys with a digit >= b), and
// finds the same threshold
// digit and the same number of ties still to take.  The suffix sums also give,
// for every CTA, its keys above the threshold digit, and after the last digit
// its keys equal to the threshold, so the output offsets need no further
// exchange.  CTA r calls out(i, rank) for its chosen keys (ties in slot order,
// ranks after those of CTAs 0..r-1) and the function returns the cluster
// total.  Each thread keeps its contiguous chunk of keys in registers.
template <class Out>
__device__ int cluster_select(const uint32_t* keys, int n, int K, int crank, RxSmem& fs, WsHeader* hdr, Out out) {
  constexpr int KPT = (RX_MAX_TILES * RX_TILE + RX_THREADS - 1) / RX_THREADS;   // keys per thread
  static_assert(RX_THREADS == 256, "one histogram bin per thread");
  static_assert(RX_CL <= RX_WARPS, "one warp per CTA row");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (n + RX_THREADS - 1) / RX_THREADS;                         // <= KPT
  const int i0 = min(n, tid * chunk), i1 = min(n, i0 + chunk);
  uint32_t kr[KPT];
#pragma unroll
  for (int j = 0; j < KPT; j++) kr[j] = (i0 + j < i1) ? keys[i0 + j] : 0u;
  if (tid < RX_CL) {
    fs.gt_all[tid] = 0;
    fs.eq_all[tid] = 0;
  }
  fs.hist[tid] = 0;
  __syncthreads();
  cluster_wait();        // (arrived at set-up) every CTA runs and its row barriers are initialised

  const uint32_t hist_base = tc::smem_u32(fs.hist);
  uint32_t prefix = 0, mask = 0;
  int remaining = K;
  bool take_all = false;                                   // at most K candidates in the cluster
#pragma unroll 1
  for (int pass = 0; pass < 4; pass++) {
    const int shift = 24 - 8 * pass, buf = pass & 1;
#pragma unroll
    for (int j = 0; j < KPT; j++) {
      const uint32_t k = kr[j];
      const bool ok = k != 0u && (k & mask) == prefix;
      const uint32_t digit = (k >> shift) & 255u;
      if (pass == 0) {                                     // few distinct digits: aggregate per warp
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, ok ? digit : 256u);
        if (ok && lane == __ffs(peers) - 1)
          asm volatile("red.shared.add.u32 [%0], %1;" :: "r"(hist_base + 4u * digit), "r"((uint32_t)__popc(peers)) : "memory");
      } else if (ok) {
        asm volatile("red.shared.add.u32 [%0], 1;" :: "r"(hist_base + 4u * digit) : "memory");
      }
    }
    __syncthreads();
    if (tid == 0) tc::bar_arrive_expect_tx(&fs.bar_rows[buf], (uint32_t)(RX_CL * 256 * 4));
    if (tid < 64) {                                        // push this CTA's histogram to every CTA
      const uint4 v = *reinterpret_cast<const uint4*>(&fs.hist[4 * tid]);
      const uint32_t local = tc::smem_u32(&fs.rows[buf][crank][4 * tid]), lbar = tc::smem_u32(&fs.bar_rows[buf]);
#pragma unroll
      for (int r = 0; r < RX_CL; r++) {
        uint32_t a, rb;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(r));
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(lbar), "r"(r));
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                     :: "r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rb) : "memory");
      }
    }
    // Every CTA's histogram of this pass has landed here.  A CTA pushes into
    // rows[buf] again two passes later, after it has seen this CTA's push of
    // the pass in between, which this CTA makes only after it has finished
    // reading rows[buf]; so the two buffers never overlap in use.
    if (!tc::bar_wait(&fs.bar_rows[buf], (uint32_t)((pass >> 1) & 1)) && tid == 0)
      report(hdr, CSA2_ERR_TIMEOUT, 20 + pass);
    if (warp < RX_CL) {                                    // row `warp` -> suffix sums, in place
      uint32_t* row = fs.rows[buf][warp];
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; q++) { c[q] = row[255 - 8 * lane - q]; sum += c[q]; }
      uint32_t incl = sum;                                 // bins 255 .. 255 - 8 lane - 7
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      uint32_t run = incl - sum;
#pragma unroll
      for (int q = 0; q < 8; q++) { run += c[q]; row[255 - 8 * lane - q] = run; }
    }
    __syncthreads();
    fs.hist[tid] = 0;                                      // for the next pass (pushed from registers)
    {
      uint32_t t = 0;
#pragma unroll
      for (int r = 0; r < RX_CL; r++) t += fs.rows[buf][r][tid];
      fs.suf[tid] = t;                                     // cluster keys with digit >= tid
      if (tid == 0) fs.suf[256] = 0u;
    }
    __syncthreads();
    if (pass == 0 && fs.suf[0] <= (uint32_t)remaining) {
      if (tid == 0) fs.bcast[0] = -1;                      // at most K candidates: take them all
    } else {
      const uint32_t here = fs.suf[tid], above = fs.suf[tid + 1];
      if (here >= (uint32_t)remaining && above < (uint32_t)remaining) {
        fs.bcast[0] = tid;                                 // the digit of the K-th largest key
        fs.bcast[1] = remaining - (int)above;
        fs.bcast[2] = (int)(here - above);                 // keys of the cluster in that digit's bin
      }
    }
    __syncthreads();
    const int d = fs.bcast[0];
    // the rest of the threshold bin is taken whole: the keys' remaining bits
    // need not be looked at (the usual case after the third digit)
    const bool whole = d >= 0 && fs.bcast[2] == fs.bcast[1];
    if (tid < RX_CL) {
      const uint32_t* row = fs.rows[buf][tid];
      fs.gt_all[tid] += (int)(d < 0 ? row[0] : (d < 255 ? row[d + 1] : 0u));
      if (pass == 3 || whole) fs.eq_all[tid] = (int)(row[d] - (d < 255 ? row[d + 1] : 0u));
    }
    if (d < 0) {                                           // every valid key is taken
      take_all = true;
      remaining = 0;
      break;
    }
    prefix |= (uint32_t)d << shift;
    mask |= 255u << shift;
    remaining = fs.bcast[1];
    __syncthreads();                                       // bcast read before the next pass writes it
    if (whole) break;
  }
  const uint32_t thr = prefix;
  const int take_eq = remaining;                           // keys equal to thr still to take, in slot order
  __syncthreads();
  if (warp == 0) {
    // lane r < RX_CL: CTA r's counts; ties go to the lowest CTAs first
    const int g = lane < RX_CL ? fs.gt_all[lane] : 0, e = lane < RX_CL ? fs.eq_all[lane] : 0;
    int e_incl = e;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, e_incl, off);
      if (lane >= off) e_incl += y;
    }
    const int budget = max(0, take_eq - (e_incl - e));     // ties this CTA may still take
    const int taken = min(e, budget);
    int t_incl = g + taken;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t_incl, off);
      if (lane >= off) t_incl += y;
    }
    const int my_base = __shfl_sync(0xFFFFFFFFu, t_incl - g - taken, crank);
    const int my_budget = __shfl_sync(0xFFFFFFFFu, budget, crank);
    const int total = __shfl_sync(0xFFFFFFFFu, t_incl, 31);
    if (lane == 0) {
      fs.bcast[0] = my_base;
      fs.bcast[1] = my_budget;
      fs.bcast[2] = total;
    }
  }
  int gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < KPT; j++) {
    const uint32_t k = kr[j];
    if (k == 0u) continue;
    const uint32_t km = k & mask;                          // digits fixed so far (all 32 bits after 4 passes)
    if (take_all || km > thr) gt++;
    else if (km == thr) eq++;
  }
  // one scan of (gt, eq) packed in 16-bit halves (a CTA holds < 2^16 keys)
  int both_tot;
  const int both_before = cta_exclusive_scan((gt << 16) | eq, fs, &both_tot);   // (its barriers publish bcast)
  const int gt_before = both_before >> 16, eq_before = both_before & 0xFFFF;
  const int my_base = fs.bcast[0], my_budget = fs.bcast[1], total = fs.bcast[2];
  const int mine_eq = max(0, min(eq, my_budget - eq_before));
  int r = my_base + gt_before + min(eq_before, my_budget);
  int used = 0;
#pragma unroll
  for (int j = 0; j < KPT; j++) {
    const uint32_t k = kr[j];
    if (k == 0u) continue;
    const uint32_t km = k & mask;
    bool take = take_all || km > thr;
    if (!take && km == thr && used < mine_eq) { take = true; used++; }
    if (take) out(i0 + j, r++);
  }
  return total;                    // every push into this CTA has landed
}

__global__ void __launch_bounds__(RX_THREADS, 1) reindex_select_kernel(IsParams p) {
  extern __shared__ unsigned char smem_raw[];
  RxSmem& sm = *reinterpret_cast<RxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bq = (int)(blockIdx.x / RX_CL), crank = (int)(blockIdx.x % RX_CL);
  const int b = bq / p.Q;

  // ---- set-up: TMEM, barriers, head weights, this CTA's pool blocks
  if (warp == 0) tc::tmem_alloc(&sm.tmem_base, RX_TMEM_COLS);
  if (tid == 0) {
    for (int r = 0; r < RX_ROUNDS; r++) tc::bar_init(&sm.mma_done[r], 2);   // one commit per issuing thread
    tc::bar_init(&sm.bar_rows[0], 1);
    tc::bar_init(&sm.bar_rows[1], 1);
    tc::bar_init_fence();
  }
  // everything above reads no input: with programmatic dependent launch it
  // overlaps the previous kernel, which may have produced the pool or the queries
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[b]);
  if (nv > p.cap) {
    if (tid == 0 && crank == 0) report(p.hdr, CSA2_ERR_BOUNDS, nv);
    nv = p.cap;
  }
  const int64_t n_slots = (int64_t)p.M * BLK;
  const int64_t t0 = (int64_t)crank * p.entries_per_cta;          // first tile of this CTA
  int64_t t1 = t0 + p.entries_per_cta;
  const int64_t n_tiles = ceil_div(n_slots, RX_TILE);
  if (t1 > n_tiles) t1 = n_tiles;
  const int n = (int)(t1 > t0 ? t1 - t0 : 0);                    // <= RX_MAX_TILES (host)
  const int64_t row_base = (int64_t)b * p.cap;

  if (tid < HI) sm.w[tid] = p.w_head[(int64_t)bq * HI + tid];
  for (int i = tid; i < n * 16; i += RX_THREADS) {
    const int64_t pi = t0 * 16 + i;
    int32_t blk = pi < p.M ? p.pool[(int64_t)bq * p.M + pi] : -1;
    if (blk >= 0 && (int64_t)blk * BLK >= p.cap) {
      report(p.hdr, CSA2_ERR_BOUNDS, blk);
      blk = -1;
    }
    sm.pool[i] = blk;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  // waited for before the first histogram push; the init fence above releases
  // the row barriers, so the arrival itself is relaxed
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---- 1. copies: warp w takes tiles w, w + 8, w + 16; one warp instruction per block
  for (int i = warp; i < n; i += RX_WARPS) {
    uint8_t* codes = sm.tile[i];
    const int32_t my_blk = sm.pool[i * 16 + (lane & 15)];
    const int r = lane >> 2, c = lane & 3;                      // entry of the block, 16-byte chunk
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
  if (warp == RX_WARPS - 1) quantize_index_query_warp(p.q_idx + (int64_t)bq * HI * DI, sm.qcodes, sm.sfb);
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc::fence_proxy_async_smem();                                 // copies and query codes feed the tensor cores
  __syncthreads();

  // ---- 2. the query's scale words to TMEM lane 32 q + head of every quarter q
  // (the tiles' words follow by tcgen05.cp, each just before its MMAs)
  if (warp < 4) {
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    tc::tmem_st_x1(tmem + lane_off + RX_SFB_COL, sm.sfb[lane]);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // ---- 3. MMAs in rounds of RX_ROUND tiles, then the scores of the round as keys
  const int q4 = warp & 3;                                      // TMEM lane quarter of this warp
  const int m = q4 * 32 + lane;                                 // tile row = slot within the tile
  const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
  bool ok_all = true;
  for (int r0 = 0, round = 0; r0 < n; r0 += RX_ROUND, round++) {
    const int rn = min(RX_ROUND, n - r0);
    if (lane == 0 && warp < 2) {             // two issuing threads: even and odd tiles of the round
      const uint64_t bdesc = tc::smem_desc(tc::smem_u32(sm.qcodes), 16, 512, tc::SW_64B);
      constexpr uint32_t id0 = tc::idesc_mxf4(RX_TILE, HI, 0, 0);
      constexpr uint32_t id1 = tc::idesc_mxf4(RX_TILE, HI, 2, 2);
      for (int j = warp; j < rn; j += 2) {
        const int i = r0 + j;
        const uint64_t adesc = tc::smem_desc(tc::smem_u32(sm.tile[i]), 16, 512, tc::SW_64B);
        const uint32_t d = tmem + RX_ACC_COL + j * HI, sfa = tmem + RX_SFA_COL + i * 4;
        tc::tmem_cp_32x128b_warpx4(sfa, tc::smem_desc(tc::smem_u32(sm.tile[i] + RX_CODES), 128, 128, tc::SW_NONE));
        tc::mma_mxf4(d, adesc, bdesc, id0, sfa, tmem + RX_SFB_COL, 0);
        tc::mma_mxf4(d, adesc + 2, bdesc + 2, id1, sfa, tmem + RX_SFB_COL, 1);   // next 32 bytes of K
      }
      tc::commit(&sm.mma_done[round]);
    }
    __syncwarp();
    if (!tc::bar_wait(&sm.mma_done[round], 0)) {
      if (lane == 0) report(p.hdr, CSA2_ERR_TIMEOUT, 2);
      ok_all = false;
    }
    tc::fence_after_sync();
    if (ok_all) {
      unsigned long long w2[HI / 2];
      pack_head_weights(sm.w, w2);
      // warps 0..3 take the even accumulators and warps 4..7 the odd ones,
      // four TMEM loads in flight per batch
      for (int jb = warp >> 2; jb < rn; jb += 8) {
        uint32_t acc[4][32];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          const int j = jb + 2 * jj;
          if (j < rn) tc::tmem_ld_x32_nowait(tmem + lane_off + RX_ACC_COL + j * HI, acc[jj]);
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          const int j = jb + 2 * jj;
          if (j >= rn) break;
          float v[32];
#pragma unroll
          for (int h = 0; h < HI; h++) v[h] = __uint_as_float(acc[jj][h]);
          const float sc = index_head_sum(v, w2);
          const int u = (r0 + j) * RX_TILE + m;                 // slot within this CTA
          const int32_t blk = sm.pool[u / BLK];
          const int64_t e = (int64_t)blk * BLK + (u % BLK);
          const bool ok = blk >= 0 && e < nv && t0 * RX_TILE + u < n_slots;
          sm.keys[u] = ok ? float_key(sc) : 0u;
        }
      }
    } else {
      for (int j = warp >> 2; j < rn; j += 2) sm.keys[(r0 + j) * RX_TILE + m] = 0u;
    }
    tc::fence_before_sync();
    __syncthreads();                                            // accumulators free for the next round
    tc::fence_after_sync();
  }
  if (warp == 0) tc::tmem_dealloc(tmem, RX_TMEM_COLS);

  // ---- 4. exact top-K over the whole pool, across the cluster
  int32_t* sel = p.sel + (int64_t)bq * p.K;
  const int ns = cluster_select(sm.keys, n * RX_TILE, p.K, crank, sm, p.hdr, [&](int i, int r) {
    sel[r] = sm.pool[i / BLK] * BLK + (i % BLK);
  });
  // the attention may be scheduled now (it reads sel after its own wait, which
  // returns once this grid has completed and its writes are visible)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (crank == RX_CL - 1)
    for (int i = ns + tid; i < p.K; i += RX_THREADS) sel[i] = -1;
}

cudaError_t launch_reindex_select(IsParams p, cudaStream_t stream) {
  if (p.B == 0 || p.Q == 0) return cudaSuccess;
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.ensure([](int) {
    return cudaFuncSetAttribute(reindex_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RX_SMEM);
  });
  if (e != cudaSuccess) return e;
  const int64_t tiles = ceil_div((int64_t)p.M * BLK, RX_TILE);
  p.entries_per_cta = ceil_div(tiles, RX_CL);     // tiles per CTA (<= 22)
  if (p.entries_per_cta > RX_MAX_TILES) return cudaErrorInvalidValue;
  const int64_t BQ = (int64_t)p.B * p.Q;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(BQ * RX_CL));
  cfg.blockDim = dim3(RX_THREADS);
  cfg.dynamicSmemBytes = RX_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = RX_CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // set-up overlaps the previous kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, reindex_select_kernel, p);
}

}  // namespace csa2
