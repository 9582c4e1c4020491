// (b) HSI candidate blocks and top-K entry selection.
//
// Sources: "4. 层维度(下):CSA2 与每 token 890 字节" §4.7 (g_r(t) = max over the
// block of 8, TopM over blocks with M = 2048, pool P_t = union of the chosen
// blocks, |P_t| <= 16384; the block holding the newest visible position is set
// to +inf); "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4 (the last block
// is padded with -inf before the block max; the Full layer's own top-K is taken
// over all visible entries; Reindex layers choose inside the pool).
//
// Selection is an exact radix select on order-preserving 32-bit keys of the
// binary32 scores (four 8-bit digit passes, most significant first, with
// warp-aggregated shared-memory histograms), followed by an order-preserving
// compaction that keeps every key above the threshold and the lowest-index
// keys equal to it.  Output ids are ascending and padded with -1.
#include <mutex>

#include "host_once.cuh"
#include "params.cuh"

namespace csa2 {

constexpr int SEL_THREADS = 1024;

// ------------------------------------------------------------------ block max
struct BlockMaxParams {
  const float* scores;   // [B*Q][max_n]
  const int64_t* q_pos;
  const int32_t* n_entries;
  int m, Q;
  int64_t max_n, nb_max;
  uint32_t* gkeys;       // [B*Q][nb_max]
  int64_t per_row;       // CTAs per row
};

__global__ void block_max_kernel(BlockMaxParams p) {
  const int64_t bq = (int64_t)blockIdx.x / p.per_row;
  const int64_t r = ((int64_t)blockIdx.x % p.per_row) * blockDim.x + threadIdx.x;
  int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[bq / p.Q]);
  if (nv > p.max_n) nv = p.max_n;
  const int64_t nb = ceil_div(nv, BLK);
  if (r >= nb) return;
  const float* s = p.scores + (int64_t)bq * p.max_n + r * BLK;
  float g = -INFINITY;
  int64_t lim = nv - r * BLK;
  if (lim > BLK) lim = BLK;
  for (int i = 0; i < lim; i++) g = fmaxf(g, s[i]);
  if (r == (nv - 1) / BLK) g = INFINITY;     // newest visible block is always kept
  p.gkeys[(int64_t)bq * p.nb_max + r] = float_key(g);
}

// ------------------------------------------------------------- block helpers
struct ScanSmem {
  uint32_t hist[256];
  long long warp_sums[SEL_THREADS / 32];
  long long bcast[4];
};

// exclusive prefix sum over the block; returns this thread's offset, and the total in *total
__device__ long long block_exclusive_scan(long long v, ScanSmem& sm, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    long long y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sm.warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = (lane < SEL_THREADS / 32) ? sm.warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      long long y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    sm.warp_sums[lane] = w;      // inclusive
  }
  __syncthreads();
  long long base = (warp > 0) ? sm.warp_sums[warp - 1] : 0;
  *total = sm.warp_sums[SEL_THREADS / 32 - 1];
  __syncthreads();
  return base + x - v;
}

// Key source: valid(i) and key(i) for i in [0, n).
struct FullKeys {             // scores of entries 0..n-1
  const float* s;
  __device__ bool get(int64_t i, uint32_t& k) const { k = float_key(s[i]); return true; }
};
struct PoolKeys {             // pool layout: -inf marks a slot outside the domain
  const float* s;
  __device__ bool get(int64_t i, uint32_t& k) const {
    float v = s[i];
    k = float_key(v);
    return v != -INFINITY;
  }
};
struct RawKeys {              // precomputed keys (block maxima)
  const uint32_t* k;
  __device__ bool get(int64_t i, uint32_t& kk) const { kk = k[i]; return true; }
};
struct IdentityIds { __device__ int64_t operator()(int64_t i) const { return i; } };
struct PoolIds {
  const int32_t* blocks;
  __device__ int64_t operator()(int64_t s) const { return (int64_t)blocks[s / BLK] * BLK + (s % BLK); }
};

// Selects the K largest keys of n (ties to the lower position) and writes
// ids(position) ascending into out[0..K), padding with -1.  Whole block.
template <class Keys, class Ids>
__device__ void radix_select_block(const Keys& keys, const Ids& ids, int64_t n, int K, int32_t* out,
                                   ScanSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // number of valid keys
  long long cnt = 0;
  for (int64_t i = tid; i < n; i += SEL_THREADS) {
    uint32_t k;
    cnt += keys.get(i, k) ? 1 : 0;
  }
  long long n_valid;
  block_exclusive_scan(cnt, sm, &n_valid);

  uint32_t thr = 0;          // threshold key
  long long take_eq = 0;     // keys == thr to keep (lowest positions first)
  if (n_valid > K) {
    uint32_t prefix = 0, mask = 0;
    long long remaining = K;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += SEL_THREADS) sm.hist[i] = 0;
      __syncthreads();
      for (int64_t base = 0; base < n; base += SEL_THREADS) {
        int64_t i = base + tid;
        uint32_t k = 0;
        bool ok = (i < n) && keys.get(i, k) && ((k & mask) == prefix);
        uint32_t digit = ok ? ((k >> shift) & 255u) : 256u;
        uint32_t peers = __match_any_sync(0xFFFFFFFFu, digit);
        int leader = __ffs(peers) - 1;
        if (ok && lane == leader) atomicAdd(&sm.hist[digit], (uint32_t)__popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l .. 248-8l (descending)
        uint32_t c[8];
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < 8; q++) { c[q] = sm.hist[255 - 8 * lane - q]; sum += c[q]; }
        uint32_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += y;
        }
        uint32_t excl = incl - sum;
        unsigned hit = __ballot_sync(0xFFFFFFFFu, (long long)incl >= remaining);
        int owner = __ffs(hit) - 1;
        if (lane == owner) {
          long long cum = excl;
          int d = 255 - 8 * lane;
#pragma unroll
          for (int q = 0; q < 8; q++) {
            if (cum + c[q] >= remaining) { d = 255 - 8 * lane - q; break; }
            cum += c[q];
          }
          sm.bcast[0] = d;
          sm.bcast[1] = remaining - cum;
        }
      }
      __syncthreads();
      prefix |= (uint32_t)sm.bcast[0] << shift;
      mask |= 255u << shift;
      remaining = sm.bcast[1];
      __syncthreads();
    }
    thr = prefix;
    take_eq = remaining;
  }

  // order-preserving compaction over contiguous per-thread ranges
  const int64_t chunk = ceil_div(n, SEL_THREADS);
  const int64_t i0 = (int64_t)tid * chunk;
  const int64_t i1 = (i0 + chunk < n) ? i0 + chunk : n;
  long long gt = 0, eq = 0;
  for (int64_t i = i0; i < i1; i++) {
    uint32_t k;
    if (!keys.get(i, k)) continue;
    if (n_valid <= K || k > thr) gt++;
    else if (k == thr) eq++;
  }
  long long eq_total;
  long long eq_before = block_exclusive_scan(eq, sm, &eq_total);
  long long mine_eq = take_eq - eq_before;
  if (mine_eq < 0) mine_eq = 0;
  if (mine_eq > eq) mine_eq = eq;
  long long n_sel;
  long long off = block_exclusive_scan(gt + mine_eq, sm, &n_sel);
  long long used_eq = 0;
  for (int64_t i = i0; i < i1; i++) {
    uint32_t k;
    if (!keys.get(i, k)) continue;
    bool take = (n_valid <= K) || k > thr;
    if (!take && k == thr && used_eq < mine_eq) { take = true; used_eq++; }
    if (take) out[off++] = (int32_t)ids(i);
  }
  for (int64_t i = n_sel + tid; i < K; i += SEL_THREADS) out[i] = -1;
}

// Same selection for n <= SEL_SMEM_KEYS keys staged once in shared memory
// (key 0 marks a position outside the domain: no finite score maps to 0).
// Histograms are private per warp (plain shared atomics), summed per pass.
constexpr int SEL_SMEM_KEYS = 16384;
static_assert(SEL_SMEM_KEYS == ROW_SELECT_MIN_KEYS, "long rows start where the staged path ends");
constexpr int SEL_DYN_SMEM = SEL_SMEM_KEYS * 4 + (SEL_THREADS / 32) * 256 * 4;

template <class Keys, class Ids>
__device__ void radix_select_smem(const Keys& keys, const Ids& ids, int n, int K, int32_t* out, ScanSmem& sm,
                                  uint32_t* sk, uint32_t* whist) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long cnt = 0;
  for (int i = tid; i < n; i += SEL_THREADS) {
    uint32_t k;
    const bool ok = keys.get(i, k);
    sk[i] = ok ? k : 0u;
    cnt += ok ? 1 : 0;
  }
  long long n_valid;
  block_exclusive_scan(cnt, sm, &n_valid);      // also orders the smem key writes
  uint32_t thr = 0;
  long long take_eq = 0;
  if (n_valid > K) {
    uint32_t prefix = 0, mask = 0;
    long long remaining = K;
    uint32_t* myh = whist + warp * 256;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = lane; i < 256; i += 32) myh[i] = 0;
      __syncwarp();
      for (int base = 0; base < n; base += SEL_THREADS) {     // uniform trip count for match_any
        const int i = base + tid;
        const uint32_t k = (i < n) ? sk[i] : 0u;
        const bool ok = k != 0u && (k & mask) == prefix;
        const uint32_t digit = ok ? ((k >> shift) & 255u) : 256u;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, digit);
        if (ok && lane == __ffs(peers) - 1) atomicAdd(&myh[digit], (uint32_t)__popc(peers));
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t tot = 0;
#pragma unroll 8
        for (int w = 0; w < SEL_THREADS / 32; w++) tot += whist[w * 256 + tid];
        sm.hist[tid] = tot;
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8];
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < 8; q++) { c[q] = sm.hist[255 - 8 * lane - q]; sum += c[q]; }
        uint32_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += y;
        }
        const uint32_t excl = incl - sum;
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, (long long)incl >= remaining);
        const int owner = __ffs(hit) - 1;
        if (lane == owner) {
          long long cum = excl;
          int d = 255 - 8 * lane;
#pragma unroll
          for (int q = 0; q < 8; q++) {
            if (cum + c[q] >= remaining) { d = 255 - 8 * lane - q; break; }
            cum += c[q];
          }
          sm.bcast[0] = d;
          sm.bcast[1] = remaining - cum;
        }
      }
      __syncthreads();
      prefix |= (uint32_t)sm.bcast[0] << shift;
      mask |= 255u << shift;
      remaining = sm.bcast[1];
      __syncthreads();
    }
    thr = prefix;
    take_eq = remaining;
  }
  const bool all = n_valid <= K;
  const int chunk = (n + SEL_THREADS - 1) / SEL_THREADS;
  const int i0 = tid * chunk;
  const int i1 = (i0 + chunk < n) ? i0 + chunk : n;
  long long gt = 0, eq = 0;
  for (int i = i0; i < i1; i++) {
    const uint32_t k = sk[i];
    if (k == 0u) continue;
    if (all || k > thr) gt++;
    else if (k == thr) eq++;
  }
  long long eq_total;
  const long long eq_before = block_exclusive_scan(eq, sm, &eq_total);
  long long mine_eq = take_eq - eq_before;
  if (mine_eq < 0) mine_eq = 0;
  if (mine_eq > eq) mine_eq = eq;
  long long n_sel;
  long long off = block_exclusive_scan(gt + mine_eq, sm, &n_sel);
  long long used_eq = 0;
  for (int i = i0; i < i1; i++) {
    const uint32_t k = sk[i];
    if (k == 0u) continue;
    bool take = all || k > thr;
    if (!take && k == thr && used_eq < mine_eq) { take = true; used_eq++; }
    if (take) out[off++] = (int32_t)ids(i);
  }
  for (long long i = n_sel + tid; i < K; i += SEL_THREADS) out[i] = -1;
}

// ------------------------------------------------------------------ kernels
struct BlockTopParams {
  const uint32_t* gkeys;
  const int64_t* q_pos;
  const int32_t* n_entries;
  int m, Q, M;
  int64_t nb_max;
  int32_t* pool_blocks;
};

__global__ void __launch_bounds__(SEL_THREADS) block_topm_kernel(BlockTopParams p) {
  __shared__ ScanSmem sm;
  extern __shared__ uint32_t dyn[];
  const int bq = blockIdx.x;
  int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[bq / p.Q]);
  if (nv > p.nb_max * BLK) nv = p.nb_max * BLK;
  const int64_t nb = ceil_div(nv, BLK);
  RawKeys keys{p.gkeys + (int64_t)bq * p.nb_max};
  int32_t* out = p.pool_blocks + (int64_t)bq * p.M;
  if (nb <= SEL_SMEM_KEYS)
    radix_select_smem(keys, IdentityIds{}, (int)nb, p.M, out, sm, dyn, dyn + SEL_SMEM_KEYS);
  else
    radix_select_block(keys, IdentityIds{}, nb, p.M, out, sm);
}

struct SelectParams {
  const float* scores;
  const int64_t* q_pos;
  const int32_t* n_entries;
  const int32_t* pool;     // null = all visible
  int m, Q, M, K;
  int64_t max_n;
  int32_t* sel;
};

__global__ void __launch_bounds__(SEL_THREADS) select_topk_kernel(SelectParams p) {
  __shared__ ScanSmem sm;
  extern __shared__ uint32_t dyn[];
  const int bq = blockIdx.x;
  int32_t* out = p.sel + (int64_t)bq * p.K;
  if (p.pool == nullptr) {
    int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[bq / p.Q]);
    if (nv > p.max_n) nv = p.max_n;
    FullKeys keys{p.scores + (int64_t)bq * p.max_n};
    if (nv <= SEL_SMEM_KEYS)
      radix_select_smem(keys, IdentityIds{}, (int)nv, p.K, out, sm, dyn, dyn + SEL_SMEM_KEYS);
    else
      radix_select_block(keys, IdentityIds{}, nv, p.K, out, sm);
  } else {
    PoolKeys keys{p.scores + (int64_t)bq * p.M * BLK};
    PoolIds ids{p.pool + (int64_t)bq * p.M};
    radix_select_smem(keys, ids, p.M * BLK, p.K, out, sm, dyn, dyn + SEL_SMEM_KEYS);
  }
}

static cudaError_t set_select_smem() {
  static PerDeviceOnce attrs;
  return attrs.ensure([](int) {
    cudaError_t e =
        cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_DYN_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(block_topm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_DYN_SMEM);
    return e;
  });
}

cudaError_t launch_block_topk(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m,
                              int B, int Q, int64_t max_n, int M, int32_t* pool_blocks, uint32_t* gkeys,
                              cudaStream_t stream) {
  if (B == 0 || Q == 0) return cudaSuccess;
  const int64_t nb_max = ceil_div(max_n, BLK);
  if (nb_max > 0) {
    const int64_t per_row = ceil_div(nb_max, 256);
    if ((int64_t)B * Q * per_row > 0x7FFFFFFF) return cudaErrorInvalidValue;
    BlockMaxParams bp{scores, q_pos, n_entries, m, Q, max_n, nb_max, gkeys, per_row};
    block_max_kernel<<<(unsigned)((int64_t)B * Q * per_row), 256, 0, stream>>>(bp);
  }
  cudaError_t e = set_select_smem();
  if (e != cudaSuccess) return e;
  BlockTopParams tp{gkeys, q_pos, n_entries, m, Q, M, nb_max, pool_blocks};
  block_topm_kernel<<<B * Q, SEL_THREADS, SEL_DYN_SMEM, stream>>>(tp);
  return cudaGetLastError();
}

cudaError_t launch_select_topk(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m,
                               const int32_t* pool, int M, int K, int32_t* sel, int B, int Q, int64_t max_n,
                               cudaStream_t stream) {
  if (B == 0 || Q == 0) return cudaSuccess;
  cudaError_t e = set_select_smem();
  if (e != cudaSuccess) return e;
  SelectParams sp{scores, q_pos, n_entries, pool, m, Q, M, K, max_n, sel};
  select_topk_kernel<<<B * Q, SEL_THREADS, SEL_DYN_SMEM, stream>>>(sp);
  return cudaGetLastError();
}

// ------------------------------------------------ multi-CTA selection on long rows
// A Full row holds one score per visible entry (up to the whole cache: 2^20
// and more), so one CTA per row leaves most of the GPU idle and reads the row
// five times.  Rows longer than SEL_SMEM_KEYS keys take three launches instead:
//   scan 1  many CTAs per row histogram the top 12 bits of every key (entry
//           keys for the top-K, block-maximum keys for the top-M, from the
//           same read of the scores) into a per-row histogram in global
//           memory; the row's last CTA finds the threshold bin b1 (the bin
//           holding the K-th largest key) and the count above it;
//   scan 2  the same CTAs read the row again and append every key above b1
//           to the row's list of sure picks, and every key inside b1 to a
//           candidate list as a (key, ~id) composite;
//   resolve one CTA per row and kind finishes the exact selection among the
//           candidates (8-bit digit passes over the 52 bits the composites do
//           not share, stopping as soon as the threshold bin is taken whole),
//           sorts the K ids and writes them.
// Composites order by key and then by the lower id, so the result is the
// (score desc, id asc) top-K.  A threshold bin with more than RS_CAP keys
// (scores bunched far from zero, or massive ties) sends its row to the
// single-CTA radix select, which is exact for any input.
constexpr int RS_BITS = 12;
constexpr int RS_BINS = 1 << RS_BITS;
constexpr int RS_SHIFT = 32 - RS_BITS;
constexpr int RS_CAP = 8192;                     // candidates kept per row and kind
constexpr int RS_THREADS = 256;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int RS_TILE = 512;                     // entries per warp tile: lane l holds 128 i + 4 l + c
constexpr int RS_TILES = 1;                      // warp tiles loaded together
constexpr int RS_BATCH = RS_WARPS * RS_TILE * RS_TILES;   // 8,192 entries: one batch of a scan CTA
constexpr int RS_SCAN_CTAS_PER_SM = 4;           // resident scan CTAs per SM (launch bounds)
constexpr int RS_MAX_OUT = CSA2_MAX_M;           // >= CSA2_MAX_K
constexpr uint32_t RS_STAGE_EQ = 1024;           // threshold-bin candidates staged per scan CTA
static_assert(BLK == 8, "a block is the 8 entries of two neighbouring lanes");

struct RsRow {                                   // zeroed before every selection
  uint32_t hist[RS_BINS];
  uint32_t n_gt, n_eq, done, b1, above, pad[11];
};

size_t row_select_bytes(int64_t BQ) {
  const size_t per = sizeof(RsRow) + RS_MAX_OUT * sizeof(int32_t) + RS_CAP * sizeof(unsigned long long);
  return (size_t)(2 * BQ) * per + 3 * 256;
}

struct RsParams {
  const float* scores;      // [BQ][max_n]
  const int64_t* q_pos;
  const int32_t* n_entries;
  int m, Q, K, M;           // K = 0: no entry selection; M = 0: no block selection
  int64_t max_n;
  int chunks;               // scan CTAs per row
  int batches;              // batches of RS_BATCH entries per scan CTA
  int32_t* sel;             // [BQ][K]
  int32_t* pool;            // [BQ][M]
  RsRow* rows;              // [2][BQ]: entries, then blocks
  int32_t* gt;              // [2][BQ][RS_MAX_OUT]
  unsigned long long* cand; // [2][BQ][RS_CAP]
  int64_t BQ;
};

// one block's max over 8 consecutive scores, with the newest visible block forced
struct BlockScoreKeys {
  const float* s;
  int64_t nv;
  __device__ bool get(int64_t r, uint32_t& k) const {
    if (r == (nv - 1) / BLK) { k = float_key(INFINITY); return true; }
    const int64_t e0 = r * BLK;
    float g = -INFINITY;
    for (int i = 0; i < BLK && e0 + i < nv; i++) g = fmaxf(g, s[e0 + i]);
    k = float_key(g);
    return true;
  }
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned r;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
  return r;
}

// warp-aggregated append of one 32- or 64-bit item per taking lane
template <class T>
__device__ __forceinline__ void warp_append(bool take, uint32_t* counter, T* list, uint32_t cap, T item) {
  const unsigned ball = __ballot_sync(0xFFFFFFFFu, take);
  if (ball == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(ball) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, (uint32_t)__popc(ball));
  base = __shfl_sync(0xFFFFFFFFu, base, leader);
  const uint32_t at = base + (uint32_t)__popc(ball & lanemask_lt());
  if (take && at < cap) list[at] = item;
}

// Warp-aggregated append into a CTA's shared-memory staging list of cap_s
// items; items beyond it go straight to the global list.
template <class T>
__device__ __forceinline__ void stage_append(bool take, uint32_t* s_n, T* s_list, uint32_t cap_s, uint32_t* g_n,
                                             T* g_list, uint32_t g_cap, T item) {
  const unsigned ball = __ballot_sync(0xFFFFFFFFu, take);
  if (ball == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(ball) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(s_n, (uint32_t)__popc(ball));
  base = __shfl_sync(0xFFFFFFFFu, base, leader);
  const uint32_t at = base + (uint32_t)__popc(ball & lanemask_lt());
  if (take && at < cap_s) s_list[at] = item;
  warp_append<T>(take && at >= cap_s, g_n, g_list, g_cap, item);
}

// Scores of one warp tile of RS_TILE entries from t0 (a multiple of RS_TILE):
// lane l holds entries t0 + 128 i + 4 l + c (i, c < 4), -inf past nv.  VEC:
// the row is 16-byte aligned, so each group of four is one 16-byte load.
template <bool VEC>
__device__ __forceinline__ void rs_load_tile(const float* s, int t0, int nv, float (&v)[16]) {
  const int lane = threadIdx.x & 31;
  const bool full = t0 + RS_TILE <= nv;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int e = t0 + 128 * i + 4 * lane;
    if (VEC && full) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(s + e));
      v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
    } else {
#pragma unroll
      for (int c = 0; c < 4; c++) v[4 * i + c] = e + c < nv ? __ldg(s + e + c) : -INFINITY;
    }
  }
}

// Block keys of a loaded tile: block t0/8 + 16 i + l/2 is the 8 entries of
// lanes l and l^1; its key (max, or +inf for the newest block nb - 1) is valid
// in the even lane when the block exists.
__device__ __forceinline__ void rs_block_keys(const float (&v)[16], int t0, int nb, uint32_t (&bk)[4], bool (&bok)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    float g = fmaxf(fmaxf(v[4 * i], v[4 * i + 1]), fmaxf(v[4 * i + 2], v[4 * i + 3]));
    g = fmaxf(g, __shfl_xor_sync(0xFFFFFFFFu, g, 1));
    const int r = t0 / BLK + 16 * i + (lane >> 1);
    bk[i] = r == nb - 1 ? float_key(INFINITY) : float_key(g);
    bok[i] = (lane & 1) == 0 && r < nb;
  }
}

struct RsRowInfo {
  int nv, nb;                                    // < 2^31 (entry ids are int32)
  bool do_e, do_b;
};

__device__ __forceinline__ RsRowInfo rs_row_info(const RsParams& p, int64_t bq) {
  RsRowInfo r;
  int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[bq / p.Q]);
  if (nv > p.max_n) nv = p.max_n;
  r.nv = (int)nv;
  r.nb = (int)ceil_div(nv, BLK);
  r.do_e = p.K > 0 && r.nv > p.K;
  r.do_b = p.M > 0 && r.nb > p.M;
  return r;
}

// Threshold bin of a complete row histogram: the bin b1 holding the K-th
// largest key, and the number of keys in higher bins.  Whole block (RS_THREADS).
__device__ void rs_threshold(RsRow& row, int K, uint32_t* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int PER = RS_BINS / RS_THREADS;      // 8 bins per thread, descending
  uint32_t h[PER], sum = 0;
#pragma unroll
  for (int q = 0; q < PER; q++) {
    h[q] = __ldcg(&row.hist[RS_BINS - 1 - PER * tid - q]);
    sum += h[q];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp; w++) before += warp_sums[w];
  const uint32_t excl = before + incl - sum;
  if (excl < (uint32_t)K && excl + sum >= (uint32_t)K) {
    uint32_t cum = excl;
#pragma unroll
    for (int q = 0; q < PER; q++) {
      if (cum + h[q] >= (uint32_t)K) {
        row.b1 = (uint32_t)(RS_BINS - 1 - PER * tid - q);
        row.above = cum;
        break;
      }
      cum += h[q];
    }
  }
  __syncthreads();
}

template <bool VEC>
__global__ void __launch_bounds__(RS_THREADS, RS_SCAN_CTAS_PER_SM) rs_hist_kernel(RsParams p) {
  extern __shared__ uint32_t rs_dyn[];
  uint32_t* hist_e = rs_dyn;
  uint32_t* hist_b = rs_dyn + RS_BINS;
  __shared__ uint32_t warp_sums[RS_WARPS];
  __shared__ int is_last;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t bq = blockIdx.x / p.chunks;
  const int chunk = (int)(blockIdx.x % p.chunks);
  const RsRowInfo ri = rs_row_info(p, bq);
  if (!ri.do_e && !ri.do_b) return;
  RsRow& row_e = p.rows[bq];
  RsRow& row_b = p.rows[p.BQ + bq];
  for (int i = tid; i < 2 * RS_BINS / 4; i += RS_THREADS) reinterpret_cast<uint4*>(rs_dyn)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  const float* s = p.scores + bq * p.max_n;
  const int e_lo = chunk * p.batches * RS_BATCH;
  for (int bt = 0; bt < p.batches; bt++) {
  float v[RS_TILES][16];
#pragma unroll
  for (int k = 0; k < RS_TILES; k++) {
    const int t0 = e_lo + ((bt * RS_TILES + k) * RS_WARPS + warp) * RS_TILE;
    if (t0 < ri.nv) rs_load_tile<VEC>(s, t0, ri.nv, v[k]);
  }
#pragma unroll
  for (int k = 0; k < RS_TILES; k++) {
    const int t0 = e_lo + ((bt * RS_TILES + k) * RS_WARPS + warp) * RS_TILE;
    if (t0 >= ri.nv) break;                      // warp-uniform
    if (ri.do_e) {
#pragma unroll
      for (int j = 0; j < 16; j++)               // -inf past nv is counted in bin 0x007, then taken back
        atomicAdd(&hist_e[float_key(v[k][j]) >> RS_SHIFT], 1u);
    }
    if (ri.do_b) {
      uint32_t bk[4];
      bool bok[4];
      rs_block_keys(v[k], t0, ri.nb, bk, bok);
#pragma unroll
      for (int i = 0; i < 4; i++)
        if (bok[i]) atomicAdd(&hist_b[bk[i] >> RS_SHIFT], 1u);
    }
  }
  }
  if (ri.do_e && e_lo + p.batches * RS_BATCH > ri.nv && e_lo < ri.nv) {
    // the padding of the row's last tile went to the -inf bin
    const int last_t0 = (ri.nv - 1) / RS_TILE * RS_TILE;
    if (tid == 0) atomicSub(&hist_e[float_key(-INFINITY) >> RS_SHIFT], (uint32_t)(last_t0 + RS_TILE - ri.nv));
  }
  __syncthreads();
  for (int b4 = tid; b4 < RS_BINS / 4; b4 += RS_THREADS) {
    if (ri.do_e) {
      const uint4 c = reinterpret_cast<const uint4*>(hist_e)[b4];
      if (c.x) atomicAdd(&row_e.hist[4 * b4], c.x);
      if (c.y) atomicAdd(&row_e.hist[4 * b4 + 1], c.y);
      if (c.z) atomicAdd(&row_e.hist[4 * b4 + 2], c.z);
      if (c.w) atomicAdd(&row_e.hist[4 * b4 + 3], c.w);
    }
    if (ri.do_b) {
      const uint4 c = reinterpret_cast<const uint4*>(hist_b)[b4];
      if (c.x) atomicAdd(&row_b.hist[4 * b4], c.x);
      if (c.y) atomicAdd(&row_b.hist[4 * b4 + 1], c.y);
      if (c.z) atomicAdd(&row_b.hist[4 * b4 + 2], c.z);
      if (c.w) atomicAdd(&row_b.hist[4 * b4 + 3], c.w);
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&row_e.done, 1u) == (uint32_t)p.chunks - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (ri.do_e) rs_threshold(row_e, p.K, warp_sums);
  if (ri.do_b) rs_threshold(row_b, p.M, warp_sums);
}

template <bool VEC>
__global__ void __launch_bounds__(RS_THREADS, RS_SCAN_CTAS_PER_SM) rs_filter_kernel(RsParams p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bq = blockIdx.x / p.chunks;
  const int chunk = (int)(blockIdx.x % p.chunks);
  const RsRowInfo ri = rs_row_info(p, bq);
  if (!ri.do_e && !ri.do_b) return;
  RsRow& row_e = p.rows[bq];
  RsRow& row_b = p.rows[p.BQ + bq];
  const uint32_t b1e = ri.do_e ? row_e.b1 : 0xFFFFFFFFu, b1b = ri.do_b ? row_b.b1 : 0xFFFFFFFFu;
  const bool keep_e = ri.do_e && row_e.hist[b1e] <= (uint32_t)RS_CAP;
  const bool keep_b = ri.do_b && row_b.hist[b1b] <= (uint32_t)RS_CAP;
  int32_t* gt_e = p.gt + bq * RS_MAX_OUT;
  int32_t* gt_b = p.gt + (p.BQ + bq) * RS_MAX_OUT;
  unsigned long long* cd_e = p.cand + bq * RS_CAP;
  unsigned long long* cd_b = p.cand + (p.BQ + bq) * RS_CAP;
  // this CTA's picks are staged in shared memory and published with one
  // global reservation per list at the end
  constexpr uint32_t SE = RS_STAGE_EQ;
  __shared__ int32_t s_gt_e[CSA2_MAX_K], s_gt_b[CSA2_MAX_M];
  __shared__ unsigned long long s_eq_e[SE], s_eq_b[SE];
  __shared__ uint32_t s_n[4], s_base[4];
  if (tid < 4) s_n[tid] = 0;
  __syncthreads();
  const float* s = p.scores + bq * p.max_n;
  const int e_lo = chunk * p.batches * RS_BATCH;
  for (int bt = 0; bt < p.batches; bt++) {
    float v[RS_TILES][16];
#pragma unroll
    for (int k = 0; k < RS_TILES; k++) {
      const int t0 = e_lo + ((bt * RS_TILES + k) * RS_WARPS + warp) * RS_TILE;
      if (t0 < ri.nv) rs_load_tile<VEC>(s, t0, ri.nv, v[k]);
    }
#pragma unroll
    for (int k = 0; k < RS_TILES; k++) {
      const int t0 = e_lo + ((bt * RS_TILES + k) * RS_WARPS + warp) * RS_TILE;
      if (t0 >= ri.nv) break;                    // warp-uniform
      if (ri.do_e) {
        // keys in or above the threshold bin are rare: each lane marks its value
        // slots that hold one (no votes), then the warp walks the marks, one
        // slot per lane per round, with warp-aggregated appends (a rolled loop:
        // small code, usually one or two rounds)
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < 16; j++) {
          const int e = t0 + 128 * (j >> 2) + 4 * lane + (j & 3);
          mask |= (uint32_t)((float_key(v[k][j]) >> RS_SHIFT) >= b1e && e < ri.nv) << j;
        }
        while (__any_sync(0xFFFFFFFFu, mask != 0u)) {
          const bool have = mask != 0u;
          const int j = have ? __ffs(mask) - 1 : 0;
          mask &= mask - 1u;
          float x = v[k][0];
#pragma unroll
          for (int jj = 1; jj < 16; jj++) x = jj == j ? v[k][jj] : x;
          const uint32_t key = float_key(x);
          const uint32_t d = key >> RS_SHIFT;
          const int e = t0 + 128 * (j >> 2) + 4 * lane + (j & 3);
          stage_append<int32_t>(have && d > b1e, &s_n[0], s_gt_e, CSA2_MAX_K, &row_e.n_gt, gt_e, (uint32_t)p.K,
                                (int32_t)e);
          if (keep_e)
            stage_append<unsigned long long>(have && d == b1e, &s_n[1], s_eq_e, SE, &row_e.n_eq, cd_e,
                                             (uint32_t)RS_CAP,
                                             ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)e);
        }
      }
      if (ri.do_b) {
        uint32_t bk[4];
        bool bok[4];
        rs_block_keys(v[k], t0, ri.nb, bk, bok);
        // the same walk over the (even) lanes' four block keys
        uint32_t mask = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) mask |= (uint32_t)(bok[i] && (bk[i] >> RS_SHIFT) >= b1b) << i;
        while (__any_sync(0xFFFFFFFFu, mask != 0u)) {
          const bool have = mask != 0u;
          const int i = have ? __ffs(mask) - 1 : 0;
          mask &= mask - 1u;
          uint32_t key = bk[0];
#pragma unroll
          for (int ii = 1; ii < 4; ii++) key = ii == i ? bk[ii] : key;
          const uint32_t d = key >> RS_SHIFT;
          const int r = t0 / BLK + 16 * i + (lane >> 1);
          stage_append<int32_t>(have && d > b1b, &s_n[2], s_gt_b, CSA2_MAX_M, &row_b.n_gt, gt_b, (uint32_t)p.M,
                                (int32_t)r);
          if (keep_b)
            stage_append<unsigned long long>(have && d == b1b, &s_n[3], s_eq_b, SE, &row_b.n_eq, cd_b,
                                             (uint32_t)RS_CAP,
                                             ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)r);
        }
      }
    }
  }
  __syncthreads();
  if (tid < 4) {
    const uint32_t cap_s = tid == 0 ? CSA2_MAX_K : tid == 2 ? CSA2_MAX_M : SE;
    const uint32_t c = s_n[tid] < cap_s ? s_n[tid] : cap_s;
    uint32_t* g_n = tid == 0 ? &row_e.n_gt : tid == 1 ? &row_e.n_eq : tid == 2 ? &row_b.n_gt : &row_b.n_eq;
    s_base[tid] = c ? atomicAdd(g_n, c) : 0u;
    s_n[tid] = c;
  }
  __syncthreads();
  for (uint32_t i = tid; i < s_n[0]; i += RS_THREADS)
    if (s_base[0] + i < (uint32_t)p.K) gt_e[s_base[0] + i] = s_gt_e[i];
  for (uint32_t i = tid; i < s_n[1]; i += RS_THREADS)
    if (s_base[1] + i < (uint32_t)RS_CAP) cd_e[s_base[1] + i] = s_eq_e[i];
  for (uint32_t i = tid; i < s_n[2]; i += RS_THREADS)
    if (s_base[2] + i < (uint32_t)p.M) gt_b[s_base[2] + i] = s_gt_b[i];
  for (uint32_t i = tid; i < s_n[3]; i += RS_THREADS)
    if (s_base[3] + i < (uint32_t)RS_CAP) cd_b[s_base[3] + i] = s_eq_b[i];
}

constexpr int RS_RESOLVE_SMEM = RS_CAP * 8 + (SEL_THREADS / 32) * 256 * 4 + RS_MAX_OUT * 4;

__global__ void __launch_bounds__(SEL_THREADS, 1) rs_resolve_kernel(RsParams p) {
  __shared__ ScanSmem sm;
  __shared__ uint32_t n_taken;
  __shared__ uint32_t bc[3];
  extern __shared__ __align__(16) unsigned char rs_res_dyn[];
  unsigned long long* cs = reinterpret_cast<unsigned long long*>(rs_res_dyn);
  uint32_t* whist = reinterpret_cast<uint32_t*>(rs_res_dyn + RS_CAP * 8);
  int32_t* ids = reinterpret_cast<int32_t*>(rs_res_dyn + RS_CAP * 8 + (SEL_THREADS / 32) * 256 * 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t bq = blockIdx.x;
  const int kind = blockIdx.y;                   // 0: entries (top-K), 1: blocks (top-M)
  const int KK = kind ? p.M : p.K;
  if (KK <= 0) return;
  const RsRowInfo ri = rs_row_info(p, bq);
  const int64_t n = kind ? ri.nb : ri.nv;
  int32_t* out = kind ? p.pool + bq * p.M : p.sel + bq * p.K;
  if (n <= KK) {
    for (int i = tid; i < KK; i += SEL_THREADS) out[i] = i < n ? i : -1;
    return;
  }
  const float* s = p.scores + bq * p.max_n;
  const RsRow& row = p.rows[kind * p.BQ + bq];
  const uint32_t above = row.above;
  const uint32_t n_eq = row.hist[row.b1];
  if (n_eq > (uint32_t)RS_CAP) {                 // bunched threshold bin: exact single-CTA select
    if (kind) radix_select_block(BlockScoreKeys{s, ri.nv}, IdentityIds{}, n, KK, out, sm);
    else radix_select_block(FullKeys{s}, IdentityIds{}, n, KK, out, sm);
    return;
  }
  const int32_t* gt = p.gt + (kind * p.BQ + bq) * RS_MAX_OUT;
  const unsigned long long* cd = p.cand + (kind * p.BQ + bq) * RS_CAP;
  for (uint32_t i = tid; i < above; i += SEL_THREADS) ids[i] = gt[i];
  for (uint32_t i = tid; i < n_eq; i += SEL_THREADS) cs[i] = cd[i] << RS_BITS;   // drop the shared bin bits
  if (tid == 0) n_taken = 0;
  __syncthreads();
  // Candidates are unique 64-bit values (bits 63..12 = low key bits, ~id);
  // keep the `rem` largest with digit passes from the top.
  uint32_t rem = (uint32_t)KK - above;
  unsigned long long prefix = 0, mask = 0;
  if (rem < n_eq) {
    uint32_t* myh = whist + warp * 256;
    for (int shift = 56; shift >= 8; shift -= 8) {
      for (int i = lane; i < 256; i += 32) myh[i] = 0;
      __syncwarp();
      for (uint32_t base = 0; base < n_eq; base += SEL_THREADS) {
        const uint32_t i = base + tid;
        const unsigned long long c = i < n_eq ? cs[i] : 0ull;
        const bool ok = i < n_eq && (c & mask) == prefix;
        const uint32_t digit = ok ? (uint32_t)(c >> shift) & 255u : 256u;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, digit);
        if (ok && lane == __ffs(peers) - 1) atomicAdd(&myh[digit], (uint32_t)__popc(peers));
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t tot = 0;
#pragma unroll 8
        for (int w = 0; w < SEL_THREADS / 32; w++) tot += whist[w * 256 + tid];
        sm.hist[tid] = tot;
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; q++) { c[q] = sm.hist[255 - 8 * lane - q]; sum += c[q]; }
        uint32_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += y;
        }
        const uint32_t excl = incl - sum;
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= rem);
        if (lane == __ffs(hit) - 1) {
          uint32_t cum = excl;
          int d = 255 - 8 * lane;
#pragma unroll
          for (int q = 0; q < 8; q++) {
            if (cum + c[q] >= rem) { d = 255 - 8 * lane - q; break; }
            cum += c[q];
          }
          bc[0] = (uint32_t)d;
          bc[1] = rem - cum;                     // still needed from bin d
          bc[2] = sm.hist[d];
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)bc[0] << shift;
      mask |= 255ull << shift;
      rem = bc[1];
      const bool whole = bc[2] == rem;           // the rest of the bin is taken whole
      __syncthreads();
      if (whole) break;
    }
  }
  for (uint32_t base = 0; base < n_eq; base += SEL_THREADS) {
    const uint32_t i = base + tid;
    if (i < n_eq && (cs[i] & mask) >= prefix) {
      const uint32_t at = above + atomicAdd(&n_taken, 1u);
      if (at < (uint32_t)KK) ids[at] = (int32_t)~(uint32_t)(cs[i] >> RS_BITS);
    }
  }
  __syncthreads();
  if (n <= RS_CAP * 64) {
    // ascending order through a bitmap of the row (in the candidates' space,
    // now free): one bit per chosen id, then a block-wide count of set bits
    uint32_t* bm = reinterpret_cast<uint32_t*>(cs);
    const int words = (int)((n + 31) / 32);
    for (int i = tid; i < words; i += SEL_THREADS) bm[i] = 0u;
    __syncthreads();
    for (int i = tid; i < KK; i += SEL_THREADS) atomicOr(&bm[ids[i] >> 5], 1u << (ids[i] & 31));
    __syncthreads();
    const int per = (words + SEL_THREADS - 1) / SEL_THREADS;
    const int w0 = tid * per, w1 = w0 + per < words ? w0 + per : words;
    long long cnt = 0;
    for (int w = w0; w < w1; w++) cnt += __popc(bm[w]);
    long long total;
    long long at = block_exclusive_scan(cnt, sm, &total);
    for (int w = w0; w < w1; w++)
      for (uint32_t x = bm[w]; x; x &= x - 1) out[at++] = w * 32 + __ffs(x) - 1;
    return;
  }
  // longer rows: bitonic sort of the KK ids, ascending
  int P = 1;
  while (P < KK) P <<= 1;
  for (int i = KK + tid; i < P; i += SEL_THREADS) ids[i] = 0x7FFFFFFF;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = tid; t < P / 2; t += SEL_THREADS) {
        const int i = (t / j) * 2 * j + (t % j);
        const int l = i + j;
        const int32_t a = ids[i], b = ids[l];
        if ((a > b) == ((i & k) == 0)) { ids[i] = b; ids[l] = a; }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < KK; i += SEL_THREADS) out[i] = ids[i];
}

// Full-row selection of the entry top-K (K > 0) and/or the block top-M
// (M > 0) of every row, with `scratch` (row_select_bytes(B*Q), 256-byte
// aligned) as per-row histograms and lists.
cudaError_t launch_row_select(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m, int B,
                              int Q, int64_t max_n, int K, int32_t* sel, int M, int32_t* pool, void* scratch,
                              cudaStream_t stream) {
  const int64_t BQ = (int64_t)B * Q;
  if (BQ == 0) return cudaSuccess;
  if (max_n > 0x7FFFFFFF - 2 * (int64_t)RS_BATCH) return cudaErrorInvalidValue;   // entry ids are int32
  static PerDeviceOnce attrs;
  cudaError_t ae = attrs.ensure([](int) {
    cudaError_t e = cudaFuncSetAttribute(rs_resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         RS_RESOLVE_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(rs_hist_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               2 * RS_BINS * (int)sizeof(uint32_t));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(rs_hist_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               2 * RS_BINS * (int)sizeof(uint32_t));
    return e;
  });
  if (ae != cudaSuccess) return ae;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  unsigned char* cur = static_cast<unsigned char*>(scratch);
  RsParams p{};
  p.scores = scores;
  p.q_pos = q_pos;
  p.n_entries = n_entries;
  p.m = m;
  p.Q = Q;
  p.K = sel ? K : 0;
  p.M = pool ? M : 0;
  p.max_n = max_n;
  // one wave of scan CTAs where the rows allow it: batches per CTA from the total
  int dev_sms = 0;
  if ((ae = device_sms(&dev_sms)) != cudaSuccess) return ae;
  const int64_t row_batches = max_n > 0 ? ceil_div(max_n, RS_BATCH) : 1;
  int64_t per = ceil_div(BQ * row_batches, (int64_t)RS_SCAN_CTAS_PER_SM * dev_sms);
  if (per < 1) per = 1;
  if (per > row_batches) per = row_batches;
  p.batches = (int)per;
  p.chunks = (int)ceil_div(row_batches, per);
  p.sel = sel;
  p.pool = pool;
  p.BQ = BQ;
  const size_t rows_bytes = (size_t)(2 * BQ) * sizeof(RsRow);
  p.rows = reinterpret_cast<RsRow*>(cur);
  cur += up(rows_bytes);
  p.gt = reinterpret_cast<int32_t*>(cur);
  cur += up((size_t)(2 * BQ) * RS_MAX_OUT * sizeof(int32_t));
  p.cand = reinterpret_cast<unsigned long long*>(cur);
  cudaError_t e = cudaMemsetAsync(p.rows, 0, rows_bytes, stream);
  if (e != cudaSuccess) return e;
  const int64_t scan_ctas = BQ * p.chunks;
  if (scan_ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
  // 16-byte loads when every row starts 16-byte aligned
  const bool vec = (max_n % 4) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15u) == 0;
  if (vec) {
    rs_hist_kernel<true><<<(unsigned)scan_ctas, RS_THREADS, 2 * RS_BINS * sizeof(uint32_t), stream>>>(p);
    rs_filter_kernel<true><<<(unsigned)scan_ctas, RS_THREADS, 0, stream>>>(p);
  } else {
    rs_hist_kernel<false><<<(unsigned)scan_ctas, RS_THREADS, 2 * RS_BINS * sizeof(uint32_t), stream>>>(p);
    rs_filter_kernel<false><<<(unsigned)scan_ctas, RS_THREADS, 0, stream>>>(p);
  }
  rs_resolve_kernel<<<dim3((unsigned)BQ, 2), SEL_THREADS, RS_RESOLVE_SMEM, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------ fixed-scratch variant
// csa2_block_topk_static keeps its block-maximum keys in this file-scope device
// array instead of a caller-provided workspace.  4 MiB = 2^20 keys, enough for
// B * Q * ceil(max_n / 8) <= 1,048,576 (for example 64 queries over 131,072
// entries).  Every GPU that loads the library holds the array until the process
// exits.
constexpr size_t STATIC_BLOCK_KEYS = (size_t)1 << 20;
__device__ __align__(256) uint32_t g_static_block_keys[STATIC_BLOCK_KEYS];

// Device address of the array for the current device, looked up once per device
// with that device current (host code may not use the symbol itself).
static uint32_t* static_block_keys(cudaError_t* err) {
  static std::mutex mu;
  static uint32_t* ptrs[128] = {nullptr};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 128) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_block_keys);
    if (*err != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

}  // namespace csa2

extern "C" csa2_status csa2_block_topk_static(const csa2_cache* cache, const float* scores, const int64_t* q_pos,
                                              int B, int Q, int64_t max_n, int M, int32_t* pool_blocks,
                                              void* stream) {
  using namespace csa2;
  if (!cache || !cache->main_kv || !cache->idx_codes || !cache->idx_scales || !cache->n_entries)
    return CSA2_ERR_INVALID_ARG;
  if (cache->cap < 0 || (cache->cap % BLK) != 0) return CSA2_ERR_INVALID_ARG;
  if (cache->m != 1 && cache->m != 2) return CSA2_ERR_UNSUPPORTED;
  if (B < 0 || Q < 0 || max_n < 0) return CSA2_ERR_INVALID_ARG;
  if (M < 1 || M > CSA2_MAX_M) return CSA2_ERR_UNSUPPORTED;
  if ((int64_t)B * Q > ((int64_t)1 << 26)) return CSA2_ERR_UNSUPPORTED;     // as every other call
  if ((uint64_t)B * (uint64_t)Q * (uint64_t)ceil_div(max_n, BLK) > STATIC_BLOCK_KEYS) return CSA2_ERR_WORKSPACE;
  if (B == 0 || Q == 0) return CSA2_OK;
  if (!scores || !q_pos || !pool_blocks) return CSA2_ERR_INVALID_ARG;
  cudaError_t err = cudaSuccess;
  uint32_t* keys = static_block_keys(&err);
  if (!keys) return CSA2_ERR_CUDA;
  // every key the selection reads is written first by the block-max pass, so the
  // array needs no clearing between calls
  return launch_block_topk(scores, q_pos, cache->n_entries, cache->m, B, Q, max_n, M, pool_blocks, keys,
                           (cudaStream_t)stream) == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}
