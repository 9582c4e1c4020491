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
};

__global__ void block_max_kernel(BlockMaxParams p) {
  const int bq = blockIdx.y;
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
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
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_DYN_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(block_topm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_DYN_SMEM);
  if (e == cudaSuccess) attr_dev = dev;
  return e;
}

cudaError_t launch_block_topk(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m,
                              int B, int Q, int64_t max_n, int M, int32_t* pool_blocks, uint32_t* gkeys,
                              cudaStream_t stream) {
  if (B == 0 || Q == 0) return cudaSuccess;
  const int64_t nb_max = ceil_div(max_n, BLK);
  if (nb_max > 0) {
    BlockMaxParams bp{scores, q_pos, n_entries, m, Q, max_n, nb_max, gkeys};
    dim3 grid((unsigned)ceil_div(nb_max, 256), B * Q);
    block_max_kernel<<<grid, 256, 0, stream>>>(bp);
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
