// (c) Joint sparse + SWA attention over the shared 512-d latent (K = V).
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §3.3.2 (the readout
// concatenates the SWA KV with the selected main-KV entries into one sparse
// attention), §3.3.2.1 (key = value = the compressed content vector; the output
// is a convex combination of them), §2.4.4 (the FP4 cache is dequantised to a
// more precise format before attention: FP4 saves storage, it does not feed
// the matrix multiply); "4. 层维度(下):CSA2 与每 token 890 字节" §4.5.
//
// One thread-block cluster of 8 CTAs per query token.  The query's key list (K
// selected slots, then the 128 window positions) is cut into 8 equal slices;
// CTA r of the cluster
//   1. receives Q (64 heads x 512, bf16) by bulk copies multicast to the whole
//      cluster (CTA r issues rows 8r..8r+7 for all 8 CTAs), bulk-copies its
//      slice's 288-byte FP4 entries and 1 KB window rows (one mbarrier, one
//      round trip), and dequantises the entries to bf16 in shared memory
//      through a byte -> bf16x2 table and an exact bf16x2 multiply by the
//      group scale (E2M1 x E4M3 has at most 6 significant bits),
//   2. computes S = Q K^T with bf16 tensor-core MMAs (fp32 accumulate),
//   3. exchanges per-head row maxima with the other 7 CTAs through distributed
//      shared memory, forms P = exp(S - max) and O_r = P V,
//   4. after a cluster barrier, owns output dims [64r, 64r+64): it sums that slice
//      of the 8 partial O's and the 8 partial row sums over DSMEM, normalises and
//      stores bf16.
// Nothing leaves the cluster except the final output.
#include <cooperative_groups.h>

#include "params.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

constexpr int AT_THREADS = 256;
constexpr int AT_CLUSTER = 8;
constexpr int AT_MAX_KPC = 80;              // keys per CTA at K = 512
constexpr int AT_ROW = D + 8;               // padded smem row (bf16 elements): conflict-free ldmatrix
constexpr int AT_PROW = AT_MAX_KPC + 8;
constexpr int AT_Q_BYTES = H * AT_ROW * 2;              // 66,560
constexpr int AT_K_BYTES = AT_MAX_KPC * AT_ROW * 2;     // 83,200
constexpr int AT_P_BYTES = H * AT_PROW * 2;             // 11,264
constexpr int AT_STG_BYTES = AT_MAX_KPC * MAIN_BYTES;   // 23,040: FP4 entries as loaded
constexpr int AT_RED_BYTES = 3 * H * 4 + AT_MAX_KPC * 4 + 256 * 4 + 16;
constexpr int AT_SMEM = AT_Q_BYTES + AT_K_BYTES + AT_P_BYTES + AT_STG_BYTES + AT_RED_BYTES;
static_assert(AT_Q_BYTES + AT_K_BYTES >= H * D * 4, "partial O must fit over Q and K");

using tc::smem_u32;

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// keys per CTA: the slot list split 8 ways, rounded up to a multiple of 16
__host__ __device__ __forceinline__ int attn_kpc(int K) {
  int per = (K + WIN + AT_CLUSTER - 1) / AT_CLUSTER;
  return (per + 15) / 16 * 16;
}

__global__ void __cluster_dims__(AT_CLUSTER, 1, 1) __launch_bounds__(AT_THREADS, 1)
attn_cluster_kernel(AttnParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem + AT_Q_BYTES);
  uint16_t* Ps = reinterpret_cast<uint16_t*>(smem + AT_Q_BYTES + AT_K_BYTES);
  uint8_t* stg = smem + AT_Q_BYTES + AT_K_BYTES + AT_P_BYTES;
  float* red = reinterpret_cast<float*>(stg + AT_STG_BYTES);
  float* loc_max = red;              // [64] this CTA's row maxima (read by the cluster)
  float* loc_sum = red + H;          // [64] this CTA's row sums   (read by the cluster)
  float* half_max = red + 2 * H;     // [64] per warp-half scratch
  int* kvalid = reinterpret_cast<int*>(red + 3 * H);              // [80] 0 none, 1 entry, 2 window row
  uint32_t* lut = reinterpret_cast<uint32_t*>(kvalid + AT_MAX_KPC); // [256] byte -> two bf16 E2M1 values
  uint64_t* bar = reinterpret_cast<uint64_t*>(lut + 256);
  float* Opart = reinterpret_cast<float*>(smem);   // [64][512] fp32, reuses Q and K after the MMAs

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int bq = blockIdx.x / AT_CLUSTER;
  const int b = bq / p.Q;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t = p.q_pos[bq];
  const int kpc = attn_kpc(p.K);
  const int slot0 = rank * kpc;

  if (tid == 0) {
    tc::bar_init(bar, 1);
    tc::bar_init_fence();
  }
  {
    const uint32_t c = (uint32_t)tid;           // tid < 256: one table entry per thread
    lut[c] = pack_bf16x2(e2m1_value(c & 15u), e2m1_value(c >> 4));
  }
  cluster.sync();                                              // #0: every CTA's barrier is initialised

  // ---- one warp issues every copy of this CTA; the others zero empty key rows
  if (warp == 0) {
    uint32_t bytes = 0;
    for (int s = lane; s < kpc; s += 32) {
      const int gs = slot0 + s;
      int kind = 0;
      if (gs < p.K) {
        const int32_t id = p.sel[(int64_t)bq * p.K + gs];
        if (id >= 0 && id < p.cap) {
          kind = 1;
          bytes += MAIN_BYTES;
        } else if (id >= p.cap) {
          report(p.hdr, CSA2_ERR_BOUNDS, id);
        }
      } else if (gs < p.K + WIN) {
        const int64_t pos = t - (WIN - 1) + (gs - p.K);
        if (pos >= 0) {
          const int64_t row = pos - p.swa_base[b];
          if (row >= 0 && row < p.S) {
            kind = 2;
            bytes += D * 2;
          } else {
            report(p.hdr, CSA2_ERR_BOUNDS, pos);
          }
        }
      }
      kvalid[s] = kind;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) bytes += __shfl_xor_sync(0xFFFFFFFFu, bytes, off);
    if (lane == 0) tc::bar_arrive_expect_tx(bar, (uint32_t)(H * D * 2) + bytes);
    __syncwarp();
    // Q rows 8*rank .. 8*rank+7, multicast to all 8 CTAs at the same smem offset
    if (lane < 8) {
      const int r = rank * 8 + lane;
      tc::bulk_load_multicast(Qs + r * AT_ROW, p.q + ((int64_t)bq * H + r) * D, D * 2, bar, 0xFFu);
    }
    for (int s = lane; s < kpc; s += 32) {
      const int gs = slot0 + s;
      if (kvalid[s] == 1) {
        const int32_t id = p.sel[(int64_t)bq * p.K + gs];
        tc::bulk_load(stg + s * MAIN_BYTES, p.main_kv + ((int64_t)b * p.cap + id) * MAIN_BYTES, MAIN_BYTES, bar);
      } else if (kvalid[s] == 2) {
        const int64_t row = t - (WIN - 1) + (gs - p.K) - p.swa_base[b];
        tc::bulk_load(Ks + s * AT_ROW, p.swa + ((int64_t)b * p.S + row) * D, D * 2, bar);
      }
    }
  }
  __syncthreads();                                             // kvalid visible
  for (int idx = tid; idx < kpc * 64; idx += AT_THREADS) {    // zero rows of empty slots
    const int s = idx >> 6;
    if (kvalid[s] == 0) reinterpret_cast<uint4*>(Ks + s * AT_ROW)[idx & 63] = make_uint4(0, 0, 0, 0);
  }
  bool ok = tc::bar_wait(bar, 0);
  if (!ok) report(p.hdr, CSA2_ERR_TIMEOUT, 2);
  // ---- dequantise the FP4 entries: 8 code bytes = 16 channels = one E4M3 scale group
  for (int idx = tid; idx < kpc * 32; idx += AT_THREADS) {
    const int s = idx >> 5, grp = idx & 31;
    if (kvalid[s] != 1) continue;
    const uint8_t* ent = stg + s * MAIN_BYTES;
    const uint2 cb = *reinterpret_cast<const uint2*>(ent + grp * 8);
    const float sc = e4m3_value(ent[256 + grp]);
    const uint32_t sc2 = pack_bf16x2(sc, sc);
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const uint32_t byte = ((k < 4 ? cb.x : cb.y) >> (8 * (k & 3))) & 255u;
      const uint32_t v = lut[byte];
      asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[k]) : "r"(v), "r"(sc2));
    }
    uint4* d4 = reinterpret_cast<uint4*>(Ks + s * AT_ROW + grp * 16);
    d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  __syncthreads();

  // ---- S = Q K^T : warp -> heads 16*(warp%4), key half warp/4 (NTH n8-tiles)
  const int mh = warp & 3, kh = warp >> 2;
  const int nth = kpc / 16;                 // n8 tiles per half
  const int g = lane >> 2;
  float sacc[5][4];
#pragma unroll
  for (int j = 0; j < 5; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) sacc[j][e] = 0.f;
  {
    const uint16_t* a_base = Qs + (16 * mh + (lane & 15)) * AT_ROW + (lane >> 4) * 8;
    const uint16_t* b_base = Ks + (kh * nth * 8 + (lane & 7)) * AT_ROW + ((lane >> 3) & 1) * 8;
#pragma unroll 2
    for (int ks = 0; ks < D / 16; ks++) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, a_base + ks * 16);
#pragma unroll
      for (int j = 0; j < 5; j++) {
        if (j < nth) {
          uint32_t b0, b1;
          ldsm_x2(b0, b1, b_base + j * 8 * AT_ROW + ks * 16);
          mma_bf16(sacc[j], a0, a1, a2, a3, b0, b1);
        }
      }
    }
  }
  // ---- row maxima over this CTA's keys, exchanged across the cluster
  float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < 5; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int key = kh * nth * 8 + 8 * j + 2 * (lane & 3) + (e & 1);
      const float v = (j < nth && kvalid[key] != 0) ? sacc[j][e] * p.scale : -INFINITY;
      sacc[j][e] = v;
      rmax[e >> 1] = fmaxf(rmax[e >> 1], v);
    }
#pragma unroll
  for (int r = 0; r < 2; r++) {
    rmax[r] = fmaxf(rmax[r], __shfl_xor_sync(0xFFFFFFFFu, rmax[r], 1));
    rmax[r] = fmaxf(rmax[r], __shfl_xor_sync(0xFFFFFFFFu, rmax[r], 2));
  }
  if (kh == 1 && (lane & 3) == 0) {
    half_max[16 * mh + g] = rmax[0];
    half_max[16 * mh + g + 8] = rmax[1];
  }
  __syncthreads();
  if (kh == 0 && (lane & 3) == 0) {
    loc_max[16 * mh + g] = fmaxf(rmax[0], half_max[16 * mh + g]);
    loc_max[16 * mh + g + 8] = fmaxf(rmax[1], half_max[16 * mh + g + 8]);
  }
  cluster.sync();                                              // #1: maxima visible
  float gmax[2];
#pragma unroll
  for (int r = 0; r < 2; r++) {
    const int h = 16 * mh + g + 8 * r;
    float mm = -INFINITY;
#pragma unroll
    for (int c = 0; c < AT_CLUSTER; c++) mm = fmaxf(mm, cluster.map_shared_rank(loc_max, c)[h]);
    gmax[r] = (mm == -INFINITY) ? 0.f : mm;
  }
  // ---- P = exp(S - max) (bf16) and this CTA's row sums
  float rsum[2] = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 5; j++) {
    if (j < nth) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        pv[e] = (sacc[j][e] == -INFINITY) ? 0.f : __expf(sacc[j][e] - gmax[e >> 1]);
        rsum[e >> 1] += pv[e];
      }
      const int key = kh * nth * 8 + 8 * j + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(Ps + (16 * mh + g) * AT_PROW + key) = pack_bf16x2(pv[0], pv[1]);
      *reinterpret_cast<uint32_t*>(Ps + (16 * mh + g + 8) * AT_PROW + key) = pack_bf16x2(pv[2], pv[3]);
    }
  }
#pragma unroll
  for (int r = 0; r < 2; r++) {
    rsum[r] += __shfl_xor_sync(0xFFFFFFFFu, rsum[r], 1);
    rsum[r] += __shfl_xor_sync(0xFFFFFFFFu, rsum[r], 2);
  }
  if (kh == 1 && (lane & 3) == 0) {
    half_max[16 * mh + g] = rsum[0];            // reuse as half-sum scratch
    half_max[16 * mh + g + 8] = rsum[1];
  }
  __syncthreads();
  if (kh == 0 && (lane & 3) == 0) {
    loc_sum[16 * mh + g] = rsum[0] + half_max[16 * mh + g];
    loc_sum[16 * mh + g + 8] = rsum[1] + half_max[16 * mh + g + 8];
  }

  // ---- O_r = P V : warp -> heads 16*(warp%4), dims 256*(warp/4)
  const int dh = warp >> 2;
  float oacc[32][4];
#pragma unroll
  for (int j = 0; j < 32; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) oacc[j][e] = 0.f;
  {
    const uint16_t* a_base = Ps + (16 * mh + (lane & 15)) * AT_PROW + (lane >> 4) * 8;
    const int mi = lane >> 3;
    const uint16_t* b_base = Ks + ((mi & 1) * 8 + (lane & 7)) * AT_ROW + 256 * dh + (mi >> 1) * 8;
    for (int ks = 0; ks < kpc / 16; ks++) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, a_base + ks * 16);
#pragma unroll
      for (int jp = 0; jp < 16; jp++) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, b_base + ks * 16 * AT_ROW + jp * 16);
        mma_bf16(oacc[2 * jp], a0, a1, a2, a3, b0, b1);
        mma_bf16(oacc[2 * jp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  __syncthreads();                                           // all reads of Q and K done
#pragma unroll
  for (int j = 0; j < 32; j++) {
    const int col = 256 * dh + 8 * j + 2 * (lane & 3);
    *reinterpret_cast<float2*>(Opart + (16 * mh + g) * D + col) = make_float2(oacc[j][0], oacc[j][1]);
    *reinterpret_cast<float2*>(Opart + (16 * mh + g + 8) * D + col) = make_float2(oacc[j][2], oacc[j][3]);
  }
  cluster.sync();                                              // #2: partial O and sums visible

  // ---- reduce this CTA's 64-dim slice over the cluster, normalise, store bf16
  uint16_t* out = p.out + (int64_t)bq * H * D;
  for (int idx = tid; idx < H * 16; idx += AT_THREADS) {
    const int h = idx >> 4, d4 = idx & 15;
    const int col = rank * 64 + d4 * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < AT_CLUSTER; c++) {
      const float* rem = cluster.map_shared_rank(Opart, c);
      const float4 v = *reinterpret_cast<const float4*>(rem + h * D + col);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      L += cluster.map_shared_rank(loc_sum, c)[h];
    }
    const float inv = (L > 0.f) ? 1.0f / L : 0.f;
    *reinterpret_cast<uint2*>(out + h * D + col) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  }
  cluster.sync();                                              // #3: remote reads finished
}

size_t attn_partials_bytes(int64_t, int) { return 0; }

cudaError_t launch_attention(AttnParams p, int B, float*, cudaStream_t stream) {
  const int64_t BQ = (int64_t)B * p.Q;
  if (BQ == 0) return cudaSuccess;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  attn_cluster_kernel<<<(unsigned)(BQ * AT_CLUSTER), AT_THREADS, AT_SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
