// (c) Joint sparse + SWA attention over the shared 512-d latent (K = V).
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §3.3.2 (the readout
// concatenates the SWA KV with the selected main-KV entries into one sparse
// attention), §3.3.2.1 (key = value = the compressed content vector; the output
// is a convex combination of them), §2.4.4 (the FP4 cache is dequantised to a
// more precise format before attention: FP4 saves storage, it does not feed
// the matrix multiply); "4. 层维度(下):CSA2 与每 token 890 字节" §4.5.
//
// Split-KV formulation: the key list of one query (K selected slots, then the
// 128 window positions) is cut into chunks of 64 keys; one CTA per (query,
// chunk) dequantises its keys to bf16 in shared memory (exact: E2M1 x E4M3
// has at most 6 significant bits), computes S = Q K^T and O = P V with bf16
// tensor-core MMAs (fp32 accumulate), and writes the chunk's un-normalised O,
// row max and row sum.  A second kernel merges the chunks (log-sum-exp) and
// rounds to bf16.
#include "params.cuh"

namespace csa2 {

constexpr int AT_THREADS = 256;
constexpr int AT_CHUNK = 64;              // keys per CTA
constexpr int AT_ROW = D + 8;             // padded smem row (bf16 elements)
constexpr int AT_PROW = AT_CHUNK + 8;
constexpr int AT_SMEM = 2 * H * AT_ROW * 2 + H * AT_PROW * 2 + 4 * H * 4 + AT_CHUNK * 4;


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src));
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
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

__global__ void __launch_bounds__(AT_THREADS, 1) attn_chunk_kernel(AttnParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = Qs + H * AT_ROW;
  uint16_t* Ps = Ks + AT_CHUNK * AT_ROW;
  float* red_max = reinterpret_cast<float*>(Ps + H * AT_PROW);   // [2][64]
  float* red_sum = red_max + 2 * H;                                // [2][64]
  int* kvalid = reinterpret_cast<int*>(red_sum + 2 * H);           // [64]

  const int chunk = blockIdx.x, bq = blockIdx.y;
  const int b = bq / p.Q;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t = p.q_pos[bq];

  // ---- Q -> smem (cp.async)
  const uint16_t* qg = p.q + (int64_t)bq * H * D;
  for (int i = tid; i < H * D / 8; i += AT_THREADS) {
    int r = i / (D / 8), c = i % (D / 8);
    cp_async16(Qs + r * AT_ROW + c * 8, qg + r * D + c * 8);
  }
  // ---- keys of this chunk: 4 threads per key, 128 channels each
  {
    const int s = tid >> 2, part = tid & 3;
    const int gs = chunk * AT_CHUNK + s;
    uint16_t* dst = Ks + s * AT_ROW + part * 128;
    bool valid = false;
    if (gs < p.K) {
      int32_t id = p.sel[(int64_t)bq * p.K + gs];
      if (id >= 0 && id < p.cap) {
        valid = true;
        const uint8_t* ent = p.main_kv + ((int64_t)b * p.cap + id) * MAIN_BYTES;
        uint2 sc = __ldg(reinterpret_cast<const uint2*>(ent + 256 + part * 8));
        uint32_t scw[2] = {sc.x, sc.y};
#pragma unroll
        for (int v = 0; v < 4; v++) {           // 4 x 16 code bytes = 32 channels each
          uint4 cw = __ldg(reinterpret_cast<const uint4*>(ent + part * 64) + v);
          uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
          uint32_t o[16];
#pragma unroll
          for (int q = 0; q < 4; q++) {          // 4 bytes -> 8 channels of group (v*2 + q/2)
            int grp = v * 2 + q / 2;
            float s_ = e4m3_value((scw[grp / 4] >> (8 * (grp % 4))) & 255u);
#pragma unroll
            for (int bb = 0; bb < 4; bb++) {
              uint32_t byte = (w4[q] >> (8 * bb)) & 255u;
              o[q * 4 + bb] = pack_bf16x2(e2m1_value(byte & 15u) * s_, e2m1_value(byte >> 4) * s_);
            }
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + v * 32);
#pragma unroll
          for (int q = 0; q < 4; q++) d4[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      } else if (id >= p.cap) {
        if (part == 0) report(p.hdr, CSA2_ERR_BOUNDS, id);
      }
    } else if (gs < p.K + WIN) {
      int64_t pos = t - (WIN - 1) + (gs - p.K);
      if (pos >= 0) {
        int64_t row = pos - p.swa_base[b];
        if (row >= 0 && row < p.S) {
          valid = true;
          const uint16_t* src = p.swa + ((int64_t)b * p.S + row) * D + part * 128;
#pragma unroll
          for (int v = 0; v < 16; v++) cp_async16(dst + v * 8, src + v * 8);
        } else if (part == 0) {
          report(p.hdr, CSA2_ERR_BOUNDS, pos);
        }
      }
    }
    if (!valid) {
#pragma unroll
      for (int v = 0; v < 16; v++) reinterpret_cast<uint4*>(dst)[v] = make_uint4(0, 0, 0, 0);
    }
    if (part == 0) kvalid[s] = valid;
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // ---- S = Q K^T : warp -> heads 16*(warp%4), keys 32*(warp/4)
  const int mh = warp & 3, kh = warp >> 2;
  float sacc[4][4];
#pragma unroll
  for (int j = 0; j < 4; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) sacc[j][e] = 0.f;
  {
    const uint16_t* a_base = Qs + (16 * mh + (lane & 15)) * AT_ROW + (lane >> 4) * 8;
    const int mi = lane >> 3;
    const uint16_t* b_base = Ks + (32 * kh + (mi >> 1) * 8 + (lane & 7)) * AT_ROW + (mi & 1) * 8;
#pragma unroll 4
    for (int ks = 0; ks < D / 16; ks++) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, a_base + ks * 16);
#pragma unroll
      for (int jp = 0; jp < 2; jp++) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, b_base + jp * 16 * AT_ROW + ks * 16);
        mma_bf16(sacc[2 * jp], a0, a1, a2, a3, b0, b1);
        mma_bf16(sacc[2 * jp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  // ---- softmax pieces (rows g and g+8 of this warp's 16 heads)
  const int g = lane >> 2;
  float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < 4; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) {
      int key = 32 * kh + 8 * j + 2 * (lane & 3) + (e & 1);
      float v = kvalid[key] ? sacc[j][e] * p.scale : -INFINITY;
      sacc[j][e] = v;
      rmax[e >> 1] = fmaxf(rmax[e >> 1], v);
    }
#pragma unroll
  for (int r = 0; r < 2; r++) {
    rmax[r] = fmaxf(rmax[r], __shfl_xor_sync(0xFFFFFFFFu, rmax[r], 1));
    rmax[r] = fmaxf(rmax[r], __shfl_xor_sync(0xFFFFFFFFu, rmax[r], 2));
  }
  if ((lane & 3) == 0) {
    red_max[kh * H + 16 * mh + g] = rmax[0];
    red_max[kh * H + 16 * mh + g + 8] = rmax[1];
  }
  __syncthreads();
  float mrow[2], rsum[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 2; r++) {
    int h = 16 * mh + g + 8 * r;
    float mm = fmaxf(red_max[h], red_max[H + h]);
    mrow[r] = (mm == -INFINITY) ? 0.f : mm;
  }
#pragma unroll
  for (int j = 0; j < 4; j++) {
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
      pv[e] = (sacc[j][e] == -INFINITY) ? 0.f : __expf(sacc[j][e] - mrow[e >> 1]);
      rsum[e >> 1] += pv[e];
    }
    int key = 32 * kh + 8 * j + 2 * (lane & 3);
    *reinterpret_cast<uint32_t*>(Ps + (16 * mh + g) * AT_PROW + key) = pack_bf16x2(pv[0], pv[1]);
    *reinterpret_cast<uint32_t*>(Ps + (16 * mh + g + 8) * AT_PROW + key) = pack_bf16x2(pv[2], pv[3]);
  }
#pragma unroll
  for (int r = 0; r < 2; r++) {
    rsum[r] += __shfl_xor_sync(0xFFFFFFFFu, rsum[r], 1);
    rsum[r] += __shfl_xor_sync(0xFFFFFFFFu, rsum[r], 2);
  }
  if ((lane & 3) == 0) {
    red_sum[kh * H + 16 * mh + g] = rsum[0];
    red_sum[kh * H + 16 * mh + g + 8] = rsum[1];
  }
  __syncthreads();
  const int64_t part_idx = (int64_t)bq * p.n_chunks + chunk;
  if (tid < H) {
    float mm = fmaxf(red_max[tid], red_max[H + tid]);
    p.mpart[part_idx * H + tid] = mm;
    p.lpart[part_idx * H + tid] = red_sum[tid] + red_sum[H + tid];
  }

  // ---- O = P V : warp -> heads 16*(warp%4), dims 256*(warp/4)
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
#pragma unroll
    for (int ks = 0; ks < AT_CHUNK / 16; ks++) {
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
  float* og = p.opart + part_idx * H * D;
#pragma unroll
  for (int j = 0; j < 32; j++) {
    int col = 256 * dh + 8 * j + 2 * (lane & 3);
    *reinterpret_cast<float2*>(og + (16 * mh + g) * D + col) = make_float2(oacc[j][0], oacc[j][1]);
    *reinterpret_cast<float2*>(og + (16 * mh + g + 8) * D + col) = make_float2(oacc[j][2], oacc[j][3]);
  }
}

// Merge the chunks of one (query, head): block of 128 threads, 4 dims each.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnParams p) {
  const int h = blockIdx.x % H;
  const int64_t bq = blockIdx.x / H;
  const int tid = threadIdx.x;
  float M = -INFINITY;
  for (int c = 0; c < p.n_chunks; c++) M = fmaxf(M, p.mpart[(bq * p.n_chunks + c) * H + h]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  for (int c = 0; c < p.n_chunks; c++) {
    int64_t pi = bq * p.n_chunks + c;
    float mc = p.mpart[pi * H + h];
    float w = (mc == -INFINITY) ? 0.f : __expf(mc - M);
    L += w * p.lpart[pi * H + h];
    float4 o = *reinterpret_cast<const float4*>(p.opart + (pi * H + h) * D + tid * 4);
    acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
  }
  float inv = (L > 0.f) ? 1.0f / L : 0.f;
  uint2 r = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  *reinterpret_cast<uint2*>(p.out + (bq * H + h) * D + tid * 4) = r;
}

int attn_chunks(int K) { return (int)ceil_div((int64_t)K + WIN, AT_CHUNK); }

size_t attn_partials_bytes(int64_t BQ, int K) {
  return (size_t)BQ * attn_chunks(K) * H * (D + 2) * sizeof(float);
}

cudaError_t launch_attention(AttnParams p, int B, float* partials, cudaStream_t stream) {
  int64_t BQ = (int64_t)B * p.Q;
  if (BQ == 0) return cudaSuccess;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  p.n_chunks = attn_chunks(p.K);
  p.opart = partials;
  p.mpart = partials + BQ * p.n_chunks * H * D;
  p.lpart = p.mpart + BQ * p.n_chunks * H;
  dim3 grid(p.n_chunks, (unsigned)BQ);
  attn_chunk_kernel<<<grid, AT_THREADS, AT_SMEM, stream>>>(p);
  attn_combine_kernel<<<(unsigned)(BQ * H), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
