// (b) Lightning-indexer scores  s(t,j) = sum_h w_h * ReLU(q_h . k_j)
// over 32 index heads x 128 dims, with MXFP4 queries and keys.
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4 (the Full layer
// scores every causally visible main-KV position; Reindex layers score only the
// candidate pool), §2.4.4 (FP4 indexer Q and K); "4. 层维度(下):CSA2 与每 token
// 890 字节" §4.4 (index K is OCP MXFP4: E2M1 + one E8M0 scale per 32).
//
// This is the CUDA-core formulation: one thread scores one entry at a time,
// the dequantised query (32 x 128 binary32) sits in shared memory and is read
// by broadcast.  Each CTA owns one query and a slice of its entries.
#include "params.cuh"

namespace csa2 {

constexpr int IS_THREADS = 256;


// Quantise one query (32 heads x 128 dims, bf16) to MXFP4 and store the exact
// dequantised values in smem.  Warp w handles heads w, w+8, ...; lane owns 4 dims.
__device__ __forceinline__ void load_query_mxfp4(const uint16_t* q, float* qs, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  for (int h = warp; h < HI; h += IS_THREADS / 32) {
    uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + h * DI) + lane);
    float v[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xFFFFu), bf16_bits_to_f32(raw.y >> 16)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    float out[4] = {0.f, 0.f, 0.f, 0.f};
    if (amax != 0.0f) {
      int X = (int)((__float_as_uint(amax) >> 23) & 255u) - 127 - 2;
      if (X < -127) X = -127;
      if (X > 127) X = 127;
      float inv = __uint_as_float((uint32_t)(127 - X) << 23);
      float sc = e8m0_value((uint32_t)(X + 127));
      uint32_t lo = e2m1x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv));
      uint32_t hi = e2m1x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
      out[0] = e2m1_value(lo & 15u) * sc;
      out[1] = e2m1_value(lo >> 4) * sc;
      out[2] = e2m1_value(hi & 15u) * sc;
      out[3] = e2m1_value(hi >> 4) * sc;
    }
    *reinterpret_cast<float4*>(qs + h * DI + lane * 4) = make_float4(out[0], out[1], out[2], out[3]);
  }
}

// Score of one entry against the query held in smem.
__device__ __forceinline__ float score_entry(const uint8_t* codes, const uint8_t* scales,
                                             const float* qs, const float* ws) {
  float dot[HI];
#pragma unroll
  for (int h = 0; h < HI; h++) dot[h] = 0.0f;
  uint32_t sc4 = __ldg(reinterpret_cast<const uint32_t*>(scales));
#pragma unroll 1
  for (int blk = 0; blk < 4; blk++) {
    uint4 c = __ldg(reinterpret_cast<const uint4*>(codes) + blk);
    float s = e8m0_value((sc4 >> (8 * blk)) & 255u);
    uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float k[32];
#pragma unroll
    for (int i = 0; i < 32; i++) k[i] = e2m1_value((cw[i / 8] >> (4 * (i % 8))) & 15u) * s;
#pragma unroll
    for (int h = 0; h < HI; h++) {
      const float4* qh = reinterpret_cast<const float4*>(qs + h * DI + blk * 32);
      float acc = dot[h];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        float4 qv = qh[i];
        acc = fmaf(qv.x, k[4 * i], acc);
        acc = fmaf(qv.y, k[4 * i + 1], acc);
        acc = fmaf(qv.z, k[4 * i + 2], acc);
        acc = fmaf(qv.w, k[4 * i + 3], acc);
      }
      dot[h] = acc;
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < HI; h++) s = fmaf(ws[h], fmaxf(dot[h], 0.0f), s);
  return s;
}

__global__ void __launch_bounds__(IS_THREADS) index_score_kernel(IsParams p) {
  __shared__ __align__(16) float qs[HI * DI];
  __shared__ float ws[HI];
  const int bq = blockIdx.y;
  const int b = bq / p.Q;
  const int tid = threadIdx.x;
  load_query_mxfp4(p.q_idx + (int64_t)bq * HI * DI, qs, tid);
  if (tid < HI) ws[tid] = p.w_head[(int64_t)bq * HI + tid];
  __syncthreads();

  const int64_t nv = visible_entries(p.q_pos[bq], p.m, p.n_entries[b]);
  const uint8_t* codes = p.idx_codes + (int64_t)b * p.cap * IDX_CODE_BYTES;
  const uint8_t* scales = p.idx_scales + (int64_t)b * p.cap * IDX_SCALE_BYTES;
  if (nv > p.cap) {
    if (tid == 0) report(p.hdr, CSA2_ERR_BOUNDS, nv);
    return;
  }

  if (p.pool == nullptr) {
    if (nv > p.max_n) {           // the score row is too short for the visible entries
      if (tid == 0 && blockIdx.x == 0) report(p.hdr, CSA2_ERR_BOUNDS, nv);
    }
    const int64_t j0 = (int64_t)blockIdx.x * p.entries_per_cta;
    int64_t j1 = j0 + p.entries_per_cta;
    if (j1 > nv) j1 = nv;
    if (j1 > p.max_n) j1 = p.max_n;
    float* out = p.scores + (int64_t)bq * p.max_n;
    for (int64_t j = j0 + tid; j < j1; j += IS_THREADS)
      out[j] = score_entry(codes + j * IDX_CODE_BYTES, scales + j * IDX_SCALE_BYTES, qs, ws);
  } else {
    // pool mode: CTA x handles pool slots [x*epc, (x+1)*epc) * 8 entries
    const int32_t* blocks = p.pool + (int64_t)bq * p.M;
    const int64_t s0 = (int64_t)blockIdx.x * p.entries_per_cta * BLK;
    int64_t s1 = s0 + p.entries_per_cta * BLK;
    if (s1 > (int64_t)p.M * BLK) s1 = (int64_t)p.M * BLK;
    float* out = p.scores + (int64_t)bq * p.M * BLK;
    for (int64_t s = s0 + tid; s < s1; s += IS_THREADS) {
      int32_t blk = blocks[s / BLK];
      int64_t j = (int64_t)blk * BLK + (s % BLK);
      float v = -INFINITY;
      if (blk >= 0) {
        if ((int64_t)blk * BLK >= p.cap) {
          report(p.hdr, CSA2_ERR_BOUNDS, blk);
        } else if (j < nv) {
          v = score_entry(codes + j * IDX_CODE_BYTES, scales + j * IDX_SCALE_BYTES, qs, ws);
        }
      }
      out[s] = v;
    }
  }
}

cudaError_t launch_index_score(IsParams p, cudaStream_t stream) {
  if (p.B == 0 || p.Q == 0) return cudaSuccess;
  int gx;
  if (p.pool == nullptr) {
    // slice so that a query's entries spread over enough CTAs to fill the GPU
    int64_t per = 2048;
    gx = (int)ceil_div(p.max_n, per);
    if (gx < 1) gx = 1;
    p.entries_per_cta = per;
  } else {
    int64_t per_blocks = 256;   // 2048 entries per CTA
    gx = (int)ceil_div(p.M, per_blocks);
    p.entries_per_cta = per_blocks;
  }
  dim3 grid(gx, p.B * p.Q);
  index_score_kernel<<<grid, IS_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
