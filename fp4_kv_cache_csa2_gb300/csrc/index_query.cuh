// MXFP4 quantisation of one query's 32 indexer heads, the B operand of the
// block-scaled indexer MMA.  Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到
// 极致" §2.4.4 (FP4 indexer Q and K share one format); "4. 层维度(下):CSA2 与每
// token 890 字节" §4.4 (OCP MXFP4: E2M1 elements, one E8M0 scale per 32).
#pragma once

#include "common.cuh"

namespace csa2 {

// One warp, lane = head: the 128 bf16 values of head `lane` (q_heads + lane *
// 128) become 64 bytes of E2M1 codes in row `lane` of `qcodes` (SW64 K-major:
// 32 rows x 64 bytes, 16-byte unit k of row r at unit k ^ ((r >> 1) & 3)) and
// four E8M0 bytes (one per 32 values, lowest byte first) in sfb[lane].  The
// scale of a block is 2^(floor(log2 amax) - 2), clamped to the E8M0 range; an
// all-zero block gets scale byte 0 and zero codes.
// Block kb of the head (32 values in four 16-byte words u) -> its codes in
// qcodes and its scale byte, returned.
__device__ __forceinline__ uint32_t quantize_index_block(const uint4* u, int kb, int lane, uint8_t* qcodes) {
  float v[32];
#pragma unroll
  for (int c = 0; c < 4; c++) {
    const uint32_t w4[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
    for (int e = 0; e < 4; e++) {
      v[c * 8 + 2 * e] = bf16_bits_to_f32(w4[e] & 0xFFFFu);
      v[c * 8 + 2 * e + 1] = bf16_bits_to_f32(w4[e] >> 16);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(v[i]));
  uint32_t sb = 0, packed[4] = {0u, 0u, 0u, 0u};
  if (amax != 0.0f) {
    int X = (int)((__float_as_uint(amax) >> 23) & 255u) - 127 - 2;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    sb = (uint32_t)(X + 127);
    const float inv = __uint_as_float((uint32_t)(127 - X) << 23);
#pragma unroll
    for (int k = 0; k < 16; k++)
      packed[k / 4] |= e2m1x2(__fmul_rn(v[2 * k], inv), __fmul_rn(v[2 * k + 1], inv)) << (8 * (k % 4));
  }
  const int phys = lane * 64 + ((kb ^ ((lane >> 1) & 3)) * 16);        // SW64 swizzle of row `lane`
  *reinterpret_cast<uint4*>(qcodes + phys) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  return sb;
}

// The four blocks one after the other (16 live words of input at a time).
__device__ __forceinline__ void quantize_index_query_warp(const uint16_t* q_heads, uint8_t* qcodes, uint32_t* sfb) {
  const int lane = threadIdx.x & 31;
  const uint4* qh = reinterpret_cast<const uint4*>(q_heads + lane * DI);
  uint32_t sfw = 0;
#pragma unroll 1
  for (int kb = 0; kb < 4; kb++) {
    uint4 u[4];
#pragma unroll
    for (int c = 0; c < 4; c++) u[c] = __ldg(qh + 4 * kb + c);
    sfw |= quantize_index_block(u, kb, lane, qcodes) << (8 * kb);
  }
  sfb[lane] = sfw;
}

// All 16 loads of the head issued before the first block is quantised: one
// memory latency instead of four, for 64 more live registers.
__device__ __forceinline__ void quantize_index_query_warp_loads_first(const uint16_t* q_heads, uint8_t* qcodes,
                                                                      uint32_t* sfb) {
  const int lane = threadIdx.x & 31;
  const uint4* qh = reinterpret_cast<const uint4*>(q_heads + lane * DI);
  uint4 u[16];
#pragma unroll
  for (int i = 0; i < 16; i++) u[i] = __ldg(qh + i);
  uint32_t sfw = 0;
#pragma unroll
  for (int kb = 0; kb < 4; kb++) sfw |= quantize_index_block(u + 4 * kb, kb, lane, qcodes) << (8 * kb);
  sfb[lane] = sfw;
}

// Head weights of one query as 16 packed (even head, odd head) pairs.
__device__ __forceinline__ void pack_head_weights(const float* w, unsigned long long* w2) {
#pragma unroll
  for (int i = 0; i < HI / 2; i++)
    asm("mov.b64 %0, {%1, %2};" : "=l"(w2[i]) : "f"(w[2 * i]), "f"(w[2 * i + 1]));
}

// s = sum_h w_h * max(v_h, 0) over the 32 head dot products of one entry, as
// two binary32 chains (even heads and odd heads, each in head order, each term
// one fused multiply-add) added at the end.  Every indexer kernel uses this
// one order, so an entry's score does not depend on which kernel computed it.
__device__ __forceinline__ float index_head_sum(const float* v, const unsigned long long* w2) {
  unsigned long long acc;
  asm("mov.b64 %0, 0;" : "=l"(acc));
#pragma unroll
  for (int i = 0; i < HI / 2; i++) {
    unsigned long long x;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(fmaxf(v[2 * i], 0.0f)), "f"(fmaxf(v[2 * i + 1], 0.0f)));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(x), "l"(w2[i]));
  }
  float even, odd;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(even), "=f"(odd) : "l"(acc));
  return __fadd_rn(even, odd);
}

}  // namespace csa2
