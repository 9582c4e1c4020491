// Device-side helpers shared by the CSA2 kernels (product code only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

constexpr int D = CSA2_D_LATENT;          // 512
constexpr int D_ROPE = CSA2_D_ROPE;       // 64
constexpr int H = CSA2_N_HEADS;           // 64
constexpr int HI = CSA2_N_INDEX_HEADS;    // 32
constexpr int DI = CSA2_D_INDEX;          // 128
constexpr int BLK = CSA2_BLOCK;           // 8
constexpr int WIN = CSA2_WINDOW;          // 128
constexpr int MAIN_BYTES = CSA2_MAIN_ENTRY_BYTES;  // 288
constexpr int IDX_CODE_BYTES = CSA2_INDEX_CODE_BYTES;
constexpr int IDX_SCALE_BYTES = CSA2_INDEX_SCALE_BYTES;

// Workspace header: word 0 = magic, word 1 = status bits, words 2..3 = detail.
constexpr uint32_t WS_MAGIC = 0xC5A20001u;
struct WsHeader {
  uint32_t magic;
  uint32_t status;
  unsigned long long detail;
};

__device__ __forceinline__ void report(WsHeader* hdr, csa2_status code, long long detail) {
  // the first error wins; later ones are dropped
  if (atomicCAS(&hdr->status, 0u, (uint32_t)code) == 0u) {
    atomicExch(&hdr->detail, (unsigned long long)detail);
  }
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) {
  return __uint_as_float(h << 16);
}

// Visible entries of a query at raw position t: min(n_entries, floor((t+1)/m)).
__device__ __forceinline__ int64_t visible_entries(int64_t t, int m, int32_t n_entries) {
  int64_t v = (t + 1) / m;
  if (v < 0) v = 0;
  return v < (int64_t)n_entries ? v : (int64_t)n_entries;
}

// ---------------------------------------------------------------- FP4 / FP8
// E2M1 magnitudes of codes 0..7 (sign in bit 3).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  // 0, 0.5, 1, 1.5, 2, 3, 4, 6: exponent bits (code>>1)&3, mantissa code&1
  uint32_t e = (code >> 1) & 3u, m = code & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : __uint_as_float((e + 126u) << 23) * (1.0f + 0.5f * (float)m);
  return (code & 8u) ? -mag : mag;
}

// Two binary32 -> packed E2M1 byte (lo in bits 0..3), round to nearest even,
// saturating to +-6.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 b; cvt.rn.satfinite.e2m1x2.f32 b, %2, %1; cvt.u32.u8 %0, b; }"
      : "=r"(r) : "f"(lo), "f"(hi));
  return r & 0xFFu;
}

// binary32 -> E4M3 byte, round to nearest even, saturating to 448.
__device__ __forceinline__ uint32_t e4m3_byte(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return (uint32_t)r & 0xFFu;
}

// E4M3 byte -> binary32 (exact).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float mag = (e == 0) ? (float)m * 0.001953125f /* 2^-9 */
                       : __uint_as_float((e + 120u) << 23) * (1.0f + 0.125f * (float)m);
  return (b & 0x80u) ? -mag : mag;
}

// E8M0 byte -> 2^(b-127) as binary32 (b in 1..254 normal; 0 -> 2^-127 subnormal).
__device__ __forceinline__ float e8m0_value(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// Order-preserving map binary32 -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace csa2
