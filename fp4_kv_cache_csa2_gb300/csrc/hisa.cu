// HISA variant of the indexer's first stage: per-block summary keys and the
// mapping that lets the indexer scan and top-K select run over them.
//
// Source: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.4, the HISA
// paragraph: each block of consecutive positions keeps the mean of its indexer
// keys; a query first scores those block means and keeps the best blocks, then
// scores the entries of the kept blocks only.  A decode step changes only the
// newest block, so only its summary is recomputed.
//
// Summary of block r of sequence b (entries [8r, min(8r + 8, n))), in binary32
// with a fixed order so that the bytes are reproducible:
//   k_p      dequantised index key of entry 8r + p (E2M1 value x 2^(s - 127):
//            exact in binary32)
//   acc      +0, then acc = acc + k_p for p = 0, 1, ... in entry order
//   mean     acc / count, correctly rounded (count = entries in the block)
//   stored   MXFP4 of the mean by the index-K rule: per 32 dims
//            X = floor(log2 amax) - 2 clamped to [-127, 127], code =
//            E2M1(v * 2^-X) (nearest even, saturating), amax == 0 -> scale
//            byte 0 and +0 codes.
//
// Layout: one warp per block; lane l owns dims 4l..4l+3 (code bytes 2l, 2l+1,
// MX group l / 8), so a 32-dim group is 8 neighbouring lanes and its amax is
// three xor shuffles.  The kernel is a small gather (8 x 68 B read, 68 B
// written per block); a decode step runs it on one block per sequence.
#include "params.cuh"

namespace csa2 {

constexpr int HS_WARPS = 8;

__global__ void __launch_bounds__(HS_WARPS * 32) block_summary_kernel(HsParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * HS_WARPS + (threadIdx.x >> 5);   // (b, i)
  if (item >= (int64_t)p.B * p.n_blocks) return;
  const int b = (int)(item / p.n_blocks);
  const int64_t r = p.first_block[b] + item % p.n_blocks;
  int64_t n = p.n_entries[b];
  if (n > p.cap) {
    if (lane == 0 && item % p.n_blocks == 0) report(p.hdr, CSA2_ERR_BOUNDS, n);
    n = p.cap;
  }
  if (r < 0 || r * BLK >= n) return;              // no visible entry: not written
  if (r >= p.sum_cap) {
    if (lane == 0) report(p.hdr, CSA2_ERR_BOUNDS, r);
    return;
  }
  const int64_t e0 = r * BLK;
  const int cnt = (int)(n - e0 < BLK ? n - e0 : BLK);
  const uint8_t* codes = p.idx_codes + ((int64_t)b * p.cap + e0) * IDX_CODE_BYTES + 2 * lane;
  const uint8_t* scales = p.idx_scales + ((int64_t)b * p.cap + e0) * IDX_SCALE_BYTES + (lane >> 3);
  uint32_t c16[BLK], sb[BLK];
#pragma unroll
  for (int q = 0; q < BLK; q++) {                 // all loads first
    c16[q] = q < cnt ? (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(codes + q * IDX_CODE_BYTES)) : 0u;
    sb[q] = q < cnt ? (uint32_t)__ldg(scales + q * IDX_SCALE_BYTES) : 0u;
  }
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < BLK; q++) {
    if (q >= cnt) break;
    const float s = e8m0_value(sb[q]);
#pragma unroll
    for (int d = 0; d < 4; d++) acc[d] = __fadd_rn(acc[d], __fmul_rn(e2m1_value((c16[q] >> (4 * d)) & 15u), s));
  }
  const float fc = (float)cnt;
  float mean[4];
#pragma unroll
  for (int d = 0; d < 4; d++) mean[d] = __fdiv_rn(acc[d], fc);
  float amax = fmaxf(fmaxf(fabsf(mean[0]), fabsf(mean[1])), fmaxf(fabsf(mean[2]), fabsf(mean[3])));
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  uint32_t scale_byte = 0, out = 0;
  if (amax != 0.0f) {
    int X;
    const uint32_t eb = (__float_as_uint(amax) >> 23) & 255u;
    if (eb != 0) {
      X = (int)eb - 127 - 2;                      // floor(log2 amax) - 2 for normals
    } else {
      X = -127;                                   // subnormal amax: floor(log2) <= -127
    }
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    scale_byte = (uint32_t)(X + 127);
    const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2^-X, exact
    out = e2m1x2(__fmul_rn(mean[0], inv), __fmul_rn(mean[1], inv)) |
          (e2m1x2(__fmul_rn(mean[2], inv), __fmul_rn(mean[3], inv)) << 8);
  }
  const int64_t row = (int64_t)b * p.sum_cap + r;
  *reinterpret_cast<uint16_t*>(p.sum_codes + row * IDX_CODE_BYTES + 2 * lane) = (uint16_t)out;
  if ((lane & 7) == 0) p.sum_scales[row * IDX_SCALE_BYTES + (lane >> 3)] = (uint8_t)scale_byte;
}

// Per query: the summary rows it may see, written as the raw position of an
// m = 1 cache whose visible count is ceil(nv / 8); per sequence: the number of
// summary rows that exist, ceil(min(n_entries, cap) / 8).
__global__ void hisa_view_kernel(HvParams p) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < (int64_t)p.B * p.Q) {
    const int b = (int)(i / p.Q);
    int64_t nv = visible_entries(p.q_pos[i], p.m, p.n_entries[b]);
    if (nv > p.max_n) nv = p.max_n;
    if (nv > p.cap) nv = p.cap;
    p.view_pos[i] = ceil_div(nv, BLK) - 1;
  }
  if (i < p.B) {
    int64_t n = p.n_entries[i];
    if (n > p.cap) n = p.cap;
    if (n < 0) n = 0;
    p.view_n[i] = (int32_t)ceil_div(n, BLK);
  }
}

cudaError_t launch_block_summary(const HsParams& p, cudaStream_t stream) {
  const int64_t items = (int64_t)p.B * p.n_blocks;
  if (items == 0) return cudaSuccess;
  const int64_t grid = ceil_div(items, HS_WARPS);
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  block_summary_kernel<<<(unsigned)grid, HS_WARPS * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_hisa_view(const HvParams& p, cudaStream_t stream) {
  const int64_t n = (int64_t)p.B * p.Q > p.B ? (int64_t)p.B * p.Q : p.B;
  if (n == 0) return cudaSuccess;
  hisa_view_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
