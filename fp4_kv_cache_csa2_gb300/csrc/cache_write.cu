// (a) CSA2 cache write: compressor -> RMSNorm -> RoPE -> FP4 main KV, and the
// 512->128 index-K projection -> MXFP4.
//
// Sources: "4. 层维度(下):CSA2 与每 token 890 字节" §4.2 (compressor
// c_j = (w0 x_{2j-1} + w1 x_{2j}) / (w0 + w1) per channel), §4.4 (288 B main
// entry = 256 B E2M1 + 32 B E4M3 scales; 68 B index entry = 64 B E2M1 + 4 B
// E8M0); "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §2.3.1 (index K is a
// projection of the main KV entry), §2.4.4 (RMSNorm, then RoPE, then FP4 with
// one E4M3 scale per 16 channels and no global scale).
//
// Every binary32 operation that feeds a quantised byte is an explicit
// round-to-nearest intrinsic in a fixed order, so the bytes are reproducible on
// any IEEE machine that follows the same order:
//   compress   c = fma(w0, x0, w1*x1) / (w0 + w1)
//   RMSNorm    lane i owns channels 16i..16i+15: p_i = fma-chain of c^2 in
//              channel order; butterfly sum over lanes (xor 16,8,4,2,1);
//              r = 1/sqrt(ss/512 + 1e-6); y = c*r
//   RoPE       pairs (448+2i, 449+2i): y0' = fma(y0,cos,-(y1*sin)),
//              y1' = fma(y0,sin,y1*cos)
//   main FP4   per 16: s = E4M3(amax/6), code = E2M1(y/s); s == 0 -> codes +0
//   index K    k[o] = fma chain over channels 0..511 of y'[ch]*W[o][ch] from 0
//   MXFP4      per 32: X = floor(log2 amax) - 2 clamped to [-127,127];
//              code = E2M1(k * 2^-X); amax == 0 -> scale byte 0, codes +0
//
// Structure (persistent kernel, one CTA per SM, 512 threads in two roles that
// hand each 32-entry tile over through named barriers; setmaxnreg gives the
// entry pipeline 168 registers a thread and the projection 88):
//   smem  W^T as bf16 [512 ch][128 o] (128 KB, loaded once per CTA)
//         y tile   fp32 [32 entries][512 ch] (64 KB)
//   phase 1  (warps 8..15, one tile ahead) warp per entry, 4 entries per
//            warp: the 128-bit loads of all
//            four entries' token rows are issued first, then each entry is
//            compressed/normalised/rotated in registers, its 288-byte main
//            entry written and y' staged in smem (16-byte stores, no bank
//            conflicts); the next tile's token rows are prefetched into L2.
//   phase 2  (warps 0..7) each thread owns 4 outputs x 4 entries (16 independent fma
//            chains), four channels at a time; W^T row reads are contiguous
//            across the warp, y reads are broadcasts.  This phase is
//            FP32-ALU bound (65,536 fma per entry).
//   phase 3  MXFP4 of k: 8 lanes form one 32-wide block.
#include "host_once.cuh"
#include "params.cuh"

namespace csa2 {

constexpr int CW_THREADS = 512;                   // warps 0..7 projection, 8..15 entry pipeline
constexpr int CW_MATH_THREADS = 256;
constexpr int CW_LOAD_WARPS = 8;
constexpr int CW_TILE = 32;                       // entries per tile
constexpr int CW_MATH_REGS = 88;                  // setmaxnreg split of the 128 x 512 registers:
constexpr int CW_LOAD_REGS = 168;                 // 256 x 88 + 256 x 168 = 65,536
static_assert(CW_MATH_THREADS * CW_MATH_REGS + (CW_THREADS - CW_MATH_THREADS) * CW_LOAD_REGS <= 65536,
              "register split");
constexpr int CW_SMEM = D * DI * 2 + CW_TILE * D * 4;  // 131072 + 65536


__global__ void __launch_bounds__(CW_THREADS, 1) cache_write_kernel(CwParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* wt = reinterpret_cast<uint16_t*>(smem);                  // [512][128]
  float* ytile = reinterpret_cast<float*>(smem + D * DI * 2);        // [512][32]
  __shared__ int tile_valid[2][CW_TILE];           // by tile parity

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // W [128][512] -> W^T [512][128] in smem (once per CTA)
  for (int i = tid; i < DI * D / 2; i += CW_THREADS) {
    int o = i / (D / 2), ch2 = (i % (D / 2)) * 2;
    uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p.w_idx) + i);
    wt[(ch2 + 0) * DI + o] = (uint16_t)(v & 0xFFFFu);
    wt[(ch2 + 1) * DI + o] = (uint16_t)(v >> 16);
  }

  const int64_t n_local = p.T / p.m;                   // entries per sequence
  const int64_t tiles_per_seq = ceil_div(n_local, CW_TILE);
  const int64_t n_tiles = tiles_per_seq * p.B;
  __syncthreads();                                     // W^T ready

  // Two roles over the same tile sequence, handing the y tile over with named
  // barriers: FULL (1) when the entry pipeline has stored a tile's y', EMPTY (2)
  // when the projection has finished reading it.  The entry pipeline computes
  // tile i+1 in registers while the projection runs on tile i.
  if (warp >= CW_MATH_THREADS / 32) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(CW_LOAD_REGS));
    const int lwarp = warp - CW_MATH_THREADS / 32;
  for (int64_t tile = blockIdx.x, it = 0; tile < n_tiles; tile += gridDim.x, it++) {
    const int b = (int)(tile / tiles_per_seq);
    const int64_t j0 = (tile % tiles_per_seq) * CW_TILE;
    const int64_t e0 = p.entry_start[b];

    // ---------------- phase 1: warp per entry, loads of all four entries first
    constexpr int EPW = CW_TILE / CW_LOAD_WARPS;                  // entries per warp
    uint4 xr[EPW][4];                                             // rows x_{2j}, x_{2j+1} (m = 2) or x_j
    bool ok[EPW];
#pragma unroll
    for (int u = 0; u < EPW; u++) {
      const int t = lwarp + u * CW_LOAD_WARPS;
      const int64_t j = j0 + t;
      const int64_t e = e0 + j;
      bool valid = j < n_local;
      if (valid && (e < 0 || e >= p.cap || e >= p.rope_P)) {
        if (lane == 0) report(p.hdr, CSA2_ERR_BOUNDS, e);
        valid = false;
      }
      ok[u] = valid;
      if (valid) {
        const uint4* x0 = reinterpret_cast<const uint4*>(p.x + ((int64_t)b * p.T + j * p.m) * D + lane * 16);
        xr[u][0] = __ldg(x0);
        xr[u][1] = __ldg(x0 + 1);
        if (p.m == 2) {
          xr[u][2] = __ldg(x0 + D / 8);
          xr[u][3] = __ldg(x0 + D / 8 + 1);
        }
      }
    }
    // The four entries go through every step together (independent chains
    // side by side); invalid entries are computed on zeros and not stored.
    float y[EPW][16];
    if (p.m == 2) {
      float w0r[16], w1r[16];
      const float4* w0v = reinterpret_cast<const float4*>(p.w0 + lane * 16);
      const float4* w1v = reinterpret_cast<const float4*>(p.w1 + lane * 16);
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const float4 uu = __ldg(w0v + q), v = __ldg(w1v + q);
        w0r[4 * q] = uu.x; w0r[4 * q + 1] = uu.y; w0r[4 * q + 2] = uu.z; w0r[4 * q + 3] = uu.w;
        w1r[4 * q] = v.x; w1r[4 * q + 1] = v.y; w1r[4 * q + 2] = v.z; w1r[4 * q + 3] = v.w;
      }
#pragma unroll
      for (int k = 0; k < 16; k++) {
        const float den = __fadd_rn(w0r[k], w1r[k]);
#pragma unroll
        for (int u = 0; u < EPW; u++) {
          const uint32_t wa = k < 8 ? (&xr[u][0].x)[k / 2] : (&xr[u][1].x)[(k - 8) / 2];
          const uint32_t wb = k < 8 ? (&xr[u][2].x)[k / 2] : (&xr[u][3].x)[(k - 8) / 2];
          const float a = ok[u] ? bf16_bits_to_f32((wa >> (16 * (k & 1))) & 0xFFFFu) : 0.0f;
          const float bb = ok[u] ? bf16_bits_to_f32((wb >> (16 * (k & 1))) & 0xFFFFu) : 0.0f;
          y[u][k] = __fdiv_rn(__fmaf_rn(w0r[k], a, __fmul_rn(w1r[k], bb)), den);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < EPW; u++)
#pragma unroll
        for (int k = 0; k < 16; k++) {
          const uint32_t wa = k < 8 ? (&xr[u][0].x)[k / 2] : (&xr[u][1].x)[(k - 8) / 2];
          y[u][k] = ok[u] ? bf16_bits_to_f32((wa >> (16 * (k & 1))) & 0xFFFFu) : 0.0f;
        }
    }
    // RMSNorm
    float ps[EPW];
#pragma unroll
    for (int u = 0; u < EPW; u++) {
      ps[u] = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; k++) ps[u] = __fmaf_rn(y[u][k], y[u][k], ps[u]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
      for (int u = 0; u < EPW; u++) ps[u] = __fadd_rn(ps[u], __shfl_xor_sync(0xFFFFFFFFu, ps[u], off));
#pragma unroll
    for (int u = 0; u < EPW; u++) {
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ps[u], 512.0f), 1e-6f)));
#pragma unroll
      for (int k = 0; k < 16; k++) y[u][k] = __fmul_rn(y[u][k], r);
    }
    // RoPE on channels 448..511 = lanes 28..31, pairs i = 8*(lane-28) + k/2
    if (lane >= 28) {
#pragma unroll
      for (int u = 0; u < EPW; u++) {
        const int64_t e = ok[u] ? e0 + j0 + lwarp + u * CW_LOAD_WARPS : 0;
        const float4* cs = reinterpret_cast<const float4*>(p.rope_cs + (e * 32 + (lane - 28) * 8) * 2);
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const float4 v = __ldg(cs + q);          // two pairs: (cos, sin, cos, sin)
          const float y0 = y[u][4 * q], y1 = y[u][4 * q + 1], y2 = y[u][4 * q + 2], y3 = y[u][4 * q + 3];
          y[u][4 * q + 0] = __fmaf_rn(y0, v.x, -__fmul_rn(y1, v.y));
          y[u][4 * q + 1] = __fmaf_rn(y0, v.y, __fmul_rn(y1, v.x));
          y[u][4 * q + 2] = __fmaf_rn(y2, v.z, -__fmul_rn(y3, v.w));
          y[u][4 * q + 3] = __fmaf_rn(y2, v.w, __fmul_rn(y3, v.z));
        }
      }
    }
    // main FP4: this lane's 16 channels are exactly one scale group
#pragma unroll
    for (int u = 0; u < EPW; u++) {
      float amax = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; k++) amax = fmaxf(amax, fabsf(y[u][k]));
      const uint32_t sb = e4m3_byte(__fdiv_rn(amax, 6.0f));
      const float s = e4m3_value(sb);
      uint32_t packed[2] = {0u, 0u};
      if (s != 0.0f) {
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const uint32_t byte = e2m1x2(__fdiv_rn(y[u][2 * k], s), __fdiv_rn(y[u][2 * k + 1], s));
          packed[k / 4] |= byte << (8 * (k % 4));
        }
      }
      const int t = lwarp + u * CW_LOAD_WARPS;
      if (ok[u]) {
        uint8_t* ent = p.main_kv + ((int64_t)b * p.cap + e0 + j0 + t) * MAIN_BYTES;
        *reinterpret_cast<uint2*>(ent + lane * 8) = make_uint2(packed[0], packed[1]);
        ent[256 + lane] = (uint8_t)sb;
      }
    }
    if (it > 0) asm volatile("bar.sync 2, %0;" :: "n"(CW_THREADS) : "memory");   // EMPTY
#pragma unroll
    for (int u = 0; u < EPW; u++) {
      const int t = lwarp + u * CW_LOAD_WARPS;
      float4* yrow = reinterpret_cast<float4*>(ytile + t * D + lane * 16);
#pragma unroll
      for (int q = 0; q < 4; q++)
        yrow[q] = ok[u] ? make_float4(y[u][4 * q], y[u][4 * q + 1], y[u][4 * q + 2], y[u][4 * q + 3])
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) tile_valid[it & 1][t] = ok[u];
    }
    // next tile's token rows into L2 while this tile's projection runs
    {
      const int64_t nt = tile + gridDim.x;
      if (nt < n_tiles) {
        const int nb = (int)(nt / tiles_per_seq);
        const int64_t nj0 = (nt % tiles_per_seq) * CW_TILE;
        const int64_t rows = (nj0 + CW_TILE <= n_local ? CW_TILE : n_local - nj0) * p.m;
        const char* base = reinterpret_cast<const char*>(p.x + ((int64_t)nb * p.T + nj0 * p.m) * D);
        const int ltid = tid - CW_MATH_THREADS;
        for (int64_t off = (int64_t)ltid * 128; off < rows * D * 2; off += (int64_t)(CW_THREADS - CW_MATH_THREADS) * 128)
          asm volatile("prefetch.global.L2 [%0];" :: "l"(base + off));
      }
    }
    asm volatile("bar.arrive 1, %0;" :: "n"(CW_THREADS) : "memory");            // FULL
  }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(CW_MATH_REGS));
  for (int64_t tile = blockIdx.x, it = 0; tile < n_tiles; tile += gridDim.x, it++) {
    const int b = (int)(tile / tiles_per_seq);
    const int64_t j0 = (tile % tiles_per_seq) * CW_TILE;
    const int64_t e0 = p.entry_start[b];
    asm volatile("bar.sync 1, %0;" :: "n"(CW_THREADS) : "memory");              // FULL

    // ---------------- phase 2: k = W y', 4 outputs x 4 entries per thread,
    // as packed pairs of outputs (fma.rn.f32x2: two round-to-nearest fmas, the
    // same results as scalar ones), four channels at a time in channel order
    const int og = tid & 31;        // outputs 4*og .. 4*og+3
    const int eg = tid >> 5;        // entries 4*eg .. 4*eg+3
    unsigned long long acc2[2][4];  // [output pair][entry] = (out 2i, out 2i+1)
#pragma unroll
    for (int a = 0; a < 2; a++)
#pragma unroll
      for (int bq = 0; bq < 4; bq++) acc2[a][bq] = 0ull;          // (+0, +0)
    const float* yb = ytile + eg * 4 * D;                         // this thread's 4 entries
#pragma unroll 2
    for (int c4 = 0; c4 < D; c4 += 4) {
      float4 yv[4];
#pragma unroll
      for (int bq = 0; bq < 4; bq++) yv[bq] = *reinterpret_cast<const float4*>(yb + bq * D + c4);
#pragma unroll
      for (int cc = 0; cc < 4; cc++) {                              // channels in order
        const uint2 wv = *reinterpret_cast<const uint2*>(wt + (c4 + cc) * DI + og * 4);
        unsigned long long w01, w23;                                // bf16 -> fp32 pairs
        asm("mov.b64 %0, {%1, %2};" : "=l"(w01) : "r"(wv.x << 16), "r"(wv.x & 0xFFFF0000u));
        asm("mov.b64 %0, {%1, %2};" : "=l"(w23) : "r"(wv.y << 16), "r"(wv.y & 0xFFFF0000u));
#pragma unroll
        for (int bq = 0; bq < 4; bq++) {
          const float yc = cc == 0 ? yv[bq].x : cc == 1 ? yv[bq].y : cc == 2 ? yv[bq].z : yv[bq].w;
          unsigned long long yy;
          asm("mov.b64 %0, {%1, %1};" : "=l"(yy) : "f"(yc));
          asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[0][bq]) : "l"(yy), "l"(w01));
          asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[1][bq]) : "l"(yy), "l"(w23));
        }
      }
    }
    if (tile + gridDim.x < n_tiles) asm volatile("bar.arrive 2, %0;" :: "n"(CW_THREADS) : "memory");  // EMPTY
    float acc[4][4];
#pragma unroll
    for (int bq = 0; bq < 4; bq++) {
      asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[0][bq]), "=f"(acc[1][bq]) : "l"(acc2[0][bq]));
      asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2][bq]), "=f"(acc[3][bq]) : "l"(acc2[1][bq]));
    }

    // ---------------- phase 3: MXFP4 (8 lanes = one 32-wide block of outputs)
#pragma unroll
    for (int bq = 0; bq < 4; bq++) {
      const int t = eg * 4 + bq;
      const int64_t j = j0 + t;
      float amax = fmaxf(fmaxf(fabsf(acc[0][bq]), fabsf(acc[1][bq])), fmaxf(fabsf(acc[2][bq]), fabsf(acc[3][bq])));
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      if (!tile_valid[it & 1][t]) continue;     // uniform across the warp
      const int64_t e = e0 + j;
      uint32_t scale_byte, codes = 0;
      if (amax == 0.0f) {
        scale_byte = 0;
      } else {
        int ex = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;   // floor(log2 amax) for normals
        int X = ex - 2;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
        scale_byte = (uint32_t)(X + 127);
        float inv = __uint_as_float((uint32_t)(127 - X) << 23);      // 2^-X, exact
        uint32_t lo = e2m1x2(__fmul_rn(acc[0][bq], inv), __fmul_rn(acc[1][bq], inv));
        uint32_t hi = e2m1x2(__fmul_rn(acc[2][bq], inv), __fmul_rn(acc[3][bq], inv));
        codes = lo | (hi << 8);
      }
      uint8_t* cdst = p.idx_codes + ((int64_t)b * p.cap + e) * IDX_CODE_BYTES;
      *reinterpret_cast<uint16_t*>(cdst + og * 2) = (uint16_t)codes;
      if ((og & 7) == 0) p.idx_scales[((int64_t)b * p.cap + e) * IDX_SCALE_BYTES + (og >> 3)] = (uint8_t)scale_byte;
    }
  }
  }
}

// FP8 sliding-window rows: every bf16 value to E4M3 (nearest even,
// saturating at +-448, no scale).  One thread per 8 values: a 16-byte load,
// four paired conversions, an 8-byte store.
__global__ void swa_fp8_kernel(const uint16_t* __restrict__ x, int64_t n8, uint8_t* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t pk[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      uint16_t r;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
          : "=h"(r) : "f"(bf16_bits_to_f32(w[k] >> 16)), "f"(bf16_bits_to_f32(w[k] & 0xFFFFu)));
      pk[k] = r;
    }
    reinterpret_cast<uint2*>(out)[i] = make_uint2(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16));
  }
}

cudaError_t launch_swa_fp8(const uint16_t* x, int64_t n_rows, uint8_t* out, cudaStream_t stream) {
  const int64_t n8 = n_rows * (D / 8);
  if (n8 == 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return e;
  int64_t grid = ceil_div(n8, 256);
  if (grid > (int64_t)sms * 16) grid = (int64_t)sms * 16;      // grid-stride, at most 16 CTAs per SM
  swa_fp8_kernel<<<(unsigned)grid, 256, 0, stream>>>(x, n8, out);
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const CwParams& p, cudaStream_t stream, int num_sms) {
  static PerDeviceOnce attrs;
  cudaError_t err = attrs.ensure([](int) {
    return cudaFuncSetAttribute(cache_write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CW_SMEM);
  });
  if (err != cudaSuccess) return err;
  int64_t n_local = p.T / p.m;
  int64_t n_tiles = ceil_div(n_local, CW_TILE) * p.B;
  if (n_tiles == 0) return cudaSuccess;
  int grid = (int)(n_tiles < num_sms ? n_tiles : num_sms);
  cache_write_kernel<<<grid, CW_THREADS, CW_SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
