// (c) Joint sparse + SWA attention over the shared 512-d latent (K = V), on
// the 5th-generation tensor cores.
//
// Sources: "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" §3.3.2 (the readout
// concatenates the SWA KV with the selected main-KV entries into one sparse
// attention), §3.3.2.1 (key = value = the compressed content vector; the output
// is a convex combination of them), §2.4.4 (the FP4 cache is dequantised to a
// more precise format before attention: FP4 saves storage, it does not feed
// the matrix multiply); "4. 层维度(下):CSA2 与每 token 890 字节" §4.5.
//
// One CTA per query token streams its keys in chunks of 128: chunk 0 is the
// window (positions t-127 .. t), chunks 1.. are the selected slots in runs of
// 128.  One softmax over all of them is kept online (running maxima per head,
// rescaling the accumulated output only when a chunk's maximum exceeds the
// one in use by more than A_TAU, so that exp() never exceeds e^A_TAU).
// Both products run on f16 operands with fp32 accumulation:
//   * every FP4 value times its E4M3 scale has at most 6 significant bits and
//     lies between 2^-10 and 2688 in magnitude, so the f16 key is exact (E2M1
//     pairs -> f16x2 by the hardware conversion, times the scale in f16x2);
//   * E4M3 window values are f16 values; bf16 q and window rows are rounded to
//     f16 in shared memory, exact for magnitudes in [2^-14, 65504] (smaller
//     ones keep an absolute error below 2^-25; the layer's activations are
//     expected inside f16's range);
//   * P = 2^(s - m) <= 2^A_TAU is stored in f16 (11 significant bits).
//   * Q (64 heads x 512) lands once by TMA in 8 SW128 column chunks.
//   * The key buffer holds one chunk as f16 [128 keys][512] in 8 SW128 column
//     chunks of 64 dims (16 KB each).  The window chunk lands by 2-D TMA (an
//     FP8 window as 64-byte E4M3 column slices in the upper half of each column
//     chunk) and is converted in place tile by tile together with Q.  A
//     selected chunk is dequantised by the 8 math warps from registers: every
//     thread loads its key's FP4 bytes for the next chunk while the current one
//     is processed (2 threads per key, 64 dims of each 128-dim tile per
//     thread), so the gather's latency hides behind a whole chunk.
//   * S^T = K Q^T is an M=128 (keys) x N=64 (heads) x K=512 tcgen05 f16 MMA
//     product issued as four chains of 8 MMAs (dims 128t .. 128t + 127, one
//     TMEM accumulator each) by four threads; chain t starts as soon as tile t
//     of the key buffer is written.
//   * Softmax straight from TMEM (thread = key, 32 heads in registers, the four
//     partial products added; column maxima and sums by transpose-reductions
//     over the lanes, the four warps of a head half meet on a named barrier),
//     in base-2 units (the scale carries log2 e): P = 2^(S - m) becomes the
//     MN-major f16 B operand [key][head] of the second product.
//   * O^T += V^T P^T reuses the key buffer as an MN-major A operand: 4 tiles of
//     M=128 dims x N=64 heads x K=128 keys, accumulated over the chunks in TMEM,
//     issued tile after tile by one thread with a commit per tile, so that the
//     tiles complete in order.  Once tile t of a chunk is done, its two column
//     chunks are free and the next chunk's dequantisation writes them while the
//     later tiles' products run.
//   * At the end every thread divides its dim row of O^T by the head sums and
//     stores bf16 rows of the output.
// All mbarrier waits are bounded; a timeout reports CSA2_ERR_TIMEOUT and the
// kernel still runs to its end (every thread takes every barrier).
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "host_once.cuh"
#include "params.cuh"
#include "tc.cuh"

namespace csa2 {

constexpr int A_MATH_WARPS = 8;                         // dequantisation, softmax, output
constexpr int A_MATH = 32 * A_MATH_WARPS;
constexpr int A_THREADS = A_MATH + 4 * 32;              // + 4 MMA-issuing warps (one also loads, one owns TMEM)
constexpr int A_KEYS = 128;                             // keys per chunk (one M = 128 tile)
constexpr int A_CHUNK_BYTES = A_KEYS * 128;             // [128 keys][64 dims] 16-bit = 16 KB
constexpr int A_QCHUNK_BYTES = H * 128;                 // [64 heads][64 dims] 16-bit = 8 KB
constexpr int A_OFF_K = 0;                              // 8 key column chunks, 128 KB
constexpr int A_OFF_Q = 8 * A_CHUNK_BYTES;              // 8 Q column chunks, 64 KB
constexpr int A_OFF_P = A_OFF_Q + 8 * A_QCHUNK_BYTES;   // P^T [128 keys][64 heads] f16 SW128, 16 KB
constexpr int A_OFF_SMALL = A_OFF_P + A_KEYS * H * 2;
constexpr int A_TMEM_COLS = 512;
constexpr int A_S_COL = 0;                              // S^T partial of tile t at 64 t
constexpr int A_O_COL = 256;                            // O^T tile t at 256 + 64 t
constexpr float A_LOG2E = 1.4426950408889634f;
// split mode: one partial softmax state per (query, CTA): the maxima in use and
// the sums per head (base-2 units), then the unnormalised O [head][dim]
constexpr int A_PART_FLOATS = 2 * H + H * D;
constexpr int A_SPLIT_MAX_BQ = CSA2_ATTN_SPLIT_MAX_QUERIES;   // queries of a call that may be split
constexpr float A_TAU = 8.0f * A_LOG2E;                 // lazy rescale threshold: 2^A_TAU = e^8

struct AsSmall {
  int32_t ids[CSA2_MAX_K];            // the query's selected entry ids
  float red[A_MATH_WARPS][32];        // per-warp column maxima / sums (warp 4 hh + q: head 32 hh + lane)
  alignas(16) float mv[A_MATH_WARPS][32];   // each warp's maxima in use, read back by all of its lanes
  uint64_t q_full[4], win_full[4];    // TMA: Q / window column chunks 2t, 2t + 1
  uint64_t kready[4];                 // tile t (dims 128t ..) of a chunk is in the key buffer (8 arrivals)
  uint64_t s_full;                    // the four S^T chains of a chunk are done (4 commits)
  uint64_t p_ready;                   // P^T written, O^T rescaled if needed (8 arrivals)
  uint64_t pv_done[4];                // O^T tile t of a chunk is done (1 commit)
  uint32_t tmem_base;
  int err;
};
constexpr int A_SMEM = A_OFF_SMALL + (int)sizeof(AsSmall) + 1024;
static_assert(A_OFF_Q % 1024 == 0 && A_OFF_P % 1024 == 0, "SW128 regions are 1 KB aligned");
static_assert(A_SMEM <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// two bf16 (element 0 in the low half) -> two f16, round to nearest
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Eight E2M1 codes (element k in bits 4k .. 4k+3 of w) -> four f16x2 words
// (element 2i in the low half of word i): one hardware conversion per byte.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t o[4]) {
  asm("{ .reg .b8 t0, t1, t2, t3;\n mov.b32 {t0, t1, t2, t3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, t0;\n cvt.rn.f16x2.e2m1x2 %1, t1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, t2;\n cvt.rn.f16x2.e2m1x2 %3, t3; }"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// Two E4M3 bytes (element 0 in bits 0..7) -> one f16x2 word (element 0 in the
// low half).  Exact: every E4M3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  asm("{ .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(d) : "r"(two));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// byte offset of (row, byte) in a 1 KB-aligned SW128 region of 128-byte rows
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte) {
  return row * 128u + ((((byte >> 4) ^ (row & 7u)) << 4) | (byte & 15u));
}

// 2^x, approximate (the MUFU unit), subnormal results flushed to zero
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ bool as_wait(uint64_t* bar, uint32_t parity, AsSmall& sm, WsHeader* hdr, int where) {
  if (tc::bar_wait(bar, parity)) return true;
  if (atomicExch(&sm.err, 1) == 0) report(hdr, CSA2_ERR_TIMEOUT, where);
  return false;
}

// The issuing threads wait with a short sleep between polls, leaving issue
// slots to the math warps of their SM sub-partition.
__device__ __forceinline__ bool as_wait_sleepy(uint64_t* bar, uint32_t parity, AsSmall& sm, WsHeader* hdr,
                                               int where) {
  for (uint32_t it = 0; it < 4000000u; it++) {
    if (tc::bar_wait(bar, parity, 1u)) return true;
    __nanosleep(64);
  }
  if (atomicExch(&sm.err, 1) == 0) report(hdr, CSA2_ERR_TIMEOUT, where);
  return false;
}

// 32 consecutive TMEM columns of this thread's lane -> r (waited)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  tc::tmem_ld_x32_nowait(taddr, r);
  tc::tmem_wait_ld_regs(r);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                  "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                  "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                  "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                  "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

// transpose-reduction over the 32 lanes of a warp: afterwards lane l holds the
// reduction of column l (r[l] of every lane); r is destroyed
template <bool MAX>
__device__ __forceinline__ float lane_columns(float* r, int lane) {
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) {
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < k; i++) {
      const float send = upper ? r[i] : r[i + k];
      const float keep = upper ? r[i + k] : r[i];
      const float got = __shfl_xor_sync(0xFFFFFFFFu, send, k);
      r[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return r[0];
}

// SPLIT: the query's chunks are divided among p.split CTAs, which write partial
// states for attn_combine_kernel (a separate instance, so that the one-CTA
// kernel carries none of it).
template <bool SPLIT>
__global__ void __launch_bounds__(A_THREADS, 1)
attn_stream_kernel(AttnParams p, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_swa) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = tc::align_smem_1k(smem_raw);
  unsigned char* kbuf = smem + A_OFF_K;
  unsigned char* qbuf = smem + A_OFF_Q;
  unsigned char* pbuf = smem + A_OFF_P;
  AsSmall& sm = *reinterpret_cast<AsSmall*>(smem + A_OFF_SMALL);

  const int split = SPLIT ? p.split : 1;                 // CTAs per query
  const int bq = blockIdx.x / split, sp = blockIdx.x % split;
  const int b = bq / p.Q;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K;
  const int nc = 1 + (K + A_KEYS - 1) / A_KEYS;          // window chunk + selected chunks
  // this CTA's chunks (all of them unless the query is split; split <= nc)
  const int c_lo = sp * nc / split, c_hi = (sp + 1) * nc / split;
  // its selected entries: slots e_lo .. e_hi - 1
  const int e_lo = c_lo > 0 ? A_KEYS * (c_lo - 1) : 0, e_hi = min(K, A_KEYS * (c_hi - 1));

  // ---------------- set-up (reads no input: overlaps the previous kernel under PDL)
  if (warp == A_MATH_WARPS + 3) tc::tmem_alloc(&sm.tmem_base, A_TMEM_COLS);
  if (tid == 0) {
    for (int u = 0; u < 4; u++) tc::bar_init(&sm.kready[u], A_MATH_WARPS);
    tc::bar_init(&sm.s_full, 4);
    tc::bar_init(&sm.p_ready, A_MATH_WARPS);
    for (int t = 0; t < 4; t++) tc::bar_init(&sm.pv_done[t], 1);
    sm.err = 0;
    tc::bar_init_fence();
  }
  if (warp >= A_MATH_WARPS && lane == 0) {
    // issuer u owns the copy barriers of its tile (initialised here, used by it
    // before the CTA barrier below, waited on by the math warps after it)
    const int u = warp - A_MATH_WARPS;
    tc::bar_init(&sm.q_full[u], 1);
    tc::bar_init(&sm.win_full[u], 1);
    tc::bar_init_fence();
    tc::prefetch_tensormap(&map_q);
    tc::prefetch_tensormap(&map_swa);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t t = p.q_pos[bq];
  if (warp >= A_MATH_WARPS && lane == 0) {
    // tile u's Q and window column chunks by TMA, before the selection ids are
    // read and the CTA barrier: Q needs no other input and goes first
    const int u = warp - A_MATH_WARPS;
    tc::bar_arrive_expect_tx(&sm.q_full[u], 2u * A_QCHUNK_BYTES);
    for (int c = 2 * u; c < 2 * u + 2; c++)
      tc::tma_load_2d(qbuf + c * A_QCHUNK_BYTES, &map_q, c * 64, bq * H, &sm.q_full[u]);
    if (p.S > 0 && c_lo == 0) {   // rows outside this sequence's window are masked, but finite
      const int32_t row0 = (int32_t)((int64_t)b * p.S + (t - (WIN - 1) - p.swa_base[b]));
      if (p.swa_fp8) {       // [128 rows][64 B] E4M3 slices into the upper half of each column chunk
        tc::bar_arrive_expect_tx(&sm.win_full[u], 2u * (A_CHUNK_BYTES / 2));
        for (int c = 2 * u; c < 2 * u + 2; c++)
          tc::tma_load_2d(kbuf + c * A_CHUNK_BYTES + A_CHUNK_BYTES / 2, &map_swa, c * 64, row0, &sm.win_full[u]);
      } else {
        tc::bar_arrive_expect_tx(&sm.win_full[u], 2u * A_CHUNK_BYTES);
        for (int c = 2 * u; c < 2 * u + 2; c++)
          tc::tma_load_2d(kbuf + c * A_CHUNK_BYTES, &map_swa, c * 64, row0, &sm.win_full[u]);
      }
    }
    // the query's selected entries into L2 ahead of the math warps' per-chunk loads
    // (by the copy engine: the load pipe stays free): a quarter of the packed
    // selection per issuing warp here, or one 288-byte entry per id once the ids
    // are in shared memory
    if (p.packed_in && e_hi > e_lo) {
      const uint64_t first = (uint64_t)e_lo * MAIN_BYTES, total = (uint64_t)(e_hi - e_lo) * MAIN_BYTES;
      const uint64_t a0 = (total * u / 4) & ~(uint64_t)15;
      const uint64_t a1 = u == 3 ? total : ((total * (u + 1) / 4) & ~(uint64_t)15);
      if (a1 > a0)
        tc::prefetch_l2(p.packed_in + (int64_t)bq * K * MAIN_BYTES + first + a0, (uint32_t)(a1 - a0));
    }
  }
  for (int i = tid; i < K; i += A_THREADS) sm.ids[i] = p.sel[(int64_t)bq * K + i];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp >= A_MATH_WARPS) {
    // ================= MMA issuers: warp 8 + u issues, for every chunk, the S^T
    // chain of tile u (dims 128u .. 128u + 127); warp 8 also issues the four O^T tiles
    const int u = warp - A_MATH_WARPS;
    if (!p.packed_in) {      // the gathered entries into L2 (the packed ones went at the start)
      for (int i = e_lo + u * 32 + lane; i < e_hi; i += 128) {
        const int32_t id = sm.ids[i];
        if (id >= 0 && id < p.cap) tc::prefetch_l2(p.main_kv + ((int64_t)b * p.cap + id) * MAIN_BYTES, MAIN_BYTES);
      }
    }
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_f16(A_KEYS, H, 0, 0);
      constexpr uint32_t idesc_o = tc::idesc_f16(128, H, 1, 1);
      // descriptors: the 14-bit start address field (address / 16) never carries
      // (shared memory < 256 KB), so offsets are added to it directly
      const uint64_t a_s = tc::smem_desc(tc::smem_u32(kbuf + 2 * u * A_CHUNK_BYTES), 16, 1024, tc::SW_128B);
      const uint64_t b_s = tc::smem_desc(tc::smem_u32(qbuf + 2 * u * A_QCHUNK_BYTES), 16, 1024, tc::SW_128B);
      const uint64_t a_o = tc::smem_desc(tc::smem_u32(kbuf), A_CHUNK_BYTES, 1024, tc::SW_128B);
      const uint64_t b_o = tc::smem_desc(tc::smem_u32(pbuf), 8192, 1024, tc::SW_128B);
      const uint32_t s_acc = tmem + A_S_COL + 64 * u;
      bool ok = true;
      for (int c = c_lo; c < c_hi; c++) {
        const uint32_t ph = (uint32_t)(c - c_lo) & 1u;
        ok = as_wait_sleepy(&sm.kready[u], ph, sm, p.hdr, 31) && ok;
        tc::fence_after_sync();
        if (ok) {                                     // S^T partial of tile u: column chunks 2u, 2u + 1
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const uint32_t off = (uint32_t)((i >> 2) * A_CHUNK_BYTES + (i & 3) * 32) >> 4;
            const uint32_t offq = (uint32_t)((i >> 2) * A_QCHUNK_BYTES + (i & 3) * 32) >> 4;
            tc::mma_f16(s_acc, a_s + off, b_s + offq, idesc_s, i ? 1u : 0u);
          }
        }
        tc::commit(&sm.s_full);
        if (u != 0) continue;
        // O^T += V^T P^T over this chunk's 128 keys, tile by tile from one thread:
        // the tiles complete in order, so the next chunk's dequantisation of tile
        // 0 starts after one tile's products instead of all four
        ok = as_wait_sleepy(&sm.p_ready, ph, sm, p.hdr, 33) && ok;
        tc::fence_after_sync();
#pragma unroll 1
        for (int v = 0; v < 4; v++) {
          if (ok) {
            const uint64_t a_v = a_o + (uint32_t)(2 * v * A_CHUNK_BYTES >> 4);
#pragma unroll
            for (int ks = 0; ks < A_KEYS / 16; ks++)
              tc::mma_f16(tmem + A_O_COL + 64 * v, a_v + (uint32_t)(ks * 2048 >> 4),
                           b_o + (uint32_t)(ks * 2048 >> 4), idesc_o, (c > c_lo || ks) ? 1u : 0u);
          }
          tc::commit(&sm.pv_done[v]);
        }
      }
    }
    __syncwarp();
  } else {
    // ================= math warps
    const int q4 = warp & 3, hh = warp >> 2;          // TMEM lane quarter; head half (heads 32 hh ..)
    const int key = tid >> 1, kh = tid & 1;           // dequantisation: key row, 64-dim half of each tile
    const int m = q4 * 32 + lane;                     // softmax / output: key row or dim row of a tile
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t xr = (uint32_t)key & 7u;
    uint4 cd[8];                                      // FP4 codes of the next chunk: tile u in cd[2u], cd[2u+1]
    uint4 scv[2];                                     // its 32 scale bytes
    bool kv = false;                                  // the next chunk's key of this thread exists
    auto prefetch = [&](int chunk) {
      const int slot = A_KEYS * (chunk - 1) + key;
      const int32_t id = slot < K ? sm.ids[slot] : -1;
      kv = id >= 0 && id < p.cap;
      if (id >= p.cap && kh == 0) report(p.hdr, CSA2_ERR_BOUNDS, id);
#pragma unroll
      for (int i = 0; i < 8; i++) cd[i] = make_uint4(0u, 0u, 0u, 0u);
      scv[0] = scv[1] = make_uint4(0u, 0u, 0u, 0u);
      if (kv) {
        const unsigned char* src = p.packed_in ? p.packed_in + ((int64_t)bq * K + slot) * MAIN_BYTES
                                               : p.main_kv + ((int64_t)b * p.cap + id) * MAIN_BYTES;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
        for (int u = 0; u < 4; u++) {
          cd[2 * u] = __ldg(s4 + 4 * u + 2 * kh);
          cd[2 * u + 1] = __ldg(s4 + 4 * u + 2 * kh + 1);
        }
        scv[0] = __ldg(s4 + 16);
        scv[1] = __ldg(s4 + 17);
      }
    };
    // tile u of the current chunk: 64 dims (column chunk 2u + kh) of this thread's key
    auto dequant_tile = [&](int u) {
      const uint4 c0 = cd[2 * u], c1 = cd[2 * u + 1];
      const uint32_t cwd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const uint4& sv = scv[u >> 1];
      const uint32_t sw = (u & 1) ? (kh ? sv.w : sv.z) : (kh ? sv.y : sv.x);   // scale bytes 8u + 4kh ..
      unsigned char* dst = kbuf + (2 * u + kh) * A_CHUNK_BYTES + key * 128;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        // the odd half walks its 16-channel groups as i ^ 2, so the two threads of a
        // key never store to the same 16-byte bank group in one instruction
        const int g = kh ? (i ^ 2) : i;
        const uint32_t wa = kh ? cwd[2 * (i ^ 2)] : cwd[2 * i];          // static indices only
        const uint32_t wb = kh ? cwd[2 * (i ^ 2) + 1] : cwd[2 * i + 1];
        const uint32_t sc2 = e4m3x2_to_f16x2(prmt(sw >> (8 * g), 0u, 0x0000u));   // the group's scale, twice
        uint32_t o[8];
        e2m1x8_to_f16(wa, o);
        e2m1x8_to_f16(wb, o + 4);
#pragma unroll
        for (int k = 0; k < 8; k++) o[k] = hmul2(o[k], sc2);
        *reinterpret_cast<uint4*>(dst + (((2u * g) ^ xr) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + (((2u * g + 1u) ^ xr) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    };
    if (max(c_lo, 1) < c_hi) prefetch(max(c_lo, 1));
    float m_used = -INFINITY;                         // max in use for head 32 hh + lane
    float l_part = 0.f;                               // sum of P over this warp's keys, head 32 hh + lane
    bool ok = true;
    // Q column chunks 2u, 2u + 1 (bf16 by TMA) rounded to f16 in place
    auto convert_q = [&](int u) {
      uint4* qv = reinterpret_cast<uint4*>(qbuf + 2 * u * A_QCHUNK_BYTES);
#pragma unroll
      for (int i = tid; i < 2 * A_QCHUNK_BYTES / 16; i += A_MATH) {
        const uint4 x = qv[i];
        qv[i] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
      }
    };
    for (int c = c_lo; c < c_hi; c++) {
      const uint32_t ph = (uint32_t)(c - c_lo) & 1u;
      // ---------------- the chunk's keys into the key buffer
      if (c == 0) {
        // Q and the window rows tile by tile (column chunks 2u, 2u + 1): bf16 rounded
        // to f16, E4M3 widened to f16, in place; then tile u is ready for its chain
#pragma unroll 1
        for (int u = 0; u < 4; u++) {
          ok = as_wait(&sm.q_full[u], 0, sm, p.hdr, 32) && ok;
          convert_q(u);
          unsigned char* kt = kbuf + 2 * u * A_CHUNK_BYTES;
          if (p.S == 0) {                             // no window rows supplied: zero keys (all masked)
#pragma unroll
            for (int i = tid; i < 2 * A_CHUNK_BYTES / 16; i += A_MATH)
              reinterpret_cast<uint4*>(kt)[i] = make_uint4(0u, 0u, 0u, 0u);
          } else if (!p.swa_fp8) {
            ok = as_wait(&sm.win_full[u], 0, sm, p.hdr, 34) && ok;
#pragma unroll 4
            for (int i = tid; i < 2 * A_CHUNK_BYTES / 16; i += A_MATH) {
              uint4* kv4 = reinterpret_cast<uint4*>(kt) + i;
              const uint4 x = *kv4;
              *kv4 = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                                bf16x2_to_f16x2(x.w));
            }
          } else {
            ok = as_wait(&sm.win_full[u], 0, sm, p.hdr, 34) && ok;
            // thread (r, h) widens row r, dims 32h .. 32h+31 of both column chunks (32
            // E4M3 bytes at 8 KB + 64 r + 32 h) into four 16-byte f16 units at their
            // SW128 places; every thread reads both chunks before any writes them
            const int r = tid >> 1, h = tid & 1;
            uint4 raw[2][2];
#pragma unroll
            for (int i = 0; i < 2; i++) {
              const uint4* src = reinterpret_cast<const uint4*>(kt + i * A_CHUNK_BYTES + A_CHUNK_BYTES / 2 + r * 64 +
                                                                h * 32);
              raw[i][0] = src[0];
              raw[i][1] = src[1];
            }
            named_sync(1, A_MATH);
#pragma unroll
            for (int i = 0; i < 2; i++) {
              unsigned char* dst = kt + i * A_CHUNK_BYTES;
#pragma unroll
              for (int j = 0; j < 4; j++) {
                const uint4& w = raw[i][j >> 1];
                const uint32_t lo = (j & 1) ? w.z : w.x, hi = (j & 1) ? w.w : w.y;   // bytes 8j .. 8j+7
                const uint4 o = make_uint4(e4m3x2_to_f16x2(lo), e4m3x2_to_f16x2(lo >> 16), e4m3x2_to_f16x2(hi),
                                           e4m3x2_to_f16x2(hi >> 16));
                *reinterpret_cast<uint4*>(dst + sw128((uint32_t)r, (uint32_t)(64 * h + 16 * j))) = o;
              }
            }
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::bar_arrive(&sm.kready[u]);
        }
      } else {
        // selected chunk: tile u's column chunks are free once chunk c-1's O^T tile u is done
        // (the first chunk of a CTA without the window also rounds Q's tile u first)
#pragma unroll
        for (int u = 0; u < 4; u++) {
          ok = as_wait(&sm.pv_done[u], ph ^ 1u, sm, p.hdr, 35) && ok;
          tc::fence_after_sync();
          if (SPLIT && c == c_lo) {
            ok = as_wait(&sm.q_full[u], 0, sm, p.hdr, 32) && ok;
            convert_q(u);
          }
          dequant_tile(u);
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::bar_arrive(&sm.kready[u]);
        }
        if (p.packed_out && kv) {                     // the selected entry, in slot order, for Reuse layers
          const int slot = A_KEYS * (c - 1) + key;
          uint4* dst = reinterpret_cast<uint4*>(p.packed_out + ((int64_t)bq * K + slot) * MAIN_BYTES);
#pragma unroll
          for (int u = 0; u < 4; u++) {
            dst[4 * u + 2 * kh] = cd[2 * u];
            dst[4 * u + 2 * kh + 1] = cd[2 * u + 1];
          }
          dst[16 + kh] = kh ? scv[1] : scv[0];
        }
      }

      // ---------------- softmax of the chunk, straight from TMEM
      ok = as_wait(&sm.s_full, ph, sm, p.hdr, 36) && ok;
      tc::fence_after_sync();
      bool valid;
      if (c == 0) {
        const int64_t pos = t - (WIN - 1) + m;
        const int64_t row = pos - p.swa_base[b];
        valid = pos >= 0 && p.S > 0 && row >= 0 && row < p.S;
        if (pos >= 0 && !valid && hh == 0) report(p.hdr, CSA2_ERR_BOUNDS, pos);
      } else {
        const int slot = A_KEYS * (c - 1) + m;
        const int32_t id = slot < K ? sm.ids[slot] : -1;
        valid = id >= 0 && id < p.cap;
      }
      float v[32], r[32];
      {
        const float sc2 = p.scale * A_LOG2E;          // base-2 logits
        uint32_t s1[32], s2[32];
        const uint32_t taddr = tmem + lane_off + A_S_COL + 32 * hh;
        tc::tmem_ld_x32_nowait(taddr, s1);
        tc::tmem_ld_x32_nowait(taddr + 64, s2);
        tc::tmem_wait_ld_regs(s1);
        tc::tmem_wait_ld_regs(s2);
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = __uint_as_float(s1[j]) + __uint_as_float(s2[j]);
        tc::tmem_ld_x32_nowait(taddr + 128, s1);
        tc::tmem_ld_x32_nowait(taddr + 192, s2);
        tc::tmem_wait_ld_regs(s1);
        tc::tmem_wait_ld_regs(s2);
#pragma unroll
        for (int j = 0; j < 32; j++)
          v[j] = valid ? (v[j] + (__uint_as_float(s1[j]) + __uint_as_float(s2[j]))) * sc2 : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < 32; j++) r[j] = v[j];
      sm.red[warp][lane] = lane_columns<true>(r, lane);
      named_sync(2 + hh, 128);                        // the four warps of this head half
      const float cm = fmaxf(fmaxf(sm.red[4 * hh][lane], sm.red[4 * hh + 1][lane]),
                             fmaxf(sm.red[4 * hh + 2][lane], sm.red[4 * hh + 3][lane]));
      // online maximum: O^T holds nothing yet (chunk 0) or only zeros (every earlier
      // key masked) while m_used is -inf; otherwise rescale only past A_TAU
      float alpha = 1.f;
      if (m_used == -INFINITY) {
        m_used = cm;
      } else if (cm > m_used + A_TAU) {
        alpha = ex2_ftz(m_used - cm);
        m_used = cm;
        l_part *= alpha;
      }
      if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // identical decision in the four warps of the half; every warp rescales
        // its lane quarter of the half's 32 heads in all four O^T tiles (chunk
        // c-1's products are complete: this chunk's S^T needed them)
        float al[32];
#pragma unroll
        for (int j = 0; j < 32; j++) al[j] = __shfl_sync(0xFFFFFFFFu, alpha, j);
#pragma unroll 1
        for (int u = 0; u < 4; u++) {
          uint32_t o[32];
          const uint32_t taddr = tmem + lane_off + A_O_COL + 64 * u + 32 * hh;
          tmem_ld32(taddr, o);
#pragma unroll
          for (int j = 0; j < 32; j++) o[j] = __float_as_uint(__uint_as_float(o[j]) * al[j]);
          tmem_st32(taddr, o);
        }
        tc::tmem_wait_st();
      }
      // every lane needs the maxima in use of all 32 heads: through shared memory
      sm.mv[warp][lane] = m_used;
      __syncwarp();
      uint32_t pk[16];
#pragma unroll
      for (int j4 = 0; j4 < 8; j4++) {
        const float4 m4 = *reinterpret_cast<const float4*>(&sm.mv[warp][4 * j4]);
        const float mj[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int j = 4 * j4 + e;
          r[j] = (v[j] == -INFINITY) ? 0.f : ex2_ftz(v[j] - mj[e]);
          if (j & 1) pk[j >> 1] = pack_f16x2(r[j - 1], r[j]);
        }
      }
      // P^T row m (heads 32 hh .. +31 = 16-byte units 4 hh .. 4 hh + 3), SW128
#pragma unroll
      for (int u = 0; u < 4; u++)
        *reinterpret_cast<uint4*>(pbuf + sw128((uint32_t)m, (uint32_t)(hh * 64 + u * 16))) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      tc::fence_proxy_async_smem();                   // P^T is read by the tensor cores
      l_part += lane_columns<false>(r, lane);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&sm.p_ready);
      // the next chunk's FP4 bytes: issued after the softmax, whose shared-memory and
      // TMEM traffic would otherwise queue behind these loads
      if (c + 1 < c_hi) prefetch(c + 1);
    }

    // ---------------- output: O^T / L, bf16 rows out[head][dim]
    for (int u = 0; u < 4; u++) ok = as_wait(&sm.pv_done[u], (uint32_t)(c_hi - 1 - c_lo) & 1u, sm, p.hdr, 37) && ok;
    tc::fence_after_sync();
    // the next kernel of the stream may be scheduled now (triggered at the start,
    // its CTAs would hold SMs idle in their own wait for this whole kernel)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    sm.red[warp][lane] = l_part;
    named_sync(2 + hh, 128);
    const float lsum = sm.red[4 * hh][lane] + sm.red[4 * hh + 1][lane] + sm.red[4 * hh + 2][lane] +
                       sm.red[4 * hh + 3][lane];
    if (!SPLIT) {
      const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
      float il[32];
#pragma unroll
      for (int j = 0; j < 32; j++) il[j] = __shfl_sync(0xFFFFFFFFu, inv, j);
      uint16_t* out = p.out + (int64_t)bq * H * D + (int64_t)(32 * hh) * D + m;
#pragma unroll 1
      for (int u = 0; u < 4; u++) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + A_O_COL + 64 * u + 32 * hh, o);
#pragma unroll
        for (int j = 0; j < 32; j++)
          out[j * D + 128 * u] = (uint16_t)(pack_bf16x2(__uint_as_float(o[j]) * il[j], 0.f) & 0xFFFFu);
      }
    } else {
      // this CTA's partial state: maxima in use and sums of heads 32 hh + lane,
      // then the unnormalised O^T rows (dim 128 u + m of heads 32 hh ..) as O[head][dim]
      float* part = p.opart + (int64_t)blockIdx.x * A_PART_FLOATS;
      if (q4 == 0) {
        part[32 * hh + lane] = m_used;
        part[H + 32 * hh + lane] = lsum;
      }
      float* op = part + 2 * H + (int64_t)(32 * hh) * D + m;
#pragma unroll 1
      for (int u = 0; u < 4; u++) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + A_O_COL + 64 * u + 32 * hh, o);
#pragma unroll
        for (int j = 0; j < 32; j++) op[j * D + 128 * u] = __uint_as_float(o[j]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == A_MATH_WARPS + 3) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, A_TMEM_COLS);
  }
}

// Split mode: the output of one query from its CTAs' partial states.  With m_s,
// l_s, O_s the maxima in use, sums and unnormalised outputs of CTA s (base-2
// units), m = max_s m_s and w_s = 2^(m_s - m): O = sum_s w_s O_s / sum_s w_s l_s,
// the softmax over the union of the CTAs' keys.  Four CTAs per query (16 heads
// each), thread = (head, 32 dims); a head whose keys are all masked gets zeros,
// as in the one-CTA path.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part, int split,
                                                           uint16_t* __restrict__ out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bq = blockIdx.x >> 2;
  const int h = (blockIdx.x & 3) * 16 + (threadIdx.x >> 4), d0 = (threadIdx.x & 15) * 32;
  const float* pb = part + (int64_t)bq * split * A_PART_FLOATS;
  float mx = -INFINITY;
  for (int s = 0; s < split; s++) mx = fmaxf(mx, pb[(int64_t)s * A_PART_FLOATS + h]);
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; i++) acc[i] = 0.f;
  float L = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < split; s++) {
      const float* ps = pb + (int64_t)s * A_PART_FLOATS;
      const float ms = ps[h];
      if (ms == -INFINITY) continue;                       // no unmasked key in this CTA's chunks
      const float w = exp2f(ms - mx);
      L += w * ps[H + h];
      const float4* o4 = reinterpret_cast<const float4*>(ps + 2 * H + (int64_t)h * D + d0);
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const float4 v = o4[i];
        acc[4 * i] += w * v.x;
        acc[4 * i + 1] += w * v.y;
        acc[4 * i + 2] += w * v.z;
        acc[4 * i + 3] += w * v.w;
      }
    }
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  uint4* o = reinterpret_cast<uint4*>(out + ((int64_t)bq * H + h) * D + d0);
#pragma unroll
  for (int i = 0; i < 4; i++)
    o[i] = make_uint4(pack_bf16x2(acc[8 * i] * inv, acc[8 * i + 1] * inv), pack_bf16x2(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                      pack_bf16x2(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv), pack_bf16x2(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
}

// ------------------------------------------------------------------ host side
// E4M3 matrix [rows][512] with unswizzled boxes of 64 bytes x box_rows rows.
static bool encode_u8_rows512(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, rows};
  cuuint64_t strides[1] = {(cuuint64_t)D};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 matrix [rows][512] with SW128 boxes of 64 columns x box_rows rows.
static bool encode_bf16_rows512(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Partial states for a split call: calls of up to A_SPLIT_MAX_BQ queries may be
// split over as many CTAs per query as they have chunks.
size_t attn_partials_bytes(int64_t BQ, int K) {
  if (BQ <= 0 || BQ > A_SPLIT_MAX_BQ) return 0;
  const int64_t nc = 1 + (K + A_KEYS - 1) / A_KEYS;
  return (size_t)(BQ * nc * A_PART_FLOATS) * sizeof(float);
}

int attn_split_max_queries() { return A_SPLIT_MAX_BQ; }

cudaError_t launch_attention(AttnParams p, int B, float* part, cudaStream_t stream) {
  const int64_t BQ = (int64_t)B * p.Q;
  if (BQ == 0) return cudaSuccess;
  const int nc = 1 + (p.K + A_KEYS - 1) / A_KEYS;
  if (p.split < 1) p.split = 1;
  if (p.split > nc) p.split = nc;                               // at least one chunk per CTA
  if (p.split > 1 && (part == nullptr || BQ > A_SPLIT_MAX_BQ)) return cudaErrorInvalidValue;
  p.opart = part;
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.ensure([](int) {
    cudaError_t r = cudaFuncSetAttribute(attn_stream_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, A_SMEM);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(attn_stream_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, A_SMEM);
  });
  if (e != cudaSuccess) return e;
  CUtensorMap map_q, map_swa;
  if (!encode_bf16_rows512(&map_q, p.q, (uint64_t)BQ * H, 64)) return cudaErrorInvalidValue;
  const uint64_t swa_rows = (uint64_t)B * (uint64_t)(p.S > 0 ? p.S : 1);
  const bool swa_ok = p.swa_fp8 ? encode_u8_rows512(&map_swa, p.swa, swa_rows, A_KEYS)
                                : encode_bf16_rows512(&map_swa, p.swa, swa_rows, A_KEYS);
  if (!swa_ok) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(BQ * p.split));
  cfg.blockDim = dim3(A_THREADS);
  cfg.dynamicSmemBytes = A_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // set-up overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = p.split > 1 ? cudaLaunchKernelEx(&cfg, attn_stream_kernel<true>, p, map_q, map_swa)
                   : cudaLaunchKernelEx(&cfg, attn_stream_kernel<false>, p, map_q, map_swa);
  if (e != cudaSuccess || p.split == 1) return e;
  cudaLaunchConfig_t cc = {};
  cc.gridDim = dim3((unsigned)(BQ * 4));
  cc.blockDim = dim3(256);
  cc.stream = stream;
  cc.attrs = attr;
  cc.numAttrs = 1;
  return cudaLaunchKernelEx(&cc, attn_combine_kernel, (const float*)part, p.split, p.out);
}

}  // namespace csa2
