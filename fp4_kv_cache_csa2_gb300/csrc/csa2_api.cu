// C ABI of the CSA2 layer: argument checks, workspace carving and launches.
// The operations themselves are defined in include/csa2.h.
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "common.cuh"
#include "host_once.cuh"
#include "params.cuh"

using namespace csa2;

namespace {

constexpr size_t HDR = CSA2_WS_HEADER_BYTES;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }


csa2_status check_cache(const csa2_cache* c) {
  if (!c || !c->main_kv || !c->idx_codes || !c->idx_scales || !c->n_entries) return CSA2_ERR_INVALID_ARG;
  if (c->cap < 0 || (c->cap % BLK) != 0) return CSA2_ERR_INVALID_ARG;
  if (c->m != 1 && c->m != 2) return CSA2_ERR_UNSUPPORTED;
  if (!aligned16(c->main_kv) || !aligned16(c->idx_codes) || !aligned16(c->idx_scales)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

csa2_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return CSA2_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255u) != 0) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < need) return CSA2_ERR_WORKSPACE;
  return CSA2_OK;
}

csa2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

WsHeader* header(void* ws) { return reinterpret_cast<WsHeader*>(ws); }
unsigned char* scratch(void* ws) { return reinterpret_cast<unsigned char*>(ws) + HDR; }

size_t gkeys_bytes(int B, int Q, int64_t max_n) {
  return align256((size_t)B * Q * (size_t)ceil_div(max_n, BLK) * sizeof(uint32_t));
}

bool long_rows(int64_t max_n) { return max_n > ROW_SELECT_MIN_KEYS; }

// scratch of the Full selections: per-row histograms and lists for long rows,
// block-maximum keys otherwise
size_t select_scratch_bytes(int B, int Q, int64_t max_n, bool blocks) {
  if (long_rows(max_n)) return align256(row_select_bytes((int64_t)B * Q));
  return blocks ? gkeys_bytes(B, Q, max_n) : 0;
}

// B * Q queries per call at most: every grid stays a 1-D grid below 2^31 CTAs
constexpr int64_t MAX_QUERIES = (int64_t)1 << 26;

csa2_status check_q(int B, int Q) {
  if (B < 0 || Q < 0) return CSA2_ERR_INVALID_ARG;
  if ((int64_t)B * Q > MAX_QUERIES) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

// ---------------------------------------------------------------- the calls
csa2_status do_index_score(const csa2_cache* cache, const uint16_t* q_idx, const float* w_head,
                           const int64_t* q_pos, const int32_t* pool, int M, float* scores, int B, int Q,
                           int64_t max_n, WsHeader* hdr, cudaStream_t stream) {
  IsParams p{};
  p.idx_codes = cache->idx_codes;
  p.idx_scales = cache->idx_scales;
  p.cap = cache->cap;
  p.n_entries = cache->n_entries;
  p.m = cache->m;
  p.q_idx = q_idx;
  p.w_head = w_head;
  p.q_pos = q_pos;
  p.pool = pool;
  p.M = M;
  p.scores = scores;
  p.B = B;
  p.Q = Q;
  p.max_n = max_n;
  p.hdr = hdr;
  return from_cuda(launch_index_score(p, stream));
}

csa2_status do_attention(const csa2_cache* cache, const uint16_t* q, const int32_t* sel, int K,
                         const uint16_t* swa, const int64_t* swa_base, int S, const int64_t* q_pos, float scale,
                         uint16_t* out, int B, int Q, void* part_ws, WsHeader* hdr, cudaStream_t stream,
                         const uint8_t* packed_in = nullptr, uint8_t* packed_out = nullptr, bool swa_fp8 = false,
                         int split = 1) {
  AttnParams p{};
  p.main_kv = cache->main_kv;
  p.cap = cache->cap;
  p.q = q;
  p.sel = sel;
  p.K = K;
  p.swa = swa;
  p.swa_base = swa_base;
  p.S = S;
  p.swa_fp8 = swa_fp8 ? 1 : 0;
  p.q_pos = q_pos;
  p.scale = scale;
  p.out = out;
  p.Q = Q;
  p.hdr = hdr;
  p.packed_in = packed_in;
  p.packed_out = packed_out;
  p.split = split;
  return from_cuda(launch_attention(p, B, reinterpret_cast<float*>(part_ws), stream));
}

}  // namespace

extern "C" {

int csa2_layout_version(void) { return CSA2_LAYOUT_VERSION; }

const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
    case CSA2_ERR_UNSUPPORTED: return "CSA2_ERR_UNSUPPORTED";
    case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
    case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT";
    case CSA2_ERR_BOUNDS: return "CSA2_ERR_BOUNDS";
  }
  return "CSA2_ERR_UNKNOWN";
}

csa2_status csa2_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  csa2_status st = check_ws(ws, ws_bytes, HDR);
  if (st != CSA2_OK) return st;
  return from_cuda(cudaMemsetAsync(ws, 0, HDR, (cudaStream_t)stream));
}

csa2_status csa2_sync_status(void* ws, void* stream, int64_t* detail) {
  if (!ws) return CSA2_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CSA2_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return CSA2_ERR_CUDA;
  if (detail) *detail = (int64_t)h.detail;
  if (h.status != 0) {
    if (cudaMemset(ws, 0, HDR) != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return (csa2_status)h.status;
}

csa2_status csa2_rope_table(float* cs, int64_t P, double theta) {
  if (!cs || P < 0) return CSA2_ERR_INVALID_ARG;
  double inv_freq[32];
  for (int i = 0; i < 32; i++) inv_freq[i] = std::pow(theta, -(double)(2 * i) / 64.0);
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 1;
  if (nt > 32) nt = 32;
  if (P < 65536) nt = 1;
  auto work = [&](int64_t p0, int64_t p1) {
    for (int64_t p = p0; p < p1; p++)
      for (int i = 0; i < 32; i++) {
        double ang = (double)p * inv_freq[i];
        cs[(p * 32 + i) * 2 + 0] = (float)std::cos(ang);
        cs[(p * 32 + i) * 2 + 1] = (float)std::sin(ang);
      }
  };
  std::vector<std::thread> th;
  int64_t per = (P + nt - 1) / nt;
  for (unsigned k = 0; k < nt; k++) {
    int64_t a = k * per, b = std::min<int64_t>(P, a + per);
    if (a >= b) break;
    th.emplace_back(work, a, b);
  }
  for (auto& x : th) x.join();
  return CSA2_OK;
}

csa2_status csa2_compress_quantize(const csa2_cache* cache, const uint16_t* x, int B, int T,
                                   const int64_t* entry_start, const float* w0, const float* w1,
                                   const float* rope_cs, int64_t rope_P, const uint16_t* w_idx, void* ws,
                                   size_t ws_bytes, void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if (B < 0 || T < 0 || rope_P < 0) return CSA2_ERR_INVALID_ARG;
  if (T % cache->m != 0) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return check_ws(ws, ws_bytes, HDR);
  if (!x || !entry_start || !rope_cs || !w_idx) return CSA2_ERR_INVALID_ARG;
  if (cache->m == 2 && (!w0 || !w1)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(rope_cs) || !aligned16(w_idx)) return CSA2_ERR_INVALID_ARG;
  if (cache->m == 2 && (!aligned16(w0) || !aligned16(w1))) return CSA2_ERR_INVALID_ARG;
  st = check_ws(ws, ws_bytes, HDR);
  if (st != CSA2_OK) return st;
  CwParams p{};
  p.main_kv = cache->main_kv;
  p.idx_codes = cache->idx_codes;
  p.idx_scales = cache->idx_scales;
  p.cap = cache->cap;
  p.m = cache->m;
  p.x = x;
  p.B = B;
  p.T = T;
  p.entry_start = entry_start;
  p.w0 = w0;
  p.w1 = w1;
  p.rope_cs = rope_cs;
  p.rope_P = rope_P;
  p.w_idx = w_idx;
  p.hdr = header(ws);
  int sms = 0;
  if (device_sms(&sms) != cudaSuccess) return CSA2_ERR_CUDA;
  return from_cuda(launch_cache_write(p, (cudaStream_t)stream, sms));
}

csa2_status csa2_index_score(const csa2_cache* cache, const uint16_t* q_idx, const float* w_head,
                             const int64_t* q_pos, const int32_t* pool_blocks, int M, float* scores, int B, int Q,
                             int64_t max_n, void* ws, size_t ws_bytes, void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if ((st = check_q(B, Q)) != CSA2_OK) return st;
  if (max_n < 0) return CSA2_ERR_INVALID_ARG;
  if (pool_blocks && (M < 1 || M > CSA2_MAX_M)) return CSA2_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, HDR)) != CSA2_OK) return st;
  if (B == 0 || Q == 0) return CSA2_OK;
  if (!q_idx || !w_head || !q_pos || !scores) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q_idx)) return CSA2_ERR_INVALID_ARG;
  return do_index_score(cache, q_idx, w_head, q_pos, pool_blocks, M, scores, B, Q, max_n, header(ws),
                        (cudaStream_t)stream);
}

size_t csa2_block_topk_workspace_size(int B, int Q, int64_t max_n) {
  if (B < 0 || Q < 0 || max_n < 0) return 0;
  return HDR + select_scratch_bytes(B, Q, max_n, true);
}

csa2_status csa2_block_topk(const csa2_cache* cache, const float* scores, const int64_t* q_pos, int B, int Q,
                            int64_t max_n, int M, int32_t* pool_blocks, void* ws, size_t ws_bytes, void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if ((st = check_q(B, Q)) != CSA2_OK) return st;
  if (max_n < 0) return CSA2_ERR_INVALID_ARG;
  if (M < 1 || M > CSA2_MAX_M) return CSA2_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, csa2_block_topk_workspace_size(B, Q, max_n))) != CSA2_OK) return st;
  if (B == 0 || Q == 0) return CSA2_OK;
  if (!scores || !q_pos || !pool_blocks) return CSA2_ERR_INVALID_ARG;
  if (long_rows(max_n))
    return from_cuda(launch_row_select(scores, q_pos, cache->n_entries, cache->m, B, Q, max_n, 0, nullptr, M,
                                       pool_blocks, scratch(ws), (cudaStream_t)stream));
  return from_cuda(launch_block_topk(scores, q_pos, cache->n_entries, cache->m, B, Q, max_n, M, pool_blocks,
                                     reinterpret_cast<uint32_t*>(scratch(ws)), (cudaStream_t)stream));
}

size_t csa2_select_topk_workspace_size(int B, int Q, int64_t max_n) {
  if (B < 0 || Q < 0 || max_n < 0) return 0;
  return HDR + select_scratch_bytes(B, Q, max_n, false);
}

csa2_status csa2_select_topk(const csa2_cache* cache, const float* scores, const int64_t* q_pos,
                             const int32_t* pool_blocks, int M, int K, int32_t* sel, int B, int Q, int64_t max_n,
                             void* ws, size_t ws_bytes, void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if ((st = check_q(B, Q)) != CSA2_OK) return st;
  if (max_n < 0) return CSA2_ERR_INVALID_ARG;
  if (K < 1 || K > CSA2_MAX_K) return CSA2_ERR_UNSUPPORTED;
  if (pool_blocks && (M < 1 || M > CSA2_MAX_M)) return CSA2_ERR_UNSUPPORTED;
  const size_t need = pool_blocks ? HDR : csa2_select_topk_workspace_size(B, Q, max_n);
  if ((st = check_ws(ws, ws_bytes, need)) != CSA2_OK) return st;
  if (B == 0 || Q == 0) return CSA2_OK;
  if (!scores || !q_pos || !sel) return CSA2_ERR_INVALID_ARG;
  if (!pool_blocks && long_rows(max_n))
    return from_cuda(launch_row_select(scores, q_pos, cache->n_entries, cache->m, B, Q, max_n, K, sel, 0, nullptr,
                                       scratch(ws), (cudaStream_t)stream));
  return from_cuda(launch_select_topk(scores, q_pos, cache->n_entries, cache->m, pool_blocks, M, K, sel, B, Q,
                                      max_n, (cudaStream_t)stream));
}

csa2_status csa2_swa_quantize_fp8(const uint16_t* x, int64_t n_rows, uint8_t* out, void* stream) {
  if (n_rows < 0) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return CSA2_ERR_INVALID_ARG;
  return from_cuda(launch_swa_fp8(x, n_rows, out, (cudaStream_t)stream));
}

size_t csa2_attn_workspace_size(int B, int Q, int K) {
  if (B < 0 || Q < 0 || K < 0) return 0;
  return HDR + align256(attn_partials_bytes((int64_t)B * Q, K));
}

csa2_status csa2_sparse_swa_attn(const csa2_cache* cache, const uint16_t* q, const int32_t* sel, int K,
                                 const uint16_t* swa, const int64_t* swa_base_pos, int S, const int64_t* q_pos,
                                 float scale, uint16_t* out, int B, int Q, void* ws, size_t ws_bytes,
                                 void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if ((st = check_q(B, Q)) != CSA2_OK) return st;
  if (K < 0 || K > CSA2_MAX_K) return CSA2_ERR_UNSUPPORTED;
  if (S < 0 || !std::isfinite(scale)) return CSA2_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, csa2_attn_workspace_size(B, Q, K))) != CSA2_OK) return st;
  if (B == 0 || Q == 0) return CSA2_OK;
  if (!q || (K > 0 && !sel) || !swa || !swa_base_pos || !q_pos || !out) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(swa) || !aligned16(out)) return CSA2_ERR_INVALID_ARG;
  return do_attention(cache, q, sel, K, swa, swa_base_pos, S, q_pos, scale, out, B, Q, scratch(ws), header(ws),
                      (cudaStream_t)stream);
}

csa2_status csa2_block_summary(const csa2_cache* cache, const int64_t* first_block, int64_t n_blocks, int B,
                               uint8_t* sum_codes, uint8_t* sum_scales, int64_t sum_cap, void* ws, size_t ws_bytes,
                               void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if (B < 0 || n_blocks < 0 || sum_cap < 0) return CSA2_ERR_INVALID_ARG;
  if ((sum_cap % BLK) != 0) return CSA2_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, HDR)) != CSA2_OK) return st;
  if (B == 0 || n_blocks == 0) return CSA2_OK;
  if (!first_block || !sum_codes || !sum_scales) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(sum_codes) || !aligned16(sum_scales)) return CSA2_ERR_INVALID_ARG;
  HsParams p{};
  p.idx_codes = cache->idx_codes;
  p.idx_scales = cache->idx_scales;
  p.cap = cache->cap;
  p.n_entries = cache->n_entries;
  p.first_block = first_block;
  p.B = B;
  p.n_blocks = n_blocks;
  p.sum_codes = sum_codes;
  p.sum_scales = sum_scales;
  p.sum_cap = sum_cap;
  p.hdr = header(ws);
  return from_cuda(launch_block_summary(p, (cudaStream_t)stream));
}

// HISA keeps up to 2048 of its summary rows: past 4096 blocks a row goes to
// the multi-CTA selection (a single CTA spends most of its time on the
// output once M is a large part of the row)
constexpr int64_t HISA_ROW_SELECT_MIN = 4096;
bool hisa_long_rows(int64_t nb) { return nb > HISA_ROW_SELECT_MIN; }

size_t csa2_hisa_blocks_workspace_size(int B, int Q, int64_t max_n) {
  if (B < 0 || Q < 0 || max_n < 0) return 0;
  const int64_t nb = ceil_div(max_n, BLK);
  return HDR + align256((size_t)B * Q * sizeof(int64_t)) + align256((size_t)B * sizeof(int32_t)) +
         align256((size_t)B * Q * nb * sizeof(float)) +
         (hisa_long_rows(nb) ? align256(row_select_bytes((int64_t)B * Q)) : 0);
}

csa2_status csa2_hisa_blocks(const csa2_cache* cache, const uint8_t* sum_codes, const uint8_t* sum_scales,
                             int64_t sum_cap, const uint16_t* q_idx, const float* w_head, const int64_t* q_pos,
                             int B, int Q, int64_t max_n, int M, int32_t* pool_blocks, void* ws, size_t ws_bytes,
                             void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if ((st = check_q(B, Q)) != CSA2_OK) return st;
  if (max_n < 0 || sum_cap < 0 || (sum_cap % BLK) != 0) return CSA2_ERR_INVALID_ARG;
  if (M < 1 || M > CSA2_MAX_M) return CSA2_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, csa2_hisa_blocks_workspace_size(B, Q, max_n))) != CSA2_OK) return st;
  if (B == 0 || Q == 0) return CSA2_OK;
  if (!sum_codes || !sum_scales || !q_idx || !w_head || !q_pos || !pool_blocks) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(sum_codes) || !aligned16(sum_scales) || !aligned16(q_idx)) return CSA2_ERR_INVALID_ARG;
  // rows past the summary store cannot be scored
  if (ceil_div(cache->cap, BLK) > sum_cap) return CSA2_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  WsHeader* hdr = header(ws);
  unsigned char* cur = scratch(ws);
  const int64_t nb = ceil_div(max_n, BLK);
  HvParams vp{};
  vp.q_pos = q_pos;
  vp.n_entries = cache->n_entries;
  vp.m = cache->m;
  vp.B = B;
  vp.Q = Q;
  vp.cap = cache->cap;
  vp.max_n = max_n;
  vp.view_pos = reinterpret_cast<int64_t*>(cur);
  cur += align256((size_t)B * Q * sizeof(int64_t));
  vp.view_n = reinterpret_cast<int32_t*>(cur);
  cur += align256((size_t)B * sizeof(int32_t));
  float* scores = reinterpret_cast<float*>(cur);
  cur += align256((size_t)B * Q * nb * sizeof(float));
  st = from_cuda(launch_hisa_view(vp, s));
  if (st != CSA2_OK) return st;
  // the summary store read as an m = 1 cache of ceil(n / 8) rows per sequence
  csa2_cache view{};
  view.main_kv = cache->main_kv;
  view.idx_codes = const_cast<uint8_t*>(sum_codes);
  view.idx_scales = const_cast<uint8_t*>(sum_scales);
  view.cap = sum_cap;
  view.n_entries = vp.view_n;
  view.m = 1;
  st = do_index_score(&view, q_idx, w_head, vp.view_pos, nullptr, M, scores, B, Q, nb, hdr, s);
  if (st != CSA2_OK) return st;
  if (hisa_long_rows(nb))
    return from_cuda(launch_row_select(scores, vp.view_pos, vp.view_n, 1, B, Q, nb, M, pool_blocks, 0, nullptr,
                                       cur, s));
  return from_cuda(launch_select_topk(scores, vp.view_pos, vp.view_n, 1, nullptr, M, M, pool_blocks, B, Q, nb, s));
}

size_t csa2_decode_workspace_size(csa2_mode mode, int B, int Q, int64_t max_n, int M, int K) {
  if (B < 0 || Q < 0 || max_n < 0 || M < 0 || K < 0) return 0;
  size_t need = HDR + align256(attn_partials_bytes((int64_t)B * Q, K));
  if (mode == CSA2_MODE_FULL) {
    need += align256((size_t)B * Q * max_n * sizeof(float)) + select_scratch_bytes(B, Q, max_n, true);
  } else if (mode == CSA2_MODE_REINDEX) {
    need += align256((size_t)B * Q * M * BLK * sizeof(float));
  }
  return need;
}

csa2_status csa2_decode(const csa2_cache* cache, const csa2_decode_args* a, void* ws, size_t ws_bytes,
                        void* stream) {
  csa2_status st = check_cache(cache);
  if (st != CSA2_OK) return st;
  if (!a) return CSA2_ERR_INVALID_ARG;
  if (a->mode != CSA2_MODE_FULL && a->mode != CSA2_MODE_REINDEX && a->mode != CSA2_MODE_REUSE)
    return CSA2_ERR_INVALID_ARG;
  if ((st = check_q(a->B, a->Q)) != CSA2_OK) return st;
  if (a->K < 1 || a->K > CSA2_MAX_K) return CSA2_ERR_UNSUPPORTED;
  if (a->mode != CSA2_MODE_REUSE && (a->M < 1 || a->M > CSA2_MAX_M)) return CSA2_ERR_UNSUPPORTED;
  if (a->S < 0 || a->max_n < 0 || !std::isfinite(a->scale)) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2_decode_workspace_size(a->mode, a->B, a->Q, a->max_n, a->M, a->K);
  if ((st = check_ws(ws, ws_bytes, need)) != CSA2_OK) return st;
  if (a->B == 0 || a->Q == 0) return CSA2_OK;
  if (!a->q_pos || !a->q || !a->swa || !a->swa_base_pos || !a->sel || !a->out) return CSA2_ERR_INVALID_ARG;
  if (a->mode != CSA2_MODE_REUSE && (!a->q_idx || !a->w_head || !a->pool_blocks)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(a->q) || !aligned16(a->swa) || !aligned16(a->out)) return CSA2_ERR_INVALID_ARG;
  if (a->mode != CSA2_MODE_REUSE && !aligned16(a->q_idx)) return CSA2_ERR_INVALID_ARG;
  if (a->packed_sel && !aligned16(a->packed_sel)) return CSA2_ERR_INVALID_ARG;
  if (a->swa_fp8 != 0 && a->swa_fp8 != 1) return CSA2_ERR_INVALID_ARG;
  if (a->attn_split < 0) return CSA2_ERR_INVALID_ARG;
  const int split = a->attn_split > 1 ? a->attn_split : 1;
  if (split > 1 && (int64_t)a->B * a->Q > attn_split_max_queries()) return CSA2_ERR_UNSUPPORTED;
  const uint8_t* packed_in = a->mode == CSA2_MODE_REUSE ? a->packed_sel : nullptr;
  uint8_t* packed_out = a->mode == CSA2_MODE_REUSE ? nullptr : a->packed_sel;

  cudaStream_t s = (cudaStream_t)stream;
  WsHeader* hdr = header(ws);
  unsigned char* cur = scratch(ws);
  void* part = cur;
  cur += align256(attn_partials_bytes((int64_t)a->B * a->Q, a->K));
  if (a->mode == CSA2_MODE_FULL) {
    float* scores = reinterpret_cast<float*>(cur);
    cur += align256((size_t)a->B * a->Q * a->max_n * sizeof(float));
    uint32_t* gkeys = reinterpret_cast<uint32_t*>(cur);
    st = do_index_score(cache, a->q_idx, a->w_head, a->q_pos, nullptr, a->M, scores, a->B, a->Q, a->max_n, hdr, s);
    if (st != CSA2_OK) return st;
    if (long_rows(a->max_n)) {
      st = from_cuda(launch_row_select(scores, a->q_pos, cache->n_entries, cache->m, a->B, a->Q, a->max_n, a->K,
                                       a->sel, a->M, a->pool_blocks, cur, s));
      if (st != CSA2_OK) return st;
      return do_attention(cache, a->q, a->sel, a->K, a->swa, a->swa_base_pos, a->S, a->q_pos, a->scale, a->out,
                          a->B, a->Q, part, hdr, s, packed_in, packed_out, a->swa_fp8 != 0, split);
    }
    st = from_cuda(launch_block_topk(scores, a->q_pos, cache->n_entries, cache->m, a->B, a->Q, a->max_n, a->M,
                                     a->pool_blocks, gkeys, s));
    if (st != CSA2_OK) return st;
    st = from_cuda(launch_select_topk(scores, a->q_pos, cache->n_entries, cache->m, nullptr, a->M, a->K, a->sel,
                                      a->B, a->Q, a->max_n, s));
    if (st != CSA2_OK) return st;
  } else if (a->mode == CSA2_MODE_REINDEX) {
    IsParams ip{};
    ip.idx_codes = cache->idx_codes;
    ip.idx_scales = cache->idx_scales;
    ip.cap = cache->cap;
    ip.n_entries = cache->n_entries;
    ip.m = cache->m;
    ip.q_idx = a->q_idx;
    ip.w_head = a->w_head;
    ip.q_pos = a->q_pos;
    ip.pool = a->pool_blocks;
    ip.M = a->M;
    ip.B = a->B;
    ip.Q = a->Q;
    ip.max_n = a->max_n;
    ip.sel = a->sel;
    ip.K = a->K;
    ip.hdr = hdr;
    ip.scores = reinterpret_cast<float*>(cur);                   // the pool slots' keys
    st = from_cuda(launch_reindex_select(ip, s));
    if (st != CSA2_OK) return st;
  }
  return do_attention(cache, a->q, a->sel, a->K, a->swa, a->swa_base_pos, a->S, a->q_pos, a->scale, a->out, a->B,
                      a->Q, part, hdr, s, packed_in, packed_out, a->swa_fp8 != 0, split);
}

}  // extern "C"
