// Launch parameters and launcher declarations shared by the CSA2 translation units.
#pragma once

#include "common.cuh"

namespace csa2 {

struct CwParams {
  uint8_t* main_kv;
  uint8_t* idx_codes;
  uint8_t* idx_scales;
  int64_t cap;
  int m;
  const uint16_t* x;        // [B][T][512]
  int B, T;
  const int64_t* entry_start;
  const float* w0;
  const float* w1;
  const float* rope_cs;     // [P][32][2]
  int64_t rope_P;
  const uint16_t* w_idx;    // [128][512]
  WsHeader* hdr;
};

struct IsParams {
  const uint8_t* idx_codes;
  const uint8_t* idx_scales;
  int64_t cap;
  const int32_t* n_entries;
  int m;
  const uint16_t* q_idx;      // [B][Q][32][128]
  const float* w_head;        // [B][Q][32]
  const int64_t* q_pos;       // [B][Q]
  const int32_t* pool;        // [B][Q][M] or null
  int M;
  float* scores;              // [B][Q][max_n] or [B][Q][M*8]
  int B, Q;
  int64_t max_n;
  int64_t entries_per_cta;    // set by the launcher
  int64_t group0;             // first query group of this launch (index scan; set by the launcher)
  int32_t* sel;               // fused Reindex: [B][Q][K] output
  int K;
  WsHeader* hdr;
  int test_withhold;          // test hook: the producer waits on a barrier nobody arrives on (0 = off)
};

struct AttnParams {
  const uint8_t* main_kv;
  int64_t cap;
  const uint16_t* q;          // [BQ][64][512]
  const int32_t* sel;         // [BQ][K]
  int K;
  const uint16_t* swa;        // [B][S][512] bf16, or E4M3 bytes when swa_fp8
  const int64_t* swa_base;    // [B]
  int S;
  int swa_fp8;
  const int64_t* q_pos;       // [BQ]
  float scale;
  uint16_t* out;              // [BQ][64][512]
  int Q;
  const uint8_t* packed_in;   // [BQ][K][288] selected entries to read instead of gathering, or null
  uint8_t* packed_out;        // [BQ][K][288] where to write the gathered selected entries, or null
  int split;                  // CTAs per query (1: the whole query in one CTA)
  float* opart;               // split > 1: the partial states, [BQ * split][2 * 64 + 64 * 512]
  WsHeader* hdr;
};

struct HsParams {             // HISA block summaries
  const uint8_t* idx_codes;
  const uint8_t* idx_scales;
  int64_t cap;
  const int32_t* n_entries;
  const int64_t* first_block; // [B]
  int B;
  int64_t n_blocks;           // blocks per sequence from first_block
  uint8_t* sum_codes;         // [B][sum_cap][64]
  uint8_t* sum_scales;        // [B][sum_cap][4]
  int64_t sum_cap;
  WsHeader* hdr;
};

struct HvParams {             // HISA view of the summary store as an m = 1 cache
  const int64_t* q_pos;       // [B][Q]
  const int32_t* n_entries;   // [B]
  int m, B, Q;
  int64_t cap, max_n;
  int64_t* view_pos;          // [B][Q] out
  int32_t* view_n;            // [B] out
};

cudaError_t launch_cache_write(const CwParams& p, cudaStream_t stream, int num_sms);
cudaError_t launch_swa_fp8(const uint16_t* x, int64_t n_rows, uint8_t* out, cudaStream_t stream);
cudaError_t launch_index_score(IsParams p, cudaStream_t stream);
cudaError_t launch_reindex_select(IsParams p, cudaStream_t stream);
cudaError_t launch_block_topk(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m,
                              int B, int Q, int64_t max_n, int M, int32_t* pool_blocks, uint32_t* gkeys,
                              cudaStream_t stream);
cudaError_t launch_select_topk(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m,
                               const int32_t* pool, int M, int K, int32_t* sel, int B, int Q, int64_t max_n,
                               cudaStream_t stream);
// Full rows longer than ROW_SELECT_MIN_KEYS entries are selected by the
// multi-CTA histogram/filter path, with row_select_bytes(B*Q) of scratch.
constexpr int64_t ROW_SELECT_MIN_KEYS = 16384;
size_t row_select_bytes(int64_t BQ);
cudaError_t launch_row_select(const float* scores, const int64_t* q_pos, const int32_t* n_entries, int m, int B,
                              int Q, int64_t max_n, int K, int32_t* sel, int M, int32_t* pool, void* scratch,
                              cudaStream_t stream);
cudaError_t launch_attention(AttnParams p, int B, float* partials, cudaStream_t stream);
size_t attn_partials_bytes(int64_t BQ, int K);
int attn_split_max_queries();
cudaError_t launch_block_summary(const HsParams& p, cudaStream_t stream);
cudaError_t launch_hisa_view(const HvParams& p, cudaStream_t stream);

}  // namespace csa2
