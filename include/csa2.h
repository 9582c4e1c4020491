/*
 * csa2.h — C ABI of the CSA2 global-attention layer for one GB300 (sm_103a).
 *
 * The layer (DeepSeek-V4.1-Flash, as described by the web pages
 * "DeepSeek-V4.1 Flash: 把 KV Cache 压缩推到极致" [zartbot] and
 * "4. 层维度(下):CSA2 与每 token 890 字节" [dilfish]) has three parts:
 *   (a) the cache write: per-channel learned-weight compressor, RMSNorm, RoPE on
 *       the 64-d tail, FP4 main KV (E2M1 + one E4M3 scale per 16 channels,
 *       288 B/entry) and the 128-d index K projected from it, stored as MXFP4
 *       (E2M1 + one E8M0 scale per 32, 68 B/entry);
 *   (b) the hierarchical lightning indexer: per-entry scores over 32 index heads,
 *       block-of-8 maxima, top-M candidate blocks, top-K entries;
 *   (c) one joint softmax attention of 64 query heads over the selected main-KV
 *       entries plus a 128-token bf16 sliding window, with key = value = the
 *       shared 512-d latent.
 * Decode layers run in Full, Reindex or Reuse mode ([zartbot] §2.3.2, §3.2).
 *
 * Conventions (all entry points):
 *   - Every tensor pointer is DEVICE memory owned by the caller, unless the
 *     argument says "host".  The library never allocates, frees or
 *     synchronises inside a call (except csa2_sync_status and csa2_rope_table,
 *     which is host-only).
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work; they are asynchronous and stream ordered.
 *   - The return value reports argument, configuration and launch errors.
 *     Errors that only the device can see (an index out of range, a window row
 *     the caller did not supply) are OR-ed into a status word inside the
 *     workspace `ws`; read and clear it with csa2_sync_status.
 *   - `ws` is caller-owned device scratch of `ws_bytes` bytes, 256-byte
 *     aligned, initialised once with csa2_workspace_init.  Its first
 *     CSA2_WS_HEADER_BYTES hold the status word.  Calls that overlap on the GPU
 *     must not share a workspace.
 *   - The library keeps no state between calls other than per-device launch
 *     attributes, set once per device under a lock, so any number of host
 *     threads may call it at once (each with its own workspace).  No C++
 *     exception crosses this boundary.
 *   - Sizes: K <= 512, M <= 2048, m in {1, 2}, B * Q <= 67,108,864 (2^26).
 *     Other values return CSA2_ERR_UNSUPPORTED.
 *   - Visibility: a query at raw token position t sees the entries
 *     j < min(n_entries[b], floor((t+1)/m)) and the window positions
 *     max(0, t-127) .. t ([dilfish] §4.2: an m=2 entry exists once both of its
 *     tokens do).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA2_LAYOUT_VERSION 1
#define CSA2_D_LATENT 512        /* head_dim: shared key/value latent          */
#define CSA2_D_ROPE 64           /* rope_head_dim: last 64 channels            */
#define CSA2_N_HEADS 64          /* n_heads: main query heads                  */
#define CSA2_N_INDEX_HEADS 32    /* index_n_heads                              */
#define CSA2_D_INDEX 128         /* index_head_dim                             */
#define CSA2_BLOCK 8             /* candidate_block_size                       */
#define CSA2_WINDOW 128          /* window_size                                */
#define CSA2_MAIN_ENTRY_BYTES 288
#define CSA2_INDEX_CODE_BYTES 64
#define CSA2_INDEX_SCALE_BYTES 4
#define CSA2_MAX_K 512
#define CSA2_ATTN_SPLIT_MAX_QUERIES 128   /* B * Q of a call whose attention may be split */
#define CSA2_MAX_M 2048
#define CSA2_WS_HEADER_BYTES 256

typedef enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned buffer */
    CSA2_ERR_UNSUPPORTED = 2,   /* m, K or M outside the supported set             */
    CSA2_ERR_WORKSPACE = 3,     /* ws missing or smaller than the call needs       */
    CSA2_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed            */
    CSA2_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up              */
    CSA2_ERR_BOUNDS = 6         /* device saw an index outside a buffer            */
} csa2_status;

typedef enum {
    CSA2_MODE_FULL = 0,         /* score all visible entries, publish pool + top-K */
    CSA2_MODE_REINDEX = 1,      /* score only the pool, publish own top-K          */
    CSA2_MODE_REUSE = 2         /* attend with the published top-K                 */
} csa2_mode;

/*
 * One source layer's global cache (caller-owned device memory).  [dilfish §4.4]
 *   main_kv     [B][cap][288]: bytes 0..255 E2M1 codes, channel 2k in the low
 *               nibble of byte k; bytes 256..287 one E4M3 scale per 16 channels.
 *   idx_codes   [B][cap][64]:  index K, E2M1 codes, dim 2k in the low nibble.
 *   idx_scales  [B][cap][4]:   index K, one E8M0 scale (2^(byte-127)) per 32 dims.
 *   cap         entries per sequence, a multiple of 8 (the candidate block size),
 *               so that every sequence and every block starts 16-byte aligned in
 *               all three arrays.
 *   n_entries   device [B]: entries valid per sequence (maintained by the caller).
 *   m           compression ratio of the source layer: 2 (Encoder) or 1 (Decoder).
 * All three arrays need 16-byte aligned base pointers.
 */
typedef struct {
    uint8_t *main_kv;
    uint8_t *idx_codes;
    uint8_t *idx_scales;
    int64_t cap;
    const int32_t *n_entries;
    int32_t m;
} csa2_cache;

/* Library version of the cache layout above (for callers that persist caches). */
int csa2_layout_version(void);

/* Human-readable name of a status code (static string). */
const char *csa2_status_string(csa2_status s);

/*
 * Writes the status header of a workspace (status word := 0).  Must be called
 * once before the first use of a workspace; enqueued on `stream`.
 */
csa2_status csa2_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * Synchronises `stream`, returns the device-side status word of `ws` (CSA2_OK
 * if no kernel reported an error since the last call) and clears it.  If
 * `detail` is not NULL it receives the first failing index the device recorded.
 */
csa2_status csa2_sync_status(void *ws, void *stream, int64_t *detail);

/*
 * RoPE table, host only: cs_host[(p*32 + i)*2 + {0,1}] = cos/sin of
 * p * theta^(-2i/64) evaluated in binary64 (pow, cos, sin of the C library)
 * and rounded to binary32, for p in [0, P).  Pairs (448+2i, 449+2i) of the
 * latent rotate with row p.  Copy it to the device once per model; theta is
 * compress_rope_theta = 160000 in the pages' configuration ([zartbot] §1.2).
 * Errors: INVALID_ARG for a null pointer or P < 0.
 */
csa2_status csa2_rope_table(float *cs_host, int64_t P, double theta);

/*
 * (a) Cache write.  [dilfish §4.2 compressor, §4.4 formats; zartbot §2.3.1
 * index K from main KV, §2.4.4 FP4 main KV quantised after RoPE]
 *   x            bf16 [B][T][512] raw latents of T consecutive tokens per
 *                sequence (T even when m = 2).
 *   entry_start  device int64 [B]: index of the first entry written per
 *                sequence; entry e = entry_start[b] + j pools tokens (2j, 2j+1)
 *                with c = (w0*x0 + w1*x1)/(w0 + w1) per channel (m = 2) or is
 *                token j (m = 1).  Its RoPE position is e.
 *   w0, w1       float [512] positive per-channel compressor weights (m = 2).
 *   rope_cs      float [rope_P][32][2] table from csa2_rope_table.
 *   w_idx        bf16 [128][512] index-K projection.
 * Per entry: RMSNorm (weight 1, eps 1e-6), rotate the 64-d tail, write the
 * 288-byte main entry and the 68-byte index entry (k = w_idx * latent before
 * quantisation).  Binary32 order is fixed so the bytes are reproducible (see
 * the CPU reference in the tests).  Entries with e >= cap or e >= rope_P are
 * skipped and raise CSA2_ERR_BOUNDS in the status word.  n_entries is not
 * modified.  Needs only the workspace header.
 */
csa2_status csa2_compress_quantize(const csa2_cache *cache, const uint16_t *x, int B, int T,
                                   const int64_t *entry_start, const float *w0,
                                   const float *w1, const float *rope_cs, int64_t rope_P,
                                   const uint16_t *w_idx, void *ws, size_t ws_bytes,
                                   void *stream);

/*
 * (b) Indexer scores.  s(t,j) = sum_h w_h * ReLU(q_h . k_j) over 32 heads
 * x 128 dims, with q_h quantised to MXFP4 like the keys.  [zartbot §2.3.4,
 * §3.3.2 (the formula itself is not legible on the pages; this is the
 * library's definition)]
 *   q_idx        bf16 [B][Q][32][128] index queries.
 *   w_head       float [B][Q][32] per-head weights.
 *   q_pos        int64 [B][Q] raw token positions of the queries.
 *   pool_blocks  NULL: score every visible entry; output scores [B][Q][max_n],
 *                entry j at column j for j < n_visible (other columns untouched).
 *                Otherwise int32 [B][Q][M] candidate block ids (-1 = none):
 *                output scores [B][Q][M*8], column 8i+r = entry
 *                8*pool_blocks[i]+r, -inf where that entry is not visible or
 *                the block id is -1.
 * Needs only the workspace header.
 */
csa2_status csa2_index_score(const csa2_cache *cache, const uint16_t *q_idx,
                             const float *w_head, const int64_t *q_pos,
                             const int32_t *pool_blocks, int M, float *scores, int B, int Q,
                             int64_t max_n, void *ws, size_t ws_bytes, void *stream);

/*
 * (b) HSI candidate blocks.  g_r = max of the scores of block r (entries
 * 8r..8r+7, invisible ones count as -inf); the block holding the newest
 * visible entry gets +inf; the M blocks with the largest g are kept, ties to
 * the lower block id.  [dilfish §4.7; zartbot §2.3.4]
 *   scores       float [B][Q][max_n] in the layout of csa2_index_score(NULL pool).
 *   pool_blocks  out int32 [B][Q][M]: chosen block ids ascending, -1 padded.
 * Workspace: csa2_block_topk_workspace_size (per-row histograms and lists
 * when max_n > 16384, the per-block maxima otherwise).
 */
size_t csa2_block_topk_workspace_size(int B, int Q, int64_t max_n);
csa2_status csa2_block_topk(const csa2_cache *cache, const float *scores, const int64_t *q_pos,
                            int B, int Q, int64_t max_n, int M, int32_t *pool_blocks,
                            void *ws, size_t ws_bytes, void *stream);

/*
 * Same result as csa2_block_topk, for callers that cannot allocate device
 * memory: for example a plugin running inside a host engine that owns every
 * byte of the GPU through its own allocator, or a latency-critical path where
 * a cudaMalloc (which may synchronise the device) is not allowed.  The pages
 * describe no such call; it exists only for this reason.
 *   - No workspace: the per-block maxima live in a 4 MiB array inside the
 *     library, so B * Q * ceil(max_n / 8) must not exceed 1,048,576 (e.g. 64
 *     queries over 131,072 entries).  Larger requests return
 *     CSA2_ERR_WORKSPACE before anything is enqueued.
 *   - The library allocates nothing here and calls no allocating routine; the
 *     array is loaded with the library and stays on every GPU that used it
 *     until the process exits.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: do not use this call
 *     on a device after cudaDeviceReset (or any teardown of its primary
 *     context) in the same process.
 *   - All calls share the one array and it keeps the previous call's contents
 *     (nothing in it needs to start at zero).  Calls that may overlap on the
 *     GPU (different streams without ordering, other threads, other processes
 *     sharing the context) race on it: serialise them.
 * Arguments and outputs are those of csa2_block_topk; device-side errors are
 * not reported (there is no status word), argument errors are returned.
 */
csa2_status csa2_block_topk_static(const csa2_cache *cache, const float *scores, const int64_t *q_pos,
                                   int B, int Q, int64_t max_n, int M, int32_t *pool_blocks, void *stream);

/*
 * (b) Top-K entries by (score desc, entry id asc).  [zartbot §2.3.4: the Full
 * layer takes its own top-K over every visible entry; Reindex layers choose
 * inside the candidate pool]
 *   pool_blocks  NULL: choose among all visible entries, scores in the
 *                [B][Q][max_n] layout.  Otherwise choose inside the pool,
 *                scores in the [B][Q][M*8] pool layout of csa2_index_score.
 *   sel          out int32 [B][Q][K]: entry ids ascending, -1 padded.
 * Workspace: the header in pool mode; csa2_select_topk_workspace_size(B, Q,
 * max_n) without a pool (per-row histograms and lists when max_n > 16384).
 */
size_t csa2_select_topk_workspace_size(int B, int Q, int64_t max_n);
csa2_status csa2_select_topk(const csa2_cache *cache, const float *scores,
                             const int64_t *q_pos, const int32_t *pool_blocks, int M, int K,
                             int32_t *sel, int B, int Q, int64_t max_n, void *ws,
                             size_t ws_bytes, void *stream);

/*
 * (c) Joint sparse + SWA attention.  o_h = sum_i softmax_i(scale * q_h . v_i) v_i
 * over the dequantised main-KV entries named by `sel` (-1 slots skipped) and
 * the window rows of positions max(0,t-127)..t; keys and values are the same
 * vectors.  [zartbot §3.3.2: SWA KV and the selected main KV in one sparse
 * attention; §3.3.2.1 key = value]
 *   q            bf16 [B][Q][64][512], already projected and rotated.
 *   sel          int32 [B][Q][K] entry ids (any order), -1 = empty slot.
 *   swa          bf16 [B][S][512] window rows; row r holds raw position
 *                swa_base_pos[b] + r.
 *   out          bf16 [B][Q][64][512].
 * A selected id >= cap, or a window position outside the supplied rows, is
 * skipped and raises CSA2_ERR_BOUNDS.  Workspace: csa2_attn_workspace_size.
 * Precision: both products run on f16 operands with fp32 accumulation.  The
 * dequantised FP4 keys and E4M3 window values are exact in f16; q and bf16
 * window rows are rounded to f16, which is exact for magnitudes in
 * [2^-14, 65504] (the layer's activations are expected inside f16's range;
 * larger magnitudes are not representable).  The probabilities are f16.
 */
size_t csa2_attn_workspace_size(int B, int Q, int K);
csa2_status csa2_sparse_swa_attn(const csa2_cache *cache, const uint16_t *q, const int32_t *sel,
                                 int K, const uint16_t *swa, const int64_t *swa_base_pos,
                                 int S, const int64_t *q_pos, float scale, uint16_t *out,
                                 int B, int Q, void *ws, size_t ws_bytes, void *stream);

/*
 * FP8 sliding-window rows.  [zartbot §2.4.4: the quantisation-sensitive SWA
 * KV keeps FP8 precision while the main KV is FP4]
 *   x      bf16 [n_rows][512] window rows.
 *   out    uint8 [n_rows][512]: out[r][c] = E4M3 of x[r][c], round to nearest
 *          even, saturating at +-448, no scale factor.
 * Both 16-byte aligned.  Errors: INVALID_ARG for null or misaligned pointers
 * or n_rows < 0.  Needs no workspace.
 */
csa2_status csa2_swa_quantize_fp8(const uint16_t *x, int64_t n_rows, uint8_t *out, void *stream);

/*
 * HISA block summaries.  [zartbot §2.3.4, the HISA paragraph: each block of
 * consecutive positions keeps the mean of its indexer keys, and a decode step
 * updates only the newest block]
 * Block r of sequence b covers entries [8r, min(8r + 8, n)), n =
 * min(n_entries[b], cap).  Its summary key is the mean of the entries'
 * dequantised index keys, computed in binary32 (the keys, exact in binary32,
 * added in entry order starting from +0, then one correctly rounded division
 * by the number of entries), stored as MXFP4 by the index-K rule.
 *   first_block  device int64 [B]: first block to compute per sequence.
 *   n_blocks     blocks computed per sequence: first_block[b] .. + n_blocks - 1.
 *   sum_codes    out [B][sum_cap][64], sum_scales out [B][sum_cap][4]: the
 *                summary of block r in row r (same format as idx_codes and
 *                idx_scales); both 16-byte aligned.
 *   sum_cap      rows per sequence, a multiple of 8, >= ceil(cap / 8).
 * Blocks with no entry (8r >= n, or r < 0) are skipped and not written; a
 * block r >= sum_cap, or n_entries[b] > cap, raises CSA2_ERR_BOUNDS in the
 * status word.  Needs only the workspace header.
 */
csa2_status csa2_block_summary(const csa2_cache *cache, const int64_t *first_block, int64_t n_blocks, int B,
                               uint8_t *sum_codes, uint8_t *sum_scales, int64_t sum_cap, void *ws,
                               size_t ws_bytes, void *stream);

/*
 * HISA candidate blocks (first stage).  Every block holding a visible entry
 * (r < ceil(nv / 8), nv = the query's visible entries, at most max_n) is
 * scored on its summary key with the indexer score of csa2_index_score, and
 * the M best blocks by (score desc, block id asc) are kept; no block is forced
 * in.  The second stage is a Reindex call (csa2_decode, mode REINDEX) given
 * these blocks as its pool.  [zartbot §2.3.4, the HISA paragraph]
 *   sum_codes, sum_scales, sum_cap  the summary store of csa2_block_summary,
 *                up to date for every visible block.
 *   q_idx, w_head, q_pos  as in csa2_index_score.
 *   pool_blocks  out int32 [B][Q][M]: chosen block ids ascending, -1 padded.
 * Workspace: csa2_hisa_blocks_workspace_size (per-query summary scores and,
 * when ceil(max_n / 8) > 4096, the long-row selection lists).
 * Errors: INVALID_ARG when sum_cap < ceil(cap / 8).
 */
size_t csa2_hisa_blocks_workspace_size(int B, int Q, int64_t max_n);
csa2_status csa2_hisa_blocks(const csa2_cache *cache, const uint8_t *sum_codes, const uint8_t *sum_scales,
                             int64_t sum_cap, const uint16_t *q_idx, const float *w_head, const int64_t *q_pos,
                             int B, int Q, int64_t max_n, int M, int32_t *pool_blocks, void *ws,
                             size_t ws_bytes, void *stream);

/*
 * One decode (or prefill-chunk) call of a CSA2 layer in a given mode.
 * [zartbot §3.2 access table; dilfish §4.3]
 *   Full:    scores every visible entry with q_idx/w_head, writes pool_blocks
 *            (top-M blocks) and sel (own top-K over all visible entries), attends.
 *   Reindex: scores only the pool_blocks' entries with its own q_idx/w_head,
 *            writes sel (top-K inside the pool), attends.
 *   Reuse:   attends with the given sel; q_idx, w_head and pool_blocks unused.
 * All pointer fields are device memory; shapes as in the calls above.
 * packed_sel (optional, NULL to skip) is a packed copy of the selected
 * entries, uint8 [B][Q][K][288], 16-byte aligned: a Full or Reindex call
 * writes the main-KV bytes of entry sel[b][q][k] to slot k (slots whose sel is
 * -1 hold unspecified bytes); a Reuse call given the sel of that call reads the
 * entries from there instead of gathering them from the cache.  The Reuse
 * layers that share a selection then read it contiguously; the result is the
 * same as without it as long as the cache entries named by sel are unchanged
 * in between (the caller's contract).
 * swa_fp8 = 1 reads the window rows as E4M3 bytes, uint8 [B][S][512] from
 * csa2_swa_quantize_fp8 (16-byte aligned); the attention takes their E4M3
 * values exactly.  Other values of swa_fp8 return CSA2_ERR_INVALID_ARG.
 * attn_split (appended last) chooses how the attention spreads a query over
 * CTAs.  0 or 1: one CTA per query walks the window and every run of 128
 * selected entries (the least SM time per query: for calls that run beside
 * others or fill the GPU).  S >= 2: the query's chunks (the window, then the
 * runs of 128 selected entries) are divided among S CTAs (at most one per
 * chunk; larger S is reduced to the chunk count), each keeping its own
 * softmax state, and a second kernel merges the states into the output
 * (the shortest call: for a call that alone leaves most SMs idle, such as a
 * small batch going through the layers one after another).  The merged
 * softmax is the same function of the scores up to rounding.  Split calls
 * need B * Q <= CSA2_ATTN_SPLIT_MAX_QUERIES (CSA2_ERR_UNSUPPORTED otherwise);
 * csa2_decode_workspace_size includes their partial states for such calls.
 * Negative values return CSA2_ERR_INVALID_ARG.
 */
typedef struct {
    csa2_mode mode;
    int B, Q;                   /* sequences, queries per sequence              */
    int M, K;                   /* candidate blocks, selected entries           */
    int S;                      /* window rows supplied per sequence            */
    int64_t max_n;              /* Full: score row length (>= max visible)      */
    float scale;                /* softmax scale, 1/sqrt(512) in the pages      */
    const int64_t *q_pos;       /* [B][Q]                                       */
    const uint16_t *q;          /* [B][Q][64][512]                              */
    const uint16_t *q_idx;      /* [B][Q][32][128]   Full, Reindex              */
    const float *w_head;        /* [B][Q][32]        Full, Reindex              */
    const uint16_t *swa;        /* [B][S][512]                                  */
    const int64_t *swa_base_pos;/* [B]                                          */
    int32_t *pool_blocks;       /* [B][Q][M]  Full: out, Reindex: in            */
    int32_t *sel;               /* [B][Q][K]  Full/Reindex: out, Reuse: in      */
    uint16_t *out;              /* [B][Q][64][512]                              */
    uint8_t *packed_sel;        /* [B][Q][K][288] or NULL: Full/Reindex out, Reuse in */
    int32_t swa_fp8;            /* 0: swa is bf16; 1: swa is E4M3 [B][S][512]   */
    int32_t attn_split;         /* CTAs per query in the attention (0 / 1: one) */
} csa2_decode_args;

size_t csa2_decode_workspace_size(csa2_mode mode, int B, int Q, int64_t max_n, int M, int K);
csa2_status csa2_decode(const csa2_cache *cache, const csa2_decode_args *args, void *ws,
                        size_t ws_bytes, void *stream);

/*
 * Test hook for the device-side timeout path; off unless a caller turns it on,
 * and never needed in production.  The pages have no counterpart.
 * While enabled (enable = 1) on the calling host thread, every index-scan
 * launch that thread makes (csa2_index_score, the scan of a Full decode)
 * first waits, with a short bound (1024 polls), on an mbarrier that no thread,
 * copy or MMA ever arrives on.  The wait gives up before the kernel has issued
 * any copy or MMA; the kernel then records CSA2_ERR_TIMEOUT (detail 2) in the
 * workspace status word, stops every warp role, frees its TMEM and returns,
 * leaving the context usable.  Its scores are not written.  enable = 0 turns
 * it off.  Errors: INVALID_ARG for any other value.
 */
csa2_status csa2_test_withhold_arrival(int enable);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */
