/*
 * sparse_mla.h -- C ABI of the GB300 (sm_103a) sparse-MLA paged decode library.
 *
 * One decode query per request b: H query heads attend over the top-k tokens an
 * indexer selected for b.  The tokens live in a paged FP8 latent cache; each
 * is gathered through the block table and dequantised, then S = q.k (576
 * dims: 512 latent + 64 rope), softmax and O = P.v (512 latent dims) run,
 * split over the top-k list with a log-sum-exp merge of the partial results.
 *
 * Sources (page titles and sections of the pages this library follows):
 *   - "Inside the Decode Performance Investigation: How One Session Cracked the
 *     Occupancy Ceiling on Blackwell GPUs", Setup (64 query heads,
 *     index_topk = 512, sparse MLA attention) and Task 1 (split kernel with
 *     nsplit splits and a combine; attention stalls on scattered FP8
 *     page-gathers).
 *   - "The 64-Block Barrier", "The Smoking Gun: Grid = (B, H)" (each block
 *     walks the top-k tokens: gather, multiply, accumulate) and "The Split-K
 *     Prescription" (split the top-k set across blocks; merge the partials
 *     with an online-softmax merge).
 *   - "The Commit That Rewrote the Bottleneck", "The Levers" (wave-aware split
 *     count: the grid should be a near multiple of the SM count).
 *
 * Conventions for every entry point:
 *   - Device pointers are caller-owned CUDA device memory, 16-byte aligned,
 *     dense row-major.  The library never allocates device memory and never
 *     synchronises the stream (except sparse_mla_read_errors), so every call
 *     except that one can be captured into a CUDA graph.
 *   - Work is enqueued on `stream` (NULL = legacy default stream).  A return
 *     of SMLA_OK means the work was enqueued; a fault inside a kernel shows up
 *     at the caller's next synchronisation.
 *   - Host-checkable errors (null pointers, unsupported shapes, small
 *     workspace) return a status and enqueue nothing.
 *   - Cache record (656 bytes per token, 64 tokens per page):
 *       bytes   0..511  latent, FP8 E4M3 (OCP "fn") codes
 *       bytes 512..527  4 little-endian fp32 scales; latent dim d uses scale[d/128]
 *       bytes 528..655  64 bf16 rope values
 *     k[d] = e4m3(code[d]) * scale[d/128] (d < 512), k[512+j] = rope[j];
 *     v = k[0..511].
 *   - A top-k entry t of request b is a logical token position.  It is used
 *     when 0 <= t < seq_lens[b]; its row is block_table[b][t/64]*64 + t%64.
 *     Other entries (-1 padding, t >= seq_lens[b]) are skipped.  An entry
 *     below seq_lens[b] whose logical page is >= max_pages_per_seq or whose
 *     physical page is outside [0, num_pages) is skipped too and sets
 *     SMLA_DEVERR_PAGE_RANGE in the workspace error word.  Duplicated entries
 *     count once per occurrence.
 *   - Outputs: out[b][h][0..511] (bf16) = sum_t softmax_t(s) v_t and
 *     lse[b][h] (fp32) = ln sum_t exp(s_t), s_t = sm_scale * q[b][h].k_t.  A
 *     request with no valid entry gets out = 0 and lse = -inf.
 *   - Numerics: dequantised K/V and the softmax weights are fp16 on chip,
 *     accumulation is fp32.  |q| and |dequantised latent| must stay below
 *     65504; larger values saturate and set SMLA_DEVERR_RANGE.
 */
#ifndef SPARSE_MLA_H
#define SPARSE_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* smla_stream_t;

typedef enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, negative size              */
  SMLA_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement               */
  SMLA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required             */
  SMLA_ERR_CUDA = 4           /* a CUDA runtime call or a kernel launch failed          */
} smla_status;

/* Bits of the device error word kept at the start of the workspace.  They are
 * OR-ed in by the kernels and stay set until sparse_mla_clear_errors(). */
#define SMLA_DEVERR_PAGE_RANGE 0x1u  /* a used top-k entry mapped outside the block table or cache */
#define SMLA_DEVERR_TIMEOUT    0x2u  /* an internal wait gave up; that call's results are invalid  */
#define SMLA_DEVERR_RANGE      0x4u  /* q or a dequantised latent exceeded the fp16 range          */
#define SMLA_DEVERR_LEN_RANGE  0x8u  /* a top-k selection length outside [0, num_cols] was clamped */

typedef struct smla_dims {
  int32_t batch;              /* B decode queries, 1 .. 65535                            */
  int32_t num_heads;          /* H in {16, 32, 64, 128}                                  */
  int32_t topk;               /* top-k entries per query, 1 .. 2048                      */
  int32_t page_size;          /* tokens per page; must be 64                             */
  int32_t max_pages_per_seq;  /* row length of block_table, >= 1                         */
  int32_t d_latent;           /* must be 512                                             */
  int32_t d_rope;             /* must be 64                                              */
  int32_t nsplit;             /* partitions of the top-k list; 0 = scheduler's choice    */
  int64_t num_pages;          /* pages in kv_cache, >= 1                                 */
  int32_t heads_per_cta;      /* heads per CTA of the split kernel: 16, 32 or 64; 0 =    */
                              /* scheduler's choice                                      */
  int32_t queries_per_request;/* s_q >= 1 (0 means 1): query b reads block_table row     */
                              /* b / s_q (several queries of one request, each with its  */
                              /* own top-k and seq_lens entry); batch must be a multiple */
  int32_t merge;              /* how partitions are merged when nsplit > 1: 0 = the      */
                              /* scheduler's choice, 1 = the merge kernel, 2 = inside    */
                              /* the split kernel (a cluster of the nsplit CTAs; needs   */
                              /* nsplit <= 8 dividing heads_per_cta <= H, else           */
                              /* SMLA_ERR_UNSUPPORTED)                                   */
} smla_dims;

typedef struct smla_plan {
  int32_t nsplit;             /* partitions of the top-k list                            */
  int32_t tokens_per_split;   /* top-k entries per partition (last may be shorter)       */
  int32_t head_groups;        /* groups of heads_per_cta heads per (query, partition)    */
  int32_t ctas;               /* grid size of the split kernel: one CTA per (query,      */
                              /* partition, head group)                                  */
  int32_t ctas_per_sm;        /* CTAs of the split kernel resident per SM                */
  int32_t sm_count;           /* SMs the plan was made for                               */
  double waves;               /* ctas / (sm_count * ctas_per_sm)                         */
  double est_us;              /* cost-model estimate of one call, microseconds           */
  size_t workspace_bytes;     /* bytes sparse_mla_decode needs with this plan            */
  int32_t heads_per_cta;      /* heads per CTA of the split kernel: 16, 32 or 64 (<= H)  */
  int32_t fused;              /* 1: the nsplit partitions of a (query, head group) run as */
                              /* one thread-block cluster and merge inside the split     */
                              /* kernel (no merge launch); 0: merge kernel when nsplit>1 */
} smla_plan;

/* Split-count scheduler, host only, no CUDA calls.  Chooses nsplit (unless
 * dims->nsplit > 0 fixes it) and the heads per CTA (unless
 * dims->heads_per_cta > 0 fixes it; chosen among 16, 32, 64 up to H) by
 * minimising a wave-quantised cost model over both: whole waves of CTAs on
 * sm_count SMs times the per-CTA time, plus the partial-result traffic and
 * the merge.  sparse_mla_decode and sparse_mla_split use the heads per CTA
 * this returns for their dims.  Returns
 * SMLA_ERR_INVALID_ARG for null pointers or sm_count < 1, SMLA_ERR_UNSUPPORTED
 * for shapes outside smla_dims' stated ranges.  "The Commit That Rewrote the
 * Bottleneck", "The Levers"; "Inside the Decode Performance Investigation",
 * Task 1. */
int sparse_mla_plan_for(const smla_dims* dims, int32_t sm_count, smla_plan* plan);

/* As sparse_mla_plan_for, with sm_count read from CUDA device `device`
 * (cudaDeviceGetAttribute; no allocation, no synchronisation).  Returns
 * SMLA_ERR_CUDA if the attribute query fails. */
int sparse_mla_plan(const smla_dims* dims, int32_t device, smla_plan* plan);

/* Workspace bytes sparse_mla_decode needs for `nsplit` partitions: a 256-byte
 * header (error word) plus, when nsplit > 1, fp32 partials o_part
 * [B][nsplit][H][512] and lse_part [B][nsplit][H].  Host only.  Returns 0 for
 * a null or invalid dims. */
size_t sparse_mla_workspace_size(const smla_dims* dims, int32_t nsplit);

/* Full decode: split kernel (a6) then, when nsplit > 1, the merge (a7).
 *   q           bf16 [B][H][576]
 *   kv_cache    uint8 [num_pages][64][656] (record layout above)
 *   block_table int32 [B / queries_per_request][max_pages_per_seq]
 *   topk_idx    int32 [B][topk]
 *   seq_lens    int32 [B]
 *   sm_scale    score scale (1/sqrt(576) for DeepSeek MLA)
 *   out         bf16 [B][H][512]        (written)
 *   lse         fp32 [B][H]             (written)
 *   workspace   >= sparse_mla_workspace_size(dims, plan.nsplit) bytes; its
 *               first 4 bytes are the device error word.  Concurrent calls
 *               must not share a workspace.
 * dims->nsplit = 0 lets the scheduler choose (sparse_mla_plan on the current
 * device).  Returns SMLA_ERR_WORKSPACE if workspace_bytes is too small. */
int sparse_mla_decode(const smla_dims* dims, const void* q, const void* kv_cache,
                      const int32_t* block_table, const int32_t* topk_idx,
                      const int32_t* seq_lens, float sm_scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, smla_stream_t stream);

/* Split step alone (a1..a6): partition s of query b covers top-k positions
 * [s*L, min((s+1)*L, topk)) with L = ceil(topk / nsplit).  Writes
 * o_part [B][nsplit][H][512] = that partition's normalised output (fp32) and
 * lse_part [B][nsplit][H] = its log-sum-exp (-inf when the partition holds no
 * valid entry, with o_part = 0).  err_word: device uint32 the kernel ORs
 * SMLA_DEVERR_* bits into (may be NULL).  "The 64-Block Barrier", "The
 * Split-K Prescription". */
int sparse_mla_split(const smla_dims* dims, int32_t nsplit, const void* q, const void* kv_cache,
                     const int32_t* block_table, const int32_t* topk_idx, const int32_t* seq_lens,
                     float sm_scale, float* o_part, float* lse_part, uint32_t* err_word,
                     smla_stream_t stream);

/* sparse_mla_decode that also reports the index -> address step (a1) as the
 * decode itself performed it: rows_out[b][i] (int64, [B][topk], 8-byte
 * aligned) receives the physical row (page * 64 + slot) whose record the split
 * kernel's gather warps loaded for top-k entry i of query b, or -1 for an
 * entry they skipped (rules above).  Every entry is written once per head
 * group (the same value).  Same launches as sparse_mla_decode, with the extra
 * stores; meant for checking that the decode gathers exactly the rows the
 * top-k list names ("Inside the Decode Performance Investigation", Task 1:
 * scattered FP8 page-gathers).  Returns SMLA_ERR_INVALID_ARG for a null or
 * misaligned rows_out, else as sparse_mla_decode. */
int sparse_mla_decode_rows(const smla_dims* dims, const void* q, const void* kv_cache,
                           const int32_t* block_table, const int32_t* topk_idx,
                           const int32_t* seq_lens, float sm_scale, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, int64_t* rows_out,
                           smla_stream_t stream);

/* Test hook for the split kernel's failure path: every wait of the kernel's
 * internal pipeline (one thread group waiting for another's shared-memory
 * tile, an MMA or a bulk copy) gives up after `ns` nanoseconds of the GPU's
 * global timer, sets SMLA_DEVERR_TIMEOUT and leaves that call's outputs
 * unwritten; the waits that drain in-flight MMAs and copies before the kernel
 * exits keep their own limit.  Applies to launches made after the call, from
 * every host thread.  ns = 0 restores the default (one second).  A limit far
 * below a tile's latency makes every launch fail: it exists to test that such
 * a failure is reported and leaves the context usable.  Host only; returns
 * SMLA_OK. */
int sparse_mla_debug_set_wait_limit(uint64_t ns);

/* Shapes of one KV append call. */
typedef struct smla_append_dims {
  int32_t tokens;             /* new tokens to write, >= 0                               */
  int32_t num_requests;       /* rows of block_table, >= 1                               */
  int32_t page_size;          /* tokens per page; must be 64                             */
  int32_t max_pages_per_seq;  /* row length of block_table, >= 1                         */
  int32_t d_latent;           /* must be 512                                             */
  int32_t d_rope;             /* must be 64                                              */
  int64_t num_pages;          /* pages in kv_cache, >= 1                                 */
} smla_append_dims;

/* FP8 KV append: the write side of the cache sparse_mla_decode reads (the
 * step before the decode: "Inside the Decode Performance Investigation",
 * Task 1, paged FP8 latent cache with per-block scales).  For every new token
 * i, with request r = requests[i] (or i when requests is NULL) and logical
 * position t = positions[i], writes the 656-byte record at page
 * block_table[r][t / 64], slot t % 64 of kv_cache:
 *   scale_j = fp32(amax_j / 448) over latent dims [128 j, 128 j + 128) (1 when
 *             the block is all zero), IEEE division;
 *   code_d  = E4M3(fp32(latent_d / scale_{d / 128})), round to nearest even,
 *             saturating to +-448;
 *   record  = [code x 512 | scale x 4 (fp32, little-endian) | rope x 64 (bf16)].
 *   latent      bf16 [tokens][512], rope bf16 [tokens][64] (16-byte aligned)
 *   block_table int32 [num_requests][max_pages_per_seq]
 *   requests    int32 [tokens] or NULL; positions int32 [tokens]
 *   kv_cache    uint8 [num_pages][64][656] (written; other records untouched)
 *   err_word    device uint32 (may be NULL): a token whose request, position
 *               or page is out of range is skipped and sets
 *               SMLA_DEVERR_PAGE_RANGE.
 * Tokens that map to the same record race (the last write wins).  Returns
 * SMLA_ERR_INVALID_ARG for null or misaligned pointers and bad shapes,
 * SMLA_ERR_UNSUPPORTED for page_size / d_latent / d_rope other than 64 / 512
 * / 64, SMLA_ERR_CUDA if the launch fails.  Asynchronous on `stream`. */
int sparse_mla_kv_append(const smla_append_dims* dims, const void* latent, const void* rope,
                         const int32_t* block_table, const int32_t* requests, const int32_t* positions,
                         void* kv_cache, uint32_t* err_word, smla_stream_t stream);

/* Shapes of one top-k selection call. */
typedef struct smla_topk_dims {
  int32_t batch;          /* queries (rows of scores), >= 0                               */
  int32_t num_cols;       /* scored positions per row, 1 .. 1048576                       */
  int64_t row_stride;     /* elements between consecutive rows of scores, >= num_cols     */
  int32_t k;              /* positions kept per query, 1 .. 2048                           */
  int32_t cluster_ctas;   /* CTAs per row: 0 = chosen by the library, else 1 .. 16         */
} smla_topk_dims;

/* Top-k selection over indexer scores: the step that produces topk_idx for
 * the decode ("Inside the Decode Performance Investigation", The Setup:
 * index_topk = 512 positions per query; the indexer launches of the per-step
 * kernel inventory).  For query b with len = seq_lens[b] (clamped to
 * [0, num_cols]; a clamped length sets SMLA_DEVERR_LEN_RANGE):
 *   len <= k: topk_idx[b] = 0, 1, ..., len - 1, then -1 up to k;
 *   len >  k: the k positions p < len of largest scores[b][p], ranked by IEEE
 *             754 totalOrder on the float32 patterns (-0 below +0, NaNs beyond
 *             the infinities by sign), equal patterns ranked by lower position
 *             first; written in increasing position order.
 *   scores   float32 [batch][row_stride] (4-byte aligned; 16-byte aligned with
 *            row_stride % 4 == 0 takes 16-byte loads), read only below len
 *   seq_lens int32 [batch]; topk_idx int32 [batch][k] (written)
 *   err_word device uint32 (may be NULL).
 * Returns SMLA_ERR_INVALID_ARG for null or misaligned pointers and bad
 * shapes, SMLA_ERR_UNSUPPORTED for num_cols > 1048576 or k > 2048 (or a fixed
 * cluster_ctas whose chunk exceeds 65536 positions), SMLA_ERR_CUDA if the
 * launch fails (clusters of more than 8 CTAs, used only for rows longer than
 * 524288 positions, need the device to co-schedule them).  Asynchronous on
 * `stream`. */
int sparse_mla_topk_select(const smla_topk_dims* dims, const float* scores, const int32_t* seq_lens,
                           int32_t* topk_idx, uint32_t* err_word, smla_stream_t stream);

/* The launch shape sparse_mla_topk_select uses for dims on a device with
 * sm_count SMs (host only, no CUDA call): clusters of *cluster_ctas CTAs,
 * each CTA holding *chunk_positions positions of one row (a multiple of 2048,
 * at most 65536, cluster_ctas x chunk_positions >= num_cols).  A row spans
 * at most one cluster; with a power-of-two cluster size and at most 2048
 * rows, rows that need fewer chunks than the cluster has CTAs share clusters
 * (packed by their chunk count on the device, from seq_lens).  dims->cluster_ctas > 0 is kept as
 * given.  Returns SMLA_ERR_INVALID_ARG for bad shapes or pointers,
 * SMLA_ERR_UNSUPPORTED when no shape fits. */
int sparse_mla_topk_plan_for(const smla_topk_dims* dims, int32_t sm_count, int32_t* cluster_ctas,
                             int32_t* chunk_positions);

/* Log-sum-exp merge (a7) of nsplit partials:
 *   lse[b][h] = ln sum_s exp(lse_part[b][s][h])   (-inf if every partial is -inf)
 *   out[b][h][d] = sum_s exp(lse_part[b][s][h] - lse[b][h]) * o_part[b][s][h][d]  (bf16; 0 if empty)
 * nsplit in [1, 64].  "The 64-Block Barrier", "The Split-K Prescription"
 * (online-softmax merge of the partial results). */
int sparse_mla_combine(int32_t batch, int32_t num_heads, int32_t nsplit, const float* o_part,
                       const float* lse_part, void* out, float* lse, smla_stream_t stream);

/* Index -> address step (a1) alone: rows_out[b][i] (int64) = physical row
 * block_table[b][t/64]*64 + t%64 of top-k entry t = topk_idx[b][i], or -1
 * when the entry is skipped (rules above).  "Inside the Decode Performance
 * Investigation", Task 1 (scattered FP8 page-gathers). */
int sparse_mla_gather_rows(const smla_dims* dims, const int32_t* block_table,
                           const int32_t* topk_idx, const int32_t* seq_lens, int64_t* rows_out,
                           smla_stream_t stream);

/* Zero the device error word of a workspace (enqueued on stream). */
int sparse_mla_clear_errors(void* workspace, smla_stream_t stream);

/* Copy the device error word of a workspace to *flags.  Synchronises `stream`;
 * not capturable. */
int sparse_mla_read_errors(const void* workspace, uint32_t* flags, smla_stream_t stream);

/* Static description of a status code. */
const char* sparse_mla_status_string(int status);

/* Decode that allocates nothing and needs no workspace argument.  The pages
 * have no counterpart: it exists for callers that cannot allocate device
 * memory -- plugins hosted by an engine that owns the whole device pool and
 * hands out no workspace, code running while a stream is being captured into
 * a CUDA graph, host paths that must not risk cudaMalloc's implicit device
 * synchronisation.  Same inputs, outputs and kernels as sparse_mla_decode;
 * the split partials and the device error word live in a file-scope device
 * array of 32 MiB (SMLA_NOALLOC_SCRATCH_BYTES) that every GPU loading the
 * library holds until the process exits.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, once per device, with that device current); make
 *     that first call before any stream capture on the device.
 *   - Shapes whose partials do not fit (sparse_mla_workspace_size > 32 MiB for
 *     the chosen nsplit) return SMLA_ERR_WORKSPACE and enqueue nothing; use
 *     sparse_mla_decode with a caller workspace or a smaller nsplit then.
 *   - No cudaMalloc, cudaFree or allocating library call is made.
 *   - Every call shares the array and leaves its contents behind: the error
 *     word is cleared at the start of each call and holds that call's
 *     SMLA_DEVERR_* bits afterwards (sparse_mla_noalloc_read_errors), and
 *     calls that overlap on the GPU (other streams, other threads) race on the
 *     array and must be ordered by the caller.
 *   - Dims are checked as sparse_mla_decode checks them, with the same status
 *     codes.
 *   - The device address is cached per device index for the life of the
 *     process; after cudaDeviceReset the library must not be called again. */
#define SMLA_NOALLOC_SCRATCH_BYTES (32u << 20)
int sparse_mla_decode_noalloc(const smla_dims* dims, const void* q, const void* kv_cache,
                              const int32_t* block_table, const int32_t* topk_idx, const int32_t* seq_lens,
                              float sm_scale, void* out, float* lse, smla_stream_t stream);

/* Copy the device error word of the last sparse_mla_decode_noalloc call on the
 * current device (SMLA_DEVERR_* bits) to *flags.  Enqueued on `stream`, then
 * synchronises it (not capturable); order it after that call.  No
 * allocation.  Returns SMLA_ERR_INVALID_ARG for a null flags, SMLA_ERR_CUDA if
 * the copy fails.  The pages have no counterpart: it completes the
 * workspace-free entry point above. */
int sparse_mla_noalloc_read_errors(uint32_t* flags, smla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H */
