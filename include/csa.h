/*
 * csa.h -- C ABI of libcsa: the data-parallel hot path of DeepSeek-V4's hybrid
 * attention (CSA, compressed sparse attention, and HCA, heavily compressed
 * attention) on one B300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [report]  "DeepSeek-V4: Towards Highly Efficient Million-Token Context
 *             Intelligence" (cnblogs Chinese translation of the report):
 *             §2.3.1 CSA, §2.3.2 HCA, §2.3.3 other details, §2.3.4 efficiency,
 *             §3.5.1 KV cache layout, §4.2.1 model settings, §5.2.1 FP4 QAT.
 *   [hf]      "DeepSeek-V4: million-token context usable by agents"
 *             (translation of the Hugging Face blog post deepseekv4), section
 *             "Hybrid attention: CSA and HCA", Fig. 3 and Fig. 4.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every function returns an int status (enum csa_status).  No exception or
 *    abort crosses the ABI.  Arguments are validated on the host before any
 *    launch; a failed validation launches nothing.
 *  - Device pointers are plain pointers into the memory of the current CUDA
 *    device.  All work is enqueued asynchronously on the caller's stream; the
 *    functions never synchronize, allocate, or free.
 *  - Ownership: the caller allocates and owns every buffer (inputs, outputs,
 *    cache pools, page tables, workspaces).  The library's own state is a
 *    per-device cache of how many attention CTA clusters the device holds at
 *    once (looked up on first use) and the fixed array of
 *    csa_index_topk_noalloc.
 *  - Alignment: every device pointer must be 16-byte aligned (CSA_ERR_ALIGN);
 *    cache pools and workspaces must be 1024-byte aligned.
 *  - Tensors are dense row-major with the shapes stated; there are no strides
 *    (one exception: w of the indexer may be one vector shared by every row).
 *  - Positions are 0-based raw-token positions.  For a query at position t the
 *    visible compressed blocks are j < N_c(t) = floor((t + 1) / m): block j
 *    covers raw tokens [j m, (j + 1) m) and must end at or before t.
 *  - Device-side faults are never raised on purpose.  Kernels that detect a
 *    bad value at run time (a NaN index score, a selected index out of range,
 *    a page id outside the pool, a sequence index outside the batch, a
 *    bounded wait that ran out) skip the access and record a status code in
 *    the first 4 bytes of the workspace; csa_workspace_status() reads it back.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

typedef struct CUstream_st* csa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

#define CSA_ABI_VERSION 2

enum csa_status {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1, /* null pointer, bad enum, negative size, NaN score seen */
  CSA_ERR_SHAPE = 2,       /* sizes inconsistent or beyond what the kernels support */
  CSA_ERR_ALIGN = 3,       /* pointer not 16-byte (pool/workspace: 1024-byte) aligned */
  CSA_ERR_UNSUPPORTED = 4, /* valid but unimplemented dtype / shape combination */
  CSA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than *_workspace_size() */
  CSA_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
  CSA_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up (device status) */
};

enum csa_dtype {
  CSA_F32 = 0,
  CSA_BF16 = 1,
  CSA_E4M3 = 2, /* OCP FP8 E4M3 (finite max 448) */
  CSA_E2M1 = 3, /* FP4, two per byte, even element in the low nibble */
};

/* Flags shared by the calls that take a flags field.
 * CSA_FLAG_OVERLAP_PREVIOUS: the call's kernels may start while the kernel
 * launched just before them on the stream is still running (programmatic
 * dependent launch) and wait for it only before reading what it writes.
 * Before that wait they read the call's inputs, so the caller guarantees
 * that the previous kernel does not write them: for csa_index_score /
 * csa_index_topk the queries q, head weights w, pos and seq; for csa_attend /
 * hca_attend the queries q and seq; csa_compress (append) states its own
 * condition.  Without the flag the calls start after the previous kernel has
 * finished, as usual on a stream. */
enum csa_call_flags { CSA_FLAG_OVERLAP_PREVIOUS = 0x100, CSA_FLAG_AFTER_APPEND = 0x200 };
/* CSA_FLAG_AFTER_APPEND (csa_index_score / csa_index_topk; implies
 * CSA_FLAG_OVERLAP_PREVIOUS): the kernel launched just before the call is the
 * decode append of this key store ([report] §3.5.1), which writes at most the
 * last visible key of each query (block N_c(t) - 1).  The scoring then reads
 * every older key before it waits for that kernel, so the append is hidden
 * behind the key stream. */

/* The CUDA runtime's message for the error behind the calling thread's last
 * CSA_ERR_CUDA ("no error" if there was none).  Static string, never NULL. */
CSA_API const char* csa_last_cuda_error(void);
/* Returns CSA_ABI_VERSION. */
CSA_API int csa_abi_version(void);
/* Static string for a status code (never NULL). */
CSA_API const char* csa_status_string(int status);

/* ==========================================================================
 * Paged compressed cache  ([report] §3.5.1, §2.3.4; [hf] "Hybrid attention")
 * ==========================================================================
 * The classical part of the heterogeneous KV cache holds compressed entries in
 * fixed-size pages.  A page spans P entries; P must be a multiple of 128 so a
 * page covers a whole multiple of lcm(4, 128) raw tokens for both m = 4 and
 * m = 128 ([report] §3.5.1: raw tokens per block any multiple of lcm(m, m')).
 * Entry e of sequence b lives in page page_table[b * max_pages + e / P] at
 * slot e % P.  Pages are addressed by int32 page ids into one pool.
 *
 * KV pool (format CSA_KV_POOL_FP8): entries of D = 576 = 512 content + 64 RoPE
 * dims ([report] §2.3.4: content dims FP8, RoPE dims BF16).  One page is
 * csa_kv_page_bytes(P) = 644 * P bytes, structure of arrays:
 *     content  e4m3 [P][512]  at byte 0
 *     rope     bf16 [P][64]   at byte 512 * P
 *     scale    f32  [P]       at byte 640 * P
 * Entry value = (scale * e4m3(content), bf16(rope)).  On write, scale =
 * amax(content) / 448 (float32 IEEE division; 1 if that is 0) and
 * content code = e4m3_rne_satfinite(c / scale) (float32 division).
 *
 * Indexer-key pool, BF16 (format CSA_INDEX_POOL_BF16): keys of d_I = 128.
 * One page is 256 * P bytes, split into tiles of 128 entries (32 KiB each).
 * Inside a tile, dims [0, 64) and [64, 128) form two 16 KiB halves; in a half,
 * entry row r (0..127) occupies bytes [r * 128, r * 128 + 128) with its eight
 * 16-byte chunks permuted: dims 8c .. 8c+7 of the half sit in chunk c ^ (r % 8).
 * (The tensor-core 128-byte swizzle, so a tile can be copied to shared memory
 * as is.)  Byte offset of (entry slot s, dim d) in a page:
 *     (s / 128) * 32768 + (d / 64) * 16384 + (s % 128) * 128
 *       + ((((d % 64) / 8) ^ (s % 8)) * 16) + (d % 8) * 2
 *
 * Indexer-key pool, FP4 (format CSA_INDEX_POOL_E2M1): keys of d_I = 128 in
 * e2m1 with one e4m3 scale per 16 elements ([report] §5.2.1; the pages name
 * MXFP4, the workload definition fixes e2m1 with per-16 FP8 scales).  One page
 * is 72 * P bytes:  codes u8 [P][64] at byte 0 (element 2i in the low nibble
 * of byte i), scales e4m3 [P][8] at byte 64 * P.  On write, per block of 16:
 * s = e4m3_rne(amax / 6) (float32 division), element = e2m1_rne_satfinite(x / s)
 * with s decoded; a block whose s is 0 stores all-zero codes.
 *
 * State cache ([report] §3.5.1: preallocated state for the sliding window and
 * the uncompressed tail).  Per stream (KV or indexer key):
 *     ring      bf16 [B][R][dim], raw token at position p in slot p % R, R >= m
 *     tail_gate f32  [B][m][dim], gate logits of position p in slot p % m
 * The uncompressed tail's raw tokens are read from the ring (tail < m <= R).
 * For the KV stream R = 128 = W, so the same ring is the attention window.
 */
enum csa_format {
  CSA_FMT_DENSE_F32 = 0,      /* dense float32 [B][capacity][dim]        */
  CSA_FMT_DENSE_BF16 = 1,     /* dense bf16   [B][capacity][dim]         */
  CSA_FMT_KV_POOL_FP8 = 2,    /* KV pool above (dim must be 576)         */
  CSA_FMT_INDEX_POOL_BF16 = 3,/* BF16 indexer pool above (dim must be 128) */
  CSA_FMT_INDEX_POOL_E2M1 = 4,/* FP4 indexer pool above (dim must be 128)  */
};

/* Page sizes in bytes for P entries per page; 0 for an invalid P / format. */
CSA_API size_t csa_page_bytes(int32_t format, int32_t page_entries);

/* Where compressed entries go / come from. */
typedef struct csa_store {
  int32_t format;             /* enum csa_format */
  int32_t dim;                /* entry width (576 for the KV pool, 128 for indexer pools) */
  void* base;                 /* dense array or pool base */
  int32_t capacity;           /* dense: entries per sequence. pools: unused */
  int32_t page_entries;       /* pools: P (multiple of 128) */
  const int32_t* page_table;  /* pools: [B][max_pages] page ids */
  int32_t max_pages;          /* pools: row length of page_table */
  int32_t num_pages;          /* pools: pages in the pool; base holds num_pages * page bytes */
} csa_store;
/* Page ids and sequence indices are device data, so they are checked on the
 * device: a page id outside [0, num_pages) or a sequence index outside
 * [0, batch) is never dereferenced.  The access is skipped (a read gives
 * zeros, a write is dropped) and CSA_ERR_INVALID_ARG is recorded in the
 * call's status word; results of that call are then unspecified. */

/* Quantize float32 entries into a store.  src f32 [B][n][dim] -> entries
 * [first, first + n) of every sequence.  This is the write half of the
 * compressor ([report] §2.3.4 storage formats), exposed so callers can
 * populate caches.  Element-exact: the codes equal the formulas above. */
typedef struct csa_cache_write_params {
  uint32_t struct_size;
  int32_t batch, n, first;
  const float* src;
  csa_store dst;
  int32_t* status;            /* optional (NULL: none): device word that records a
                                 page id outside the pool (CSA_ERR_INVALID_ARG);
                                 a workspace's first word can serve */
} csa_cache_write_params;
CSA_API int csa_cache_write(const csa_cache_write_params* p, csa_stream_t stream);

/* ==========================================================================
 * Step 1: compressor  ([report] §2.3.1, §2.3.2; [hf] "Hybrid attention")
 * ==========================================================================
 * c_j[d] = sum_{i in block j} softmax_i(g_i[d] + bias[i - j m][d]) * k_i[d]
 * The softmax runs over the m positions of the block, per channel d, in
 * float32 (expf); a partial block stays in the tail.  In modes DENSE and
 * APPEND blocks do not overlap; the _AB modes below add CSA's overlap.
 *
 * mode CSA_COMPRESS_DENSE: whole sequences.  k, g: [B][n_tokens][dim] (k F32
 *   or BF16, g F32 or BF16); writes entries [0, n_tokens / m) of dst.
 * mode CSA_COMPRESS_APPEND: one decode step.  For every sequence b with
 *   L = seq_len[b] tokens so far: ring slot L % R <- k_new[b] (bf16),
 *   tail_gate slot L % m <- g_new[b]; if (L + 1) % m == 0 the block
 *   j = (L + 1) / m - 1 (positions L + 1 - m .. L, raw tokens from the ring)
 *   is pooled and written to dst entry j.  seq_len is not modified (the
 *   caller advances it), so repeating a call is idempotent.
 *   A block of m <= 16 tokens is pooled by one CTA per sequence; a larger one
 *   by a thread-block cluster of 8 CTAs per sequence (one channel slice
 *   each), which agree on the FP8 entry scale through distributed shared
 *   memory.  dim <= 640, and a multiple of 8 for m > 16 (CSA_ERR_SHAPE
 *   otherwise).
 * mode CSA_COMPRESS_WINDOW: one decode step of a layer without a compressed
 *   branch (pure sliding-window attention, [report] §4.2.1: the first layers
 *   of the Flash model): ring slot L % ring_size <- k_new[b]; m, bias, g_new,
 *   tail_gate and dst are not used.
 * mode CSA_COMPRESS_DENSE_AB / CSA_COMPRESS_APPEND_AB: overlapping
 *   compression, CSA's form ([report] §2.3.1: the hidden states give two KV
 *   sets C_a, C_b with weights Z_a, Z_b; §2.3.2: HCA compresses without
 *   overlap).  Entry j pools the a stream (k, g, bias) over its own block j
 *   and the b stream (k_b, g_b, bias_b) over the previous block j - 1, one
 *   softmax per channel over the 2 m logits:
 *     c_j[d] = sum_{i in block j} w_i k_i[d] + sum_{i in block j-1} w'_i kb_i[d]
 *   with (w, w') = softmax over {g_i[d] + bias[i - j m][d]} and
 *   {gb_i[d] + bias_b[i - (j - 1) m][d]}; entry 0 pools the a stream alone.
 *   The entry still ends at token (j + 1) m - 1.  DENSE_AB takes k_b, g_b in
 *   the dtypes of k, g.  APPEND_AB does what APPEND does and, per step, also
 *   writes k_new_b[b] / g_new_b[b] to slot L % (2 m) of tail_b /
 *   tail_gate_b, which hold the b stream of the current and the previous
 *   block; m <= 16 (CSA_ERR_UNSUPPORTED beyond).
 * No mode needs scratch memory: csa_compress_workspace_size() returns 0; a
 * workspace, when given, only carries the run-time status word.
 */
enum csa_compress_mode {
  CSA_COMPRESS_DENSE = 0,
  CSA_COMPRESS_APPEND = 1,
  CSA_COMPRESS_WINDOW = 2,
  CSA_COMPRESS_DENSE_AB = 3,
  CSA_COMPRESS_APPEND_AB = 4
};

typedef struct csa_compress_params {
  uint32_t struct_size;
  int32_t mode;
  int32_t batch, m, dim;
  const float* bias;          /* f32 [m][dim] learnable position bias */
  /* DENSE */
  int32_t n_tokens;
  const void* k; int32_t k_dtype;   /* [B][n_tokens][dim] */
  const void* g; int32_t g_dtype;   /* [B][n_tokens][dim] */
  /* APPEND */
  const int32_t* seq_len;     /* [B] device */
  const uint16_t* k_new;      /* bf16 [B][dim] */
  const float* g_new;         /* f32 [B][dim] */
  uint16_t* ring; int32_t ring_size;  /* bf16 [B][ring_size][dim] */
  float* tail_gate;           /* f32 [B][m][dim] */
  /* output */
  csa_store dst;
  /* optional: no mode needs scratch, but when a workspace of at least 4
   * bytes is given, its status word records run-time faults (a page id
   * outside the pool), read by csa_workspace_status() */
  void* workspace;
  size_t workspace_bytes;
  /* optional ([report] §2.3.3; a struct that ends before these fields means
   * none of them): every pooled entry is RMS-normalized before it is stored,
   * x / sqrt(mean(x^2) + norm_eps) * norm[d] (norm: f32 [dim], or NULL for no
   * norm), then, when rope_base > 0, its last 64 dims are turned by RoPE at
   * the raw position of its block's first token, j * m: pairs (2i, 2i + 1)
   * of those dims by the angle j m base^(-2i / 64).  Both run in float32
   * before the quantize-on-write.  RoPE needs an even dim >= 64. */
  const float* norm;
  float norm_eps;
  float rope_base;
  /* CSA_FLAG_OVERLAP_PREVIOUS or 0 (a struct that ends before this field
   * counts as 0).  With the flag an append may run alongside the kernel
   * launched just before it on the stream, which must neither read nor write
   * this call's ring, tail gates and destination entries nor write its inputs
   * (seq_len, k_new, g_new, bias, norm): for example the other stream's append
   * of the same decode step. */
  int32_t flags;
  /* the b stream of modes CSA_COMPRESS_DENSE_AB and CSA_COMPRESS_APPEND_AB
   * (a struct that ends before these fields cannot use those modes) */
  const float* bias_b;        /* f32 [m][dim] */
  const void* k_b;            /* DENSE_AB: [B][n_tokens][dim], dtype k_dtype */
  const void* g_b;            /* DENSE_AB: [B][n_tokens][dim], dtype g_dtype */
  const uint16_t* k_new_b;    /* APPEND_AB: bf16 [B][dim] */
  const float* g_new_b;       /* APPEND_AB: f32 [B][dim] */
  uint16_t* tail_b;           /* APPEND_AB: bf16 [B][2 m][dim], slot p % (2 m) */
  float* tail_gate_b;         /* APPEND_AB: f32 [B][2 m][dim], slot p % (2 m) */
} csa_compress_params;
/* Workspace bytes of a call: always 0 (no mode needs scratch). */
CSA_API size_t csa_compress_workspace_size(const csa_compress_params* p);
CSA_API int csa_compress(const csa_compress_params* p, csa_stream_t stream);

/* ==========================================================================
 * Steps 2 + 3: lightning indexer and top-k selector
 * ([report] §2.3.1 "lightning indexer", §5.2.1 BF16 index scores / FP4 QK;
 *  [hf] "Hybrid attention": FP4, ReLU-scored multi-head dot product)
 * ==========================================================================
 * For query row r (position t = pos[r], sequence b = seq[r] or r if seq is
 * NULL), over blocks j < n = N_c(t):
 *     s_j = sum_h w[r][h] * ReLU(q[r][h] . kI_b[j])
 * then keeps min(top_k, n) blocks: score descending, ties to the lower block
 * index, -0 == +0.  idx[r] holds the kept block indices ascending, padded
 * with -1 to top_k; cnt[r] = min(top_k, n).
 *
 * Key formats / arithmetic:
 *   CSA_FMT_DENSE_F32 with q F32: canonical float32 order, bit-reproducible:
 *       acc_h = fma chain over d in order; r_h = acc_h > 0 ? acc_h : 0;
 *       s = fma chain over h in order of w_h * r_h.
 *   CSA_FMT_INDEX_POOL_BF16 with q BF16: tensor-core products, float32
 *       accumulation (order unspecified).
 *   CSA_FMT_INDEX_POOL_E2M1 with q F32: q is quantized to the FP4 format of
 *       the pool (per-16 e4m3 scales) first; products of decoded values,
 *       float32 accumulation.
 * score_dtype CSA_F32 keeps float32 scores; CSA_BF16 rounds each score to
 * bf16 (RNE) before selection ([report] §5.2.1).
 * w: [T][H_I] floats, or one [H_I] vector for all rows when w_shared != 0.
 * scores_out (optional, f32 [T][score_capacity]): the score of every visible
 * block (after the bf16 rounding when score_dtype is BF16); NaN scores set
 * CSA_ERR_INVALID_ARG in the workspace status.
 */
typedef struct csa_index_params {
  uint32_t struct_size;
  int32_t num_queries;        /* T */
  int32_t batch;              /* B, sequences in the store */
  int32_t heads, dim;         /* H_I, d_I */
  int32_t m;
  int32_t max_pos;            /* host-side upper bound of pos[] (sizes the launch) */
  const void* q; int32_t q_dtype;   /* [T][H_I][d_I] */
  const float* w; int32_t w_shared;
  const int32_t* pos;         /* [T] device */
  const int32_t* seq;         /* [T] device, or NULL for seq[r] = r */
  csa_store keys;             /* compressed indexer keys */
  int32_t top_k;
  int32_t score_dtype;        /* CSA_F32 or CSA_BF16 */
  int32_t* idx;               /* [T][top_k] */
  int32_t* cnt;               /* [T] */
  float* scores_out;          /* optional [T][score_capacity] */
  int32_t score_capacity;
  int32_t flags;              /* CSA_FLAG_OVERLAP_PREVIOUS or 0 (a struct that
                                 ends before this field counts as 0) */
} csa_index_params;
CSA_API size_t csa_index_topk_workspace_size(const csa_index_params* p);
/* The two steps separately, with the same params and workspace:
 * csa_index_score writes the score of every visible block of every query row
 * into the workspace (step 2); csa_index_select selects from those scores and
 * writes idx / cnt / scores_out (step 3).  csa_index_topk does both. */
CSA_API int csa_index_score(const csa_index_params* p, void* workspace, size_t workspace_bytes,
                            csa_stream_t stream);
CSA_API int csa_index_select(const csa_index_params* p, void* workspace, size_t workspace_bytes,
                             csa_stream_t stream);
CSA_API int csa_index_topk(const csa_index_params* p, void* workspace, size_t workspace_bytes,
                   csa_stream_t stream);

/* csa_index_topk without a workspace argument.  The pages have no
 * counterpart: this is a convenience of the library.  It is meant for callers
 * that are handed their input and output buffers by a host framework that owns
 * every device allocation and exposes no allocator to them, so they cannot set
 * up a workspace of their own.
 *   - Scratch: a fixed array of 8 MiB inside the library's device memory.
 *     Every GPU that loads libcsa holds it until the process exits.  The
 *     function allocates nothing and frees nothing.
 *   - Limit: csa_index_topk_workspace_size(p) must be at most 8 MiB;
 *     otherwise CSA_ERR_WORKSPACE and nothing is launched.
 *   - Limit, exactly: 1024 + num_queries * ceil(n_max / 128) * 128 * b <= 8 MiB,
 *     n_max = (max_pos + 1) / m, b = 4 for float32 scores, 2 for BF16: up to
 *     127 queries x 16384 visible blocks of float32 scores, or 255 of BF16.
 *   - Device address: looked up with the device current, on every call made
 *     outside a stream capture (so it follows a module reload after a device
 *     reset); a call made while its stream is being captured uses the address
 *     of the device's last uncaptured call.  Make one call on a device before
 *     capturing any.
 *   - Sharing: every call, on every stream, uses the same array, and the
 *     array keeps the last call's scores.  Each call resets the status word.
 *     Calls that overlap on the GPU race on the array and give undefined
 *     results: order them on one stream.
 *   - Run-time faults (a NaN score, a page id outside the pool, a bounded
 *     wait that ran out) are recorded in the array's status word, which
 *     csa_index_topk_noalloc_status() reads.  When it is CSA_OK the results
 *     equal csa_index_topk's. */
CSA_API int csa_index_topk_noalloc(const csa_index_params* p, csa_stream_t stream);
/* Copies the status word of the last csa_index_topk_noalloc call on the
 * current device to *out (host memory) after the work queued on `stream`;
 * synchronizes the stream.  No allocation. */
CSA_API int csa_index_topk_noalloc_status(int32_t* out, csa_stream_t stream);

/* ==========================================================================
 * Steps 4 + 5: core attention
 * ([report] §2.3.1 shared-KV MQA, §2.3.2 HCA, §2.3.3 sliding window and sink;
 *  [hf] Fig. 3 / Fig. 4)
 * ==========================================================================
 * For query row r (position t, sequence b) and head h, one softmax over
 *   S = selected compressed entries (csa_attend: idx[r][0 .. cnt[r]);
 *       hca_attend: every j < N_c(t))
 *   plus the window: raw tokens at positions max(0, t - W + 1) .. t.
 * logit = scale * (q[r][h] . x); o[r][h] = sum p * x (key = value = the full
 * D-dim entry); with sink != NULL, exp(sink[h]) joins the denominator only.
 * A window token inside a selected block still counts once raw and once
 * inside the pooled entry.  lse (optional) = natural log of the denominator.
 * An empty set gives o = 0 and lse = -inf.
 *
 * Formats: kv CSA_FMT_DENSE_F32 with q F32, window F32, out F32: all-float32
 * path.  kv CSA_FMT_KV_POOL_FP8 (D = 576) with q BF16, window BF16, out BF16
 * or F32: tensor-core path, float32 accumulation.  Its MMA operands are FP16:
 * the e4m3 content codes exactly, q, the RoPE dims and window rows converted
 * from BF16 (exact within FP16's range), and the softmax weights rounded to
 * FP16; the entry scale multiplies the content part of the logit and the
 * weights of the content dims (in float32, before that rounding).
 * window: [B][win_ring][D]; position p at slot p % win_ring (a dense raw
 * sequence is a ring with win_ring >= every position).
 */
typedef struct csa_attend_params {
  uint32_t struct_size;
  int32_t num_queries;        /* T */
  int32_t batch;              /* B */
  int32_t heads, dim;         /* H, D */
  int32_t m;
  int32_t max_pos;            /* host-side upper bound of pos[] */
  const void* q; int32_t q_dtype;   /* [T][H][D] */
  const int32_t* pos;         /* [T] */
  const int32_t* seq;         /* [T] or NULL (seq[r] = r) */
  const int32_t* idx;         /* csa_attend: [T][top_k]; ignored by hca_attend */
  const int32_t* cnt;         /* csa_attend: [T] */
  int32_t top_k;
  csa_store kv;               /* compressed entries */
  int32_t window;             /* W */
  const void* win; int32_t win_dtype; int32_t win_ring;
  float scale;
  const float* sink;          /* [H] or NULL */
  void* out; int32_t out_dtype;     /* [T][H][D] */
  float* lse;                 /* [T][H] or NULL */
  int32_t flags;              /* enum csa_attend_flags | CSA_FLAG_OVERLAP_PREVIOUS
                                 (a struct that ends before this field counts
                                 as flags = 0) */
  /* query / window normalization and partial RoPE ([report] §2.3.3), on the
   * tensor-core path (a struct that ends before these fields means none):
   *   q_norm   f32 [D] or NULL: every query head is RMS-normalized,
   *            q / sqrt(mean(q^2) + norm_eps) * q_norm[d];
   *   win_norm f32 [D] or NULL: every window row likewise, as it is read
   *            (the ring keeps raw tokens: they also feed the compressor);
   *   rope_base > 0: RoPE on the last 64 dims (pairs (2i, 2i + 1), angle
   *            pos base^(-2i / 64)): the query at its position t, window rows
   *            at their positions; the compressed entries are read as stored
   *            (csa_compress rotates them at j m with the same base); and the
   *            output's last 64 dims are turned back by t, so they carry
   *            positions relative to the query.
   * Normalization and rotation run in float32 before the FP16 rounding of
   * the MMA operands. */
  const float* q_norm;
  const float* win_norm;
  float norm_eps;
  float rope_base;
} csa_attend_params;
/* CSA_ATTEND_BATCH_INVARIANT ([report] §3.3, batch invariance): a query's
 * item list is cut into splits whose number and boundaries depend only on
 * its own item count (about 160 items per split, at most 8 splits), and the
 * splits are merged in a fixed order, so a query's output and lse are
 * bitwise the same in any batch and any launch.  Without the flag the split
 * count also depends on the batch and the SM count (more parallelism for
 * small batches); results are then reproducible for a fixed launch shape. */
/* CSA_ATTEND_WINDOW_ONLY: a layer without a compressed branch (pure
 * sliding-window attention, [report] §4.2.1: the first layers of the Flash
 * model; [hf] "Hybrid attention": the MTP block): the softmax runs over the
 * window alone; kv, idx, cnt and m are not read (the path follows q_dtype:
 * BF16 the tensor-core path, F32 the float32 path). */
enum csa_attend_flags { CSA_ATTEND_BATCH_INVARIANT = 1, CSA_ATTEND_WINDOW_ONLY = 2 };
CSA_API size_t csa_attend_workspace_size(const csa_attend_params* p);
CSA_API size_t hca_attend_workspace_size(const csa_attend_params* p);
/* How a call (csa_attend when sparse != 0, else hca_attend) splits each
 * query's item list: *splits CTAs per query, merged by *merge = 0 (one split:
 * no merge), 1 (the splits of a query form a thread-block cluster and merge
 * inside the kernel, one launch) or 2 (a second kernel merges the partials,
 * two launches).  Used when a split count has to be reported or the
 * kernels of a step counted. */
CSA_API int csa_attend_plan(const csa_attend_params* p, int32_t sparse, int32_t* splits, int32_t* merge);
CSA_API int csa_attend(const csa_attend_params* p, void* workspace, size_t workspace_bytes,
               csa_stream_t stream);
CSA_API int hca_attend(const csa_attend_params* p, void* workspace, size_t workspace_bytes,
               csa_stream_t stream);

/* ==========================================================================
 * Device status
 * ========================================================================== */
/* Copies the status word of a workspace to *out (synchronizes the stream). */
CSA_API int csa_workspace_status(const void* workspace, int32_t* out, csa_stream_t stream);
/* Resets the status word to CSA_OK (asynchronous). */
CSA_API int csa_workspace_clear_status(void* workspace, csa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H_ */
