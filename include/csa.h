/*
 * csa.h — C ABI of the B300 (sm_103a) kernels for the DeepSeek-V4 Compressed
 * Sparse Attention (CSA) and Heavily Compressed Attention (HCA) forward path.
 *
 * The operator is defined only mathematically by the pages this library
 * follows: the DeepSeek-V4 technical report in Chinese translation
 * (blog.uika.cn) §2.3.1 "Compressed Sparse Attention", §2.3.2 "Heavily
 * Compressed Attention", §2.3.3 (RMS-normalised q / entries, partial RoPE with
 * the output rotated back, sliding window, attention sink) and §2.3.4 (FP8 /
 * BF16 KV storage, FP4 indexer QK), and the paper notes at
 * awesome.papernotes.org ("关键设计 1" / "关键设计 2" equations).
 *
 * Conventions shared by every call:
 *   - Every pointer is caller-owned DEVICE memory of the current CUDA device,
 *     except where a comment says otherwise.  The library never allocates,
 *     frees or synchronises in these calls; work is enqueued on `stream`
 *     (a cudaStream_t passed as void*, NULL = the legacy default stream).
 *   - Stream order holds for every call.  The attention kernel of a short
 *     csa_attend / hca_attend launch (at most 4 work items per CTA: decode)
 *     is enqueued with programmatic stream serialisation: its CTAs may set
 *     up barriers and tensor memory while the previous kernel on the stream
 *     still runs, but they read and write no global memory before that
 *     kernel has completed.
 *   - Tensors are dense and row-major in the shapes given (last dim fastest).
 *   - Argument, shape and alignment errors are returned before any launch.
 *     CSA_ERR_CUDA means a launch or runtime call failed (cudaGetLastError
 *     text via csa_last_cuda_error()).  Faults found on the device (a bounded
 *     wait that gave up, an out-of-range index, a negative position, a window
 *     token outside its buffer, a block-table entry outside its pool, a
 *     histogram that disagrees with its scores) set a sticky device error
 *     word that csa_device_error() reads; the offending rows are left out.
 *   - Query positions: q_pos is a DEVICE array int32 [B, Tq]; q_pos[b,i] is
 *     the absolute token position t of query row i of batch row b, so every
 *     sequence of a batch may sit at its own context length (§2.3.1: the
 *     visibility rule is per query t).  q_pos = NULL means t = i for every
 *     batch row (causal prefill from token 0).  Compressed entry s is visible
 *     to the query at t iff (s+1)*m <= t+1, and its RoPE position is
 *     m*(s+1)-1; entries at s >= N are never read, whatever t.  T mod m tail
 *     tokens are not compressed (§3.6.1: they wait in a buffer).  The host
 *     cannot see device arrays: a position below 0 sets the device error
 *     word's bad-index bit, and that row is treated as seeing nothing
 *     (scores -inf, no index, output 0).
 *   - Window rows: win_base is a DEVICE array int32 [B]; row j of batch row
 *     b's window buffer holds raw token win_base[b] + j (NULL = 0 for every
 *     batch row).  A window token outside a batch row's buffer sets the
 *     bad-index bit and is left out of that query's row set.
 */
#ifndef CSA_B300_H
#define CSA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,  /* null pointer, bad size or misaligned pointer */
  CSA_ERR_UNSUPPORTED = 2,  /* valid arguments for which the library has no kernel */
  CSA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  CSA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  CSA_ERR_TIMEOUT = 5,      /* device error word: a bounded wait gave up */
  CSA_ERR_DEVICE = 6        /* device error word: other device-side fault */
} csa_status_t;

/* Element formats. */
typedef enum {
  CSA_DT_F32 = 0,            /* float32 */
  CSA_DT_BF16 = 1,           /* bfloat16 */
  CSA_DT_E4M3_BF16ROPE = 2,  /* KV rows: first d-r dims e4m3fn bytes times one float32
                                scale per row, last r (RoPE) dims bfloat16 (§2.3.4) */
  CSA_DT_E2M1_BLOCK16 = 3    /* indexer q/K: e2m1 codes two per byte (element 2j in the
                                low nibble of byte j) times one e4m3fn scale byte per
                                16 consecutive elements (§3.4 FP4 indexer QK path) */
} csa_dtype_t;

/* ---------------------------------------------------------------------------
 * Paged rows — the heterogeneous KV-cache layout of §3.6.1 (inference
 * framework): the cache is cut into blocks of lcm(m, m') raw tokens, so one
 * block holds lcm/m CSA entries (and as many indexer keys) and lcm/m' HCA
 * entries, and one block table per sequence addresses every pool; the sliding
 * window and the not-yet-compressed tail live in a fixed-size state cache.
 * A csa_pages_t maps the logical rows j of sequence b (entry index s, or the
 * window row of a token) to rows of a pool shared by all sequences:
 *   block_table == NULL: flat layout, row b * rows + j (rows = N or T_win);
 *   otherwise pool row block_table[b * max_blocks + j / block_rows] * block_rows
 *            + j % block_rows (block_table: DEVICE int32 [B, max_blocks]).
 *   ring (window rows only): token p sits at logical row p mod T_win, so a
 *            fixed buffer of T_win rows per sequence takes one new token per
 *            decode step in place; the tokens present are still
 *            win_base[b] .. win_base[b] + T_win - 1.
 * A block-table entry outside [0, num_blocks) read on the device sets the
 * bad-index bit of the device error word, and its rows are left out (index:
 * left unread, their scores undefined).  Only the table entries of logical
 * blocks the call reads are read (entries: blocks < ceil(N / block_rows)).
 * A zero-filled csa_pages_t is the flat layout. */
typedef struct {
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t block_rows;
  int32_t num_blocks;
  int32_t ring;
} csa_pages_t;

/* A set of key=value rows (compressed entries or raw window tokens).
 *   dtype F32 / BF16 : data = [B, rows, d]; scale, rope unused.
 *   dtype E4M3_BF16ROPE : data = e4m3 [B, rows, d-r], scale = float32 [B, rows],
 *                         rope = bf16 [B, rows, r].
 *   With pages.block_table set, data / scale / rope are pools of
 *   num_blocks * block_rows rows in the same per-row formats.
 *   flags: 0, or CSA_KV_ROTATED for compressed entries whose last r dims are
 *          already rotated at their own position m*(s+1)-1 (csa_compress_ex
 *          with rope_dims = r writes them so); the attention then does not
 *          rotate them again.  Window rows are always stored unrotated. */
#define CSA_KV_ROTATED 1
typedef struct {
  int32_t dtype;
  int32_t flags;
  const void* data;
  const float* scale;
  const void* rope;
  csa_pages_t pages;
} csa_kv_t;

/* ---------------------------------------------------------------------------
 * Block pool — host-side allocator of the physical blocks behind a paged
 * cache (§3.6.1).  Blocks are ids 0 .. num_blocks-1; the pool hands out free
 * ids and takes them back, and refuses to take back an id that is not
 * allocated.  Host memory only: these calls touch no GPU.  A pool is not
 * thread-safe; guard it if several host threads share it.
 * ------------------------------------------------------------------------- */
typedef struct csa_block_pool csa_block_pool_t;
/* NULL when num_blocks is not in [1, 2^30] or memory runs out. */
csa_block_pool_t* csa_block_pool_create(int32_t num_blocks);
void csa_block_pool_destroy(csa_block_pool_t* pool);
int32_t csa_block_pool_free_count(const csa_block_pool_t* pool);
/* n ids into ids[0..n) (HOST array), lowest free ids first after creation;
 * CSA_ERR_WORKSPACE (nothing taken) when fewer than n are free. */
csa_status_t csa_block_pool_alloc(csa_block_pool_t* pool, int32_t n, int32_t* ids);
/* Returns n ids; CSA_ERR_INVALID_ARG (nothing returned) if any id is out of
 * range, not allocated, or repeated. */
csa_status_t csa_block_pool_release(csa_block_pool_t* pool, int32_t n, const int32_t* ids);

/* ---------------------------------------------------------------------------
 * csa_compress — softmax-weighted block compression of per-token entries.
 * CSA (§2.3.1 compression equations): entry i, channel c = sum over the a-rows
 * of block i and the b-rows of block i-1 of softmax_rows(Z + B)[j,c] * C[j,c];
 * entry 0 has no previous block (its softmax runs over the m a-rows alone).
 * HCA (§2.3.2): pass Cb = Zb = NULL; entry i uses the m rows of block i only.
 *   Ca, Za (and Cb, Zb): [B, T, d] in `dtype` (F32 or BF16).
 *   Ba, Bb: optional learnable position biases [m, d] float32 (NULL = zero).
 *   out: [B, floor(T/m), d] in `dtype`.
 *   Requires d % 8 == 0 (BF16) or d % 4 == 0 (F32), d <= 2048, 1 <= m <= 4096,
 *   16-byte aligned tensors.
 * ------------------------------------------------------------------------- */
csa_status_t csa_compress(const void* Ca, const void* Cb, const void* Za, const void* Zb,
                          const float* Ba, const float* Bb, void* out, int B, int T, int d,
                          int m, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * csa_compress_ex — csa_compress with an optional epilogue on every
 * compressed entry, applied in this order (the producer side of the path):
 *   1. rms_norm: entry / sqrt(mean_c(entry^2) + norm_eps), times norm_weight
 *      ([d] float32 device, NULL = 1) — §2.3.3: the compressed KV entries are
 *      RMS-normalised before core attention;
 *   2. rope_dims = r > 0: the last r dims rotated by RoPE (interleaved pairs,
 *      theta_j = rope_base^(-2j/r)) at the entry's position m*(i+1)-1, so the
 *      attention can take the entries pre-rotated (CSA_KV_ROTATED).
 * opts is a HOST pointer (NULL = no epilogue, the same as csa_compress).
 * The same call with d = c_I compresses the indexer keys (K^IComp of §2.3.1).
 * rope_dims must be even, <= min(d, 128), and a multiple of 8 (BF16) or 4
 * (F32).
 *
 * out_pages: where the entries go (zero-filled: out is [B, floor(T/m), d]).
 * With out_pages.block_table set, out is a pool of num_blocks * block_rows
 * rows, and compressed entry i >= out_first of sequence b is written to
 * logical row e = out_entry0[b] + i - out_first (out_entry0: DEVICE int32 [B],
 * NULL = 0) and rotated (rope_dims > 0) at position m*(e+1)-1.  A prefill
 * writes its entries straight into the paged cache (out_first = 0,
 * out_entry0 = NULL).  A decode step passes each sequence's last 2m raw rows
 * (T = 2m) with out_first = 1, so the entry of the block that just closed
 * (local entry 1: its a-rows and the previous block's b-rows) lands at its
 * logical row; a negative out_entry0[b] writes nothing for sequence b (its
 * block did not close).  For a sequence's first block the previous block's
 * b-row logits are -inf, which gives the entry-0 rule.  out_entry0 and
 * out_first are ignored for the flat layout; the ring flag must be 0.
 * ------------------------------------------------------------------------- */
typedef struct {
  int32_t rms_norm;
  float norm_eps;
  const float* norm_weight;
  int32_t rope_dims;
  float rope_base;
  csa_pages_t out_pages;
  const int32_t* out_entry0;
  int32_t out_first;
} csa_compress_opts_t;

csa_status_t csa_compress_ex(const void* Ca, const void* Cb, const void* Za, const void* Zb,
                             const float* Ba, const float* Bb, void* out, int B, int T, int d,
                             int m, int dtype, const csa_compress_opts_t* opts, void* stream);

/* ---------------------------------------------------------------------------
 * csa_index — lightning-indexer scores (§2.3.1 "Lightning Indexer"):
 *   scores[b,i,s] = sum_h w[b,i,h] * ReLU(qI[b,i,h,:] . K[b,s,:])  if visible,
 *                   -inf                                           otherwise.
 *   dtype F32 / BF16: qI [B, Tq, H, c], K [B, N, c]; qI_sf, K_sf unused (NULL).
 *   dtype E2M1_BLOCK16: qI [B, Tq, H, c/2] bytes, qI_sf [B, Tq, H, c/16] bytes,
 *                       K [B, N, c/2] bytes, K_sf [B, N, c/16] bytes.
 *   w: [B, Tq, H] float32.  scores: [B, Tq, N] (every element written), in
 *   score_dtype F32, or BF16: each score rounded to bf16 (§3.4: index scores
 *   quantised from FP32 to BF16 for a faster top-k selector; the selection
 *   then ranks the rounded scores, ties toward the lower index).
 *   BF16 needs (H, c) in {(64,128), (64,64), (32,128), (128,128)}; E2M1 needs
 *   H in {32,64,128}, c == 128; F32 any H, c <= 256.
 * ------------------------------------------------------------------------- */
csa_status_t csa_index(const void* qI, const void* qI_sf, const float* w, const void* K,
                       const void* K_sf, const int32_t* q_pos, void* scores, int score_dtype,
                       int B, int Tq, int N, int H, int c, int m, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * csa_topk — per query row, the k visible entries with the largest scores
 * (§2.3.1 "top-k selector"; C_t = TopK_k(I_t,:)).  Ties are broken toward the
 * lower entry index.  idx[b,i,:] holds the min(k, vis) selected entry indices
 * in ascending order, then -1 up to k.
 *   scores: [B, Tq, N] in score_dtype F32 or BF16 (only s < vis(t) is read;
 *   BF16 needs N <= 16 * 32768); q_pos: [B, Tq] as above; idx: [B, Tq, k]
 *   int32.  Requires 1 <= k <= 4096.
 * ------------------------------------------------------------------------- */
csa_status_t csa_topk(const void* scores, int score_dtype, const int32_t* q_pos, int32_t* idx,
                      int B, int Tq, int N, int k, int m, void* stream);

/* ---------------------------------------------------------------------------
 * csa_index_topk — csa_index followed by csa_topk in one call, with the same
 * results (scores and index sets identical to the two separate calls).  For
 * one query row per batch row (decode) in BF16 or E2M1_BLOCK16, the index
 * kernel also counts each visible score's top 11 order-preserving key bits
 * into a per-row histogram, so the selector starts from the threshold bin
 * instead of building that histogram itself (§2.3.1 "Lightning Indexer" and
 * "top-k selector").  Other shapes run the two stages unchanged.  With
 * score_dtype BF16 the keys have 16 bits, so the selector needs one radix
 * pass below that histogram's digit instead of three.
 *   ws / ws_bytes: scratch of csa_index_topk_workspace_size(B, Tq, N, dtype)
 *   bytes (16-byte aligned; may be NULL when that size is 0).  It holds the
 *   per-row histograms and must be ZERO-FILLED before its first use; every call
 *   that returns CSA_OK and leaves the device error word clear leaves it zero
 *   again (the selector clears each histogram after reading it), so a decode
 *   loop zero-fills it once.  After a failed call, zero-fill it again.
 * ------------------------------------------------------------------------- */
csa_status_t csa_index_topk(const void* qI, const void* qI_sf, const float* w, const void* K,
                            const void* K_sf, const int32_t* q_pos, void* scores, int score_dtype,
                            int32_t* idx, int B, int Tq, int N, int H, int c, int m, int k,
                            int dtype, void* ws, size_t ws_bytes, void* stream);
size_t csa_index_topk_workspace_size(int B, int Tq, int N, int dtype);

/* ---------------------------------------------------------------------------
 * csa_index_paged / csa_index_topk_paged — csa_index / csa_index_topk with
 * the keys K (and their scales K_sf) read through K_pages (a HOST pointer;
 * NULL, or a NULL block_table, is the flat layout): K is then a pool of
 * num_blocks * block_rows key rows (K_sf the matching scale rows), addressed
 * by the same block table as the compressed entries of §3.6.1.  BF16 and
 * E2M1_BLOCK16 keys need block_rows a power of two >= 8; F32 any
 * block_rows >= 1; ring must be 0.  Results are identical to the flat calls
 * on the same logical keys.
 * ------------------------------------------------------------------------- */
csa_status_t csa_index_paged(const void* qI, const void* qI_sf, const float* w, const void* K,
                             const void* K_sf, const csa_pages_t* K_pages, const int32_t* q_pos,
                             void* scores, int score_dtype, int B, int Tq, int N, int H, int c,
                             int m, int dtype, void* stream);
csa_status_t csa_index_topk_paged(const void* qI, const void* qI_sf, const float* w,
                                  const void* K, const void* K_sf, const csa_pages_t* K_pages,
                                  const int32_t* q_pos, void* scores, int score_dtype,
                                  int32_t* idx, int B, int Tq, int N, int H, int c, int m, int k,
                                  int dtype, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * csa_attend — shared-KV multi-query core attention (§2.3.1 "Shared KV MQA",
 * §2.3.3).  For query row i at position t and head h:
 *   rows J = {compressed entries idx[b,i,:] >= 0} U {raw tokens max(0,t-n_win+1)..t}
 *   every row is both key and value; the last r dims of q and of each row are
 *   rotated by RoPE (interleaved pairs, theta_j = rope_base^(-2j/r)) at their
 *   positions (t; m*(s+1)-1 for entry s; the token position for window rows);
 *   logits = q.row / sqrt(d); p = exp(logit) / (sum exp(logits) + exp(sink[h]));
 *   o = sum p * rotated row; out = o with its last r dims rotated by -t.
 *   q: [B, Tq, n_h, d] (F32 or BF16); out: same shape and dtype as q.
 *   entries: [B, N, d] rows (F32, BF16 or E4M3_BF16ROPE), or paged through
 *        entries.pages (any block_rows >= 1; ring must be 0).
 *   win: [B, T_win, d] rows; batch row b holds raw tokens win_base[b] ..
 *        win_base[b] + T_win - 1 (win_base: device int32 [B], NULL = 0),
 *        token p at row p - win_base[b], or at row p mod T_win with
 *        win.pages.ring (the state-cache ring of §3.6.1); the rows may be paged
 *        through win.pages as well (one block of T_win rows per sequence is
 *        the usual state slot).
 *   q_pos: device int32 [B, Tq] query positions (NULL: t = i).
 *   idx: [B, Tq, k] int32 from csa_topk (-1 entries are skipped).
 *   sink: [n_h] float32.
 *   ws / ws_bytes: scratch of at least csa_attend_workspace_size(...) bytes,
 *   256-byte aligned (may be NULL when that size is 0).
 *   BF16 / E4M3 need d == 512, r == 64, n_h % 64 == 0; F32 needs d <= 512,
 *   n_h * d <= 16384.
 * ------------------------------------------------------------------------- */
csa_status_t csa_attend(const void* q, csa_kv_t entries, const int32_t* idx, csa_kv_t win,
                        const int32_t* q_pos, const int32_t* win_base, const float* sink,
                        void* out, int B, int Tq, int N, int k, int T_win, int n_h, int d, int r,
                        int m, int n_win, float rope_base, void* ws, size_t ws_bytes,
                        void* stream);

/* hca_attend — csa_attend over every visible compressed entry (block size m = m'),
 * with no index list (§2.3.2: HCA keeps shared-KV MQA but has no top-k). */
csa_status_t hca_attend(const void* q, csa_kv_t entries, csa_kv_t win, const int32_t* q_pos,
                        const int32_t* win_base, const float* sink, void* out, int B, int Tq,
                        int N, int T_win, int n_h, int d, int r, int m, int n_win,
                        float rope_base, void* ws, size_t ws_bytes, void* stream);

/* Scratch bytes csa_attend / hca_attend need for these sizes (k = 0 for HCA).
 * q_dtype / kv_dtype as in the calls.  The work split is planned for the
 * largest row set any query can have (min(k, N) or N entries plus
 * min(n_win, T_win) window rows), so it does not depend on the positions. */
size_t csa_attend_workspace_size(int B, int Tq, int N, int k, int T_win, int n_h, int d, int r,
                                 int m, int n_win, int q_dtype, int kv_dtype, int is_hca);

/* ---------------------------------------------------------------------------
 * csa_decode_step_host — one CSA decode step of one layer from HOST buffers,
 * all on `stream` in this order: the step's new inputs are copied host ->
 * device (one cudaMemcpyAsync each), csa_index_topk_paged and csa_attend run on
 * them against the device-resident cache, and the output is copied device ->
 * host.  The call returns once the work is queued: synchronise the stream
 * before reading `out_h`.  Host buffers should be pinned for the copies to
 * overlap; the pages define no such call (it is the boundary a serving loop
 * with host-side inputs uses).
 *   HOST: q_h [B, 1, n_h, d] bf16; qI_h [B, 1, H, c] bf16 (E2M1_BLOCK16: bytes
 *         [B, 1, H, c/2] with qI_sf_h [B, 1, H, c/16]); w_h [B, 1, H] float32;
 *         q_pos_h [B] int32 (each sequence's new token); win_base_h [B] int32
 *         (NULL = 0); out_h [B, 1, n_h, d] bf16.
 *   DEVICE (caller-owned, persistent): K, K_sf, K_pages (HOST pointer to the
 *         row map, NULL = flat) as in csa_index_topk_paged; entries, win as in
 *         csa_attend; sink [n_h] float32.
 *   ws / ws_bytes: device scratch of csa_decode_step_workspace_size(...)
 *         bytes, 256-byte aligned, ZERO-FILLED before its first use (it holds
 *         csa_index_topk's histograms, which every successful call leaves
 *         zero); the staged inputs, scores (float32), indices and the device
 *         output live there too.
 *   dtype: indexer dtype (BF16 or E2M1_BLOCK16); entries / win dtype as in
 *   csa_attend (BF16 or E4M3_BF16ROPE).
 * ------------------------------------------------------------------------- */
csa_status_t csa_decode_step_host(const void* q_h, const void* qI_h, const void* qI_sf_h,
                                  const float* w_h, const int32_t* q_pos_h,
                                  const int32_t* win_base_h, const void* K, const void* K_sf,
                                  const csa_pages_t* K_pages, csa_kv_t entries, csa_kv_t win,
                                  const float* sink, void* out_h, int B, int N, int H, int c, int k,
                                  int T_win, int n_h, int d, int r, int m, int n_win, int dtype,
                                  float rope_base, void* ws, size_t ws_bytes, void* stream);
size_t csa_decode_step_workspace_size(int B, int N, int H, int c, int k, int T_win, int n_h,
                                      int d, int r, int m, int n_win, int dtype, int kv_dtype);

/* ---------------------------------------------------------------------------
 * csa_attend_noalloc — csa_attend without a caller-supplied workspace.  The
 * pages define no such call; it exists for callers that cannot allocate
 * device memory: code embedded in a host application or serving engine that
 * owns every device allocation and hands this layer only its input and output
 * buffers, and latency-critical callers that cannot take the implicit
 * device-wide synchronisation of cudaMalloc / cudaFree.
 *
 * Arguments, layouts and results are those of csa_attend minus ws / ws_bytes.
 * The scratch lives in one fixed array of CSA_NOALLOC_SCRATCH_BYTES in this
 * library's device image: every GPU that loads the library holds it until
 * the process exits.  This call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   - Sizes whose scratch need (csa_attend_workspace_size) exceeds
 *     CSA_NOALLOC_SCRATCH_BYTES return CSA_ERR_WORKSPACE before any launch
 *     (csa_last_cuda_error() then gives both byte counts).  For scale: a
 *     decode row set whose chunks (at most 16) merge inside a thread-block
 *     cluster needs none (batch 4, k = 1024, V4-Pro shape); chunks that
 *     merge in smaller clusters keep 128 KB of fp32 partials per cluster;
 *     a split with more work items than SMs keeps 128 KB per item (20 MB for
 *     16 sequences at k = 4096); many query rows over few stored rows keep
 *     one rotated copy of the rows (1 KB per row).
 *   - The first call on a device (with that device current) looks up the
 *     array's device address and caches it; make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Nothing in it must start at zero (every scratch byte a call
 *     reads, that call wrote first), but calls that overlap on the GPU (other
 *     streams, other host threads) race on it: serialise them.
 * ------------------------------------------------------------------------- */
#define CSA_NOALLOC_SCRATCH_BYTES (16u << 20)
csa_status_t csa_attend_noalloc(const void* q, csa_kv_t entries, const int32_t* idx, csa_kv_t win,
                                const int32_t* q_pos, const int32_t* win_base, const float* sink,
                                void* out, int B, int Tq, int N, int k, int T_win, int n_h, int d,
                                int r, int m, int n_win, float rope_base, void* stream);

/* ---------------------------------------------------------------------------
 * csa_grouped_proj — the grouped output projection (§2.3.1 "分组输出投影":
 * the n_h head outputs are split into g groups, each group is projected to a
 * d_g-dimensional intermediate output, and those are projected to the model
 * width d; §4.2.1: V4-Pro g = 16, d_g = 1024, d = 7168).  One call computes,
 * for every group j < G,
 *     C[:, j*N : (j+1)*N] = A[:, j*K : (j+1)*K] * W[j]^T
 * in bf16 with float32 accumulation, rounded once to bf16:
 *   A: [M, lda] bf16 (the attention output [tokens, n_h * d] has lda = n_h*d
 *      and, split into G = g groups, K = (n_h / g) * d);
 *   W: [G, N, K] bf16, each group's weight output-major (row n holds the K
 *      weights of output n);
 *   C: [M, ldc] bf16.
 * The final projection is the same call with G = 1, K = g * d_g, N = d.
 * Requires K, N, lda, ldc multiples of 8, lda >= G*K, ldc >= G*N, 16-byte
 * aligned pointers.  Tensor-core tiles of 128 x 256 outputs; M, N and K need
 * not be multiples of the tile.
 * ------------------------------------------------------------------------- */
csa_status_t csa_grouped_proj(const void* A, int64_t lda, const void* W, void* C, int64_t ldc,
                              int M, int N, int K, int G, void* stream);

/* ---------------------------------------------------------------------------
 * csa_selftest_wait_timeout — a test of the library's failure detection; the
 * pages define no such call.  It runs the BF16 index kernel exactly as
 * csa_index (H = 64, c = 128, same arguments) but with a fault planted by
 * the host: CTA 0's TMA producer leaves out its first K-tile copy, and every
 * wait of the launch gives up after limit_us microseconds (1 .. 2000000; a
 * normal launch waits up to 2 s).  The MMA issuer's wait on the missing tile
 * runs out; it sets the timeout bit of the device error word and raises its
 * CTA's abort flag; the other roles leave their loops, copies already issued
 * are waited for, tensor memory is freed and the kernel returns, leaving the
 * context usable.  The scores are then undefined.  csa_device_error()
 * afterwards returns CSA_ERR_TIMEOUT (and clears the word).  The query rows
 * must see at least one entry, or no copy is issued at all.
 * ------------------------------------------------------------------------- */
csa_status_t csa_selftest_wait_timeout(const void* qI, const float* w, const void* K,
                                       const int32_t* q_pos, float* scores, int B, int Tq, int N,
                                       int m, int limit_us, void* stream);

/* Reads and clears the sticky device error word (synchronises `stream`).
 * Returns CSA_OK, CSA_ERR_TIMEOUT or CSA_ERR_DEVICE. */
csa_status_t csa_device_error(void* stream);

const char* csa_status_string(csa_status_t status);
const char* csa_last_cuda_error(void);  /* text of the last CSA_ERR_CUDA (host memory) */
int csa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_B300_H */
