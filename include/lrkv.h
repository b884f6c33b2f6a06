/*
 * lrkv.h -- C ABI of liblrkv: attention for many LoRA agents over one paged KV
 * cache kept as a shared base part plus a shared-A low-rank part.
 *
 * The method (LRAgent: Efficient KV Cache Sharing for Multi-LoRA LLM Agents,
 * arXiv 2602.01053, Abstract; and PReCache, thelatestinai.com/papers/2609.34054,
 * Abstract and Table 1): each agent i's keys and values are
 *     K_i = RoPE(X W_K + (X A_K) B_K,i),   V_i = X W_V + (X A_V) B_V,i
 * with A_K, A_V shared by all agents. The cache stores, once per token,
 *     K_base = RoPE(X W_K), V_base = X W_V        (the "base" part)
 *     L_K = X A_K, L_V = X A_V                     (the low-rank part, r columns)
 * and each agent's contribution is rebuilt inside the attention kernels:
 * the K term L_K B_K,i is rebuilt per tile on chip, rotated and added to
 * K_base; the V term is reordered as (P L_V) B_V,i ("Flash-LoRA-Attention":
 * the low-rank cache is never expanded to full width in memory).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer unless stated otherwise. Data
 *   tensors (X, W_cat, q, out, pools, B_K, B_V, workspace) must be 16-byte
 *   aligned; int32 arrays and dev_status 4-byte aligned. The caller owns all
 *   memory; the library allocates nothing and keeps no state between calls.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream). They read their inputs and write only their outputs.
 * - Sizes: hidden h, Hq query heads, Hkv kv heads (Hkv divides Hq; query head
 *   m reads kv head m / (Hq/Hkv)), head_dim d in {64, 128}, rank r in
 *   {8, 16, 32, 64}, block_size 16.
 * - dtype: LRKV_BF16 (every tensor bf16; fp32 accumulation) or LRKV_FP32
 *   (every tensor fp32; plain fp32 FMA arithmetic, no tensor cores).
 * - Paged pools (PagedAttention-style blocks of 16 tokens):
 *     base_pool [num_blocks][2][Hkv][16][d]  plane 0 = K_base (rotated), 1 = V_base
 *     lr_pool   [num_blocks][2][16][G*r]     plane 0 = L_K, 1 = L_V; group g's r
 *                                            columns at [g*r, (g+1)*r)
 * - Low-rank groups (lr_groups = G): G = 1 is the shared-A cache of LRAgent
 *   (arXiv 2602.01053, Abstract): L = X A with one A for every agent. G > 1 is
 *   PReCache's PreLRShared (thelatestinai.com/papers/2609.34054, Abstract and
 *   Figure 1): each agent has its own A; one append computes every agent's
 *   low-rank cache, L = [X A_0 | ... | X A_{G-1}], and agent a reads group a
 *   (adapter ids must then be < G, n_adapters <= G).
 *   Token at position p of a sequence whose block-table row is bt lives in
 *   block bt[p / 16], row p % 16. Each (block, plane, kv head) is one
 *   contiguous 16*d element chunk (4 KB for bf16, d = 128).
 * - Compressed base pool (kv_codec = LRKV_CODEC_POLYKV, bf16 only). This is
 *   the PolyKV codec (the abstract printed at the end of the PReCache page):
 *   keys are int8 in q8_0 blocks, and values are rotated by a Walsh-Hadamard
 *   transform and quantised to 3 bits with Lloyd-Max centroids for N(0,1).
 *   The low-rank pool is unchanged. base_pool is bytes
 *   [num_blocks][Hkv][23*d + 64], and each (block, kv head) chunk holds
 *     Kq int8    [16][d]        q8_0 codes of K_base (rotated keys)
 *     Ks fp16    [16][d/32]     q8_0 scale of each 32-dim block, max|x| / 127
 *     Vq uint8   [16][3][d/8]   value codes as three bit planes: plane b, byte
 *                               j/8, bit j%8 = bit b of dim j's 3-bit code
 *     Vn fp32    [16]           ||V_base row||
 *   A key element decodes to q * s; q = round(x / s), ties away from zero.
 *   A value row v decodes to v^ = (H/sqrt(d)) y^, with y^_j = c[code_j] ||v|| / sqrt(d)
 *   (H the Sylvester-Hadamard matrix, c the 8 Lloyd-Max centroids for N(0,1)
 *   in ascending order); code_j counts the Lloyd-Max thresholds below
 *   u_j = y_j sqrt(d) / ||v||, y = (H/sqrt(d)) v. Decode and prefill read
 *   K_i = K^_base + RoPE(L_K B_K,i), V_i = V^_base + L_V B_V,i.
 * - Block tables: int32 [rows][max_blocks] row-major.
 * - RoPE: rotate-half pairing (j, j + d/2), angle p * theta_j with
 *   theta_j = rope_base^(-2j/d), no frequency scaling. Queries arrive already
 *   rotated; the library rotates keys only.
 * - Causality: a row of q_len queries over L keys puts query k at position
 *   L - q_len + k; it sees keys at positions <= its own.
 * - Adapter id -1 = base model only (B = 0). B_K or B_V may be NULL: that
 *   factor is zero for every agent and its work is skipped.
 * - Precision (bf16): fp32 accumulation everywhere; the score product
 *   q . K_a uses fp16 operands (q converted exactly, K_a rounded once), so q
 *   and K_a elements must stay below 65504 in magnitude; P is rounded to bf16
 *   for the P V_base and P L_V products.
 * - Errors: argument problems detected on the host return before any launch
 *   (LRKV_ERR_INVALID_ARG / LRKV_ERR_UNSUPPORTED / LRKV_ERR_WORKSPACE). A failed
 *   launch returns LRKV_ERR_CUDA. Problems only visible on the device (a block
 *   id, adapter id, sequence row or position out of range) never cause an
 *   out-of-bounds access: the offending token or query is skipped and, when
 *   `dev_status` is non-NULL, the first such error code is stored there
 *   (atomic compare-and-swap from 0). The caller zeroes *dev_status and reads it
 *   back when it wants to know. Bounded waits inside kernels that give up
 *   store LRKV_ERR_TIMEOUT the same way.
 */
#ifndef LRKV_H_
#define LRKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lrkv_stream_t; /* same type as cudaStream_t */

typedef enum {
  LRKV_OK = 0,
  LRKV_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative or inconsistent size */
  LRKV_ERR_UNSUPPORTED = 2,  /* well-formed but outside the supported shapes */
  LRKV_ERR_CUDA = 3,         /* a CUDA runtime call or a kernel launch failed */
  LRKV_ERR_INDEX = 4,        /* device side: an index out of range (entry skipped) */
  LRKV_ERR_TIMEOUT = 5,      /* device side: a bounded wait gave up */
  LRKV_ERR_WORKSPACE = 6     /* workspace NULL or smaller than the *_workspace_bytes query */
} lrkv_status;

typedef enum { LRKV_BF16 = 0, LRKV_FP32 = 1 } lrkv_dtype;

typedef enum { LRKV_CODEC_NONE = 0, LRKV_CODEC_POLYKV = 1 } lrkv_codec;

typedef struct {
  int32_t hidden;     /* h */
  int32_t n_q_heads;  /* Hq */
  int32_t n_kv_heads; /* Hkv */
  int32_t head_dim;   /* d: 64 or 128 */
  int32_t rank;       /* r: 8, 16, 32 or 64 */
  int32_t block_size; /* must be 16 */
  float rope_base;    /* theta_j = rope_base^(-2j/d) */
  int32_t dtype;      /* lrkv_dtype of every tensor argument */
  int32_t lr_groups;  /* G >= 1 low-rank groups: 1 = one A shared by every agent;
                         G > 1 = agent a has its own A_K,a, A_V,a and reads group a */
  int32_t kv_codec;   /* lrkv_codec of the base pool: NONE (bf16/fp32 planes) or POLYKV */
} lrkv_config;

/*
 * lrkv_base_pool_block_bytes -- bytes of one block of base_pool for cfg (all
 * kv heads): 2*Hkv*16*d*elem for LRKV_CODEC_NONE, Hkv*(23*d + 64) for
 * LRKV_CODEC_POLYKV; 0 for an invalid configuration. Host only.
 */
size_t lrkv_base_pool_block_bytes(const lrkv_config* cfg);

/*
 * lrkv_append -- write the cache entries of T new tokens.
 *
 * Defines: LRAgent (arXiv 2602.01053), Abstract -- the base component comes
 * from the pretrained weights and the adapter component is kept in its
 * low-rank form; PReCache, Abstract -- the low-rank cache is produced once,
 * when a context segment is first processed.
 *
 * Computes Y = X W_cat^T (one GEMM over h), then for token n at position
 * positions[n] of block-table row seq_rows[n]:
 *   base_pool[blk][0][k][row][:] = RoPE(Y[n, K cols of kv head k], position)
 *   base_pool[blk][1][k][row][:] = Y[n, V cols of kv head k]
 *   lr_pool[blk][0][row][:] = Y[n, A_K cols],  lr_pool[blk][1][row][:] = Y[n, A_V cols]
 *   (all G groups' columns)
 * with blk = block_tables[seq_rows[n]][positions[n] / 16], row = positions[n] % 16.
 *
 *   X            [T][h]                 hidden states of the new tokens
 *   T            >= 0 (0: no-op)
 *   positions    int32 [T]              position of each token in its sequence
 *   seq_rows     int32 [T]              block-table row of each token (< num_seqs)
 *   block_tables int32 [num_seqs][max_blocks]
 *   W_cat        [N][h], N = 2*Hkv*d + 2*G*r: the packed projection weights in
 *                nn.Linear layout (row n = weights of output column n):
 *                rows [0, Hkv*d) = W_K^T, [Hkv*d, 2*Hkv*d) = W_V^T,
 *                next G*r rows = A_K,0^T .. A_K,G-1^T, last G*r rows = A_V,g^T
 *   base_pool, lr_pool  written (only the rows of the T tokens)
 *   num_blocks   number of blocks in both pools (block ids must be < num_blocks)
 * Tokens whose row, position or block id is out of range are skipped
 * (LRKV_ERR_INDEX in dev_status). Two tokens mapping to the same slot race.
 */
lrkv_status lrkv_append(const lrkv_config* cfg, const void* X, int32_t T,
                        const int32_t* positions, const int32_t* seq_rows,
                        const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                        const void* W_cat, void* base_pool, void* lr_pool, int64_t num_blocks,
                        int32_t* dev_status, lrkv_stream_t stream);

/*
 * lrkv_append_rebase -- lrkv_append with the base and the low-rank part of
 * the cache written from different hidden states, or only one of the parts.
 *
 * Defines: PReCache (thelatestinai.com/papers/2609.34054), Abstract and
 * Figure 1 (ReBaseShared): the shared base cache is reconstructed from
 * adapter-free hidden states, which lowers the error that the previous
 * agent's adapted representation leaves in it; the reconstruction runs either
 * alongside the adapted pass (both paths batched together, "DB") or as a
 * separate prefill after the agent's turn ("LP").
 *
 * For token n (slot as in lrkv_append):
 *   X_base != NULL: base_pool rows = RoPE(X_base W_K), X_base W_V   (re-based)
 *   X_lr   != NULL: lr_pool rows   = X_lr A_K, X_lr A_V
 * A NULL source leaves that part of the pools untouched (X_lr = NULL is the
 * base-only re-base after a turn; X_base = X_lr is exactly lrkv_append). Both
 * NULL with T > 0 is LRKV_ERR_INVALID_ARG. One launch either way; X_base and
 * X_lr are [T][h], same dtype and alignment rules as X. Other arguments,
 * errors and dev_status: as lrkv_append.
 */
lrkv_status lrkv_append_rebase(const lrkv_config* cfg, const void* X_base, const void* X_lr, int32_t T,
                               const int32_t* positions, const int32_t* seq_rows,
                               const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                               const void* W_cat, void* base_pool, void* lr_pool, int64_t num_blocks,
                               int32_t* dev_status, lrkv_stream_t stream);

/*
 * lrkv_attn_decode -- one query token per query row, many agents per context.
 *
 * Defines: LRAgent (arXiv 2602.01053), Abstract -- Flash-LoRA-Attention
 * reconstructs each agent's adapter contribution from the shared low-rank
 * cache at attention time without expanding it to full dimension, and one
 * cached context serves every agent that reads it.
 *
 * Queries are grouped by the context they read: the queries of context c are
 * rows [ctx_q_start[c], ctx_q_start[c+1]) of q; all of them are served by one
 * sweep over that context's blocks (each base / low-rank tile is read once
 * for all of them). Each query sits at position ctx_lens[c] - 1 and attends
 * keys 0 .. ctx_lens[c] - 1 through its own adapter:
 *   out[n, m, :] = softmax_t(q[n,m,:] . K_a[t, m/g, :] * scale) V_a[t, m/g, :]
 * with K_a = K_base + RoPE(L_K B_K,a) and P V_a = P V_base + (P L_V) B_V,a.
 *
 *   q            [num_queries][Hq][d]   already rotated to its position
 *   ctx_q_start  int32 [num_ctx + 1]    non-decreasing, ctx_q_start[0] = 0,
 *                                        ctx_q_start[num_ctx] = num_queries
 *   adapter_ids  int32 [num_queries]    in [-1, n_adapters)
 *   block_tables int32 [num_ctx][max_blocks]   row c = context c
 *   ctx_lens     int32 [num_ctx]        keys per context, in [1, max_ctx_len]
 *   max_ctx_len  host int, >= every ctx_lens[c] (sizes the split plan)
 *   max_q_per_ctx host int, >= every ctx_q_start[c+1] - ctx_q_start[c]
 *   B_K, B_V     [n_adapters][r][Hkv*d] or NULL (zero factor)
 *   out          [num_queries][Hq][d]   written
 *   workspace    >= lrkv_decode_workspace_bytes(...) bytes (fp32 split partials
 *                and bookkeeping); contents need no initialisation and are
 *                garbage afterwards
 * Two kernel launches: the split-KV sweep, then a merge of the splits that
 * applies B_V.
 * A context with zero queries is skipped; ctx_lens[c] outside
 * [1, max_ctx_len] or a bad block / adapter id gives LRKV_ERR_INDEX in
 * dev_status and zero output for the affected queries. A context with more
 * queries than max_q_per_ctx gives LRKV_ERR_INDEX and zero output for the
 * query heads past the planned rows; a query that no valid ctx_q_start range
 * holds (ranges that decrease, or do not cover [0, num_queries)) gives
 * LRKV_ERR_INDEX and zero output.
 */
lrkv_status lrkv_attn_decode(const lrkv_config* cfg, const void* q, int32_t num_queries,
                             const int32_t* ctx_q_start, int32_t num_ctx,
                             const int32_t* adapter_ids, const int32_t* block_tables,
                             int32_t max_blocks, const int32_t* ctx_lens, int32_t max_ctx_len,
                             int32_t max_q_per_ctx, const void* base_pool, const void* lr_pool,
                             int64_t num_blocks, const void* B_K, const void* B_V,
                             int32_t n_adapters, float scale, void* out, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, lrkv_stream_t stream);

/* Bytes of workspace lrkv_attn_decode needs for these sizes on the current
 * device (the split plan depends on the device's SM count). 0 on bad input. */
size_t lrkv_decode_workspace_bytes(const lrkv_config* cfg, int32_t num_queries, int32_t num_ctx,
                                   int32_t max_ctx_len, int32_t max_q_per_ctx);

/*
 * lrkv_attn_prefill -- a causal chunk of queries per sequence, one adapter per
 * sequence.
 *
 * Defines: LRAgent (arXiv 2602.01053), Abstract (Flash-LoRA-Attention, as for
 * decode); PReCache, Abstract (a new turn attends over the shared context
 * already cached by earlier agents plus its own new tokens).
 *
 * Sequence s owns query rows [q_start[s], q_start[s+1]) of q (q_len of them)
 * and has seq_lens[s] keys in its block-table row (its own new tokens
 * included, appended before this call). Query k sits at position
 * seq_lens[s] - q_len + k and attends keys at positions <= its own through
 * adapter adapter_ids[s].
 *
 *   q            [total_q][Hq][d]       already rotated
 *   q_start      int32 [num_seqs + 1]   non-decreasing, q_start[0] = 0,
 *                                        q_start[num_seqs] = total_q
 *   max_q_len    host int, >= every q_len (sizes the grid)
 *   seq_lens     int32 [num_seqs]       >= q_len of that sequence
 *   max_seq_len  host int, >= every seq_lens[s]
 *   adapter_ids  int32 [num_seqs]       in [-1, n_adapters)
 *   block_tables int32 [num_seqs][max_blocks]
 *   out          [total_q][Hq][d]       written
 *   workspace    may be NULL when lrkv_prefill_workspace_bytes(...) is 0
 */
lrkv_status lrkv_attn_prefill(const lrkv_config* cfg, const void* q, const int32_t* q_start,
                              int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                              const int32_t* seq_lens, int32_t max_seq_len,
                              const int32_t* adapter_ids, const int32_t* block_tables,
                              int32_t max_blocks, const void* base_pool, const void* lr_pool,
                              int64_t num_blocks, const void* B_K, const void* B_V,
                              int32_t n_adapters, float scale, void* out, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, lrkv_stream_t stream);

size_t lrkv_prefill_workspace_bytes(const lrkv_config* cfg, int32_t num_seqs, int32_t total_q,
                                    int32_t max_q_len, int32_t max_seq_len);

/*
 * lrkv_attn_mixed -- one call for a mixed batch: decode queries and causal
 * prefill chunks over the same pools and adapters.
 *
 * Defines: Efficient Multi-Adapter LLM Serving via Cross-Model KV-Cache Reuse
 * with Activated LoRA, "Builds on" (SARATHI: decodes piggybacked on chunked
 * prefills in one batch); PReCache, Figure 4 (serving, where agents' prefills
 * and decodes share the GPU). Each part computes exactly what
 * lrkv_attn_decode and lrkv_attn_prefill compute for it: the result is
 * bitwise that of the two calls made one after the other.
 *
 * The two parts run at the same time: the prefill on `stream`, the decode on
 * a second stream of the library's own, forked from `stream` by an event and
 * joined back to it by another before the call returns, so work queued on
 * `stream` afterwards sees both outputs. The decode's CTAs then take the SMs
 * the prefill grid leaves idle in its last wave. The second stream and the
 * two events are created on the first mixed call of each host thread on each
 * device and kept until the process exits (also when that thread ends before
 * it); make that first call outside any stream capture. Later calls may be captured into a CUDA graph (the fork and
 * the join become graph edges).
 *
 *   dec, pre   either may be NULL or describe an empty batch (num_queries or
 *              num_ctx 0; num_seqs or total_q 0); with one part empty the
 *              other runs on `stream` alone.
 *   Fields of lrkv_decode_batch and lrkv_prefill_batch: as the arguments of
 *   the same names of lrkv_attn_decode and lrkv_attn_prefill; the pools,
 *   the adapter factors, n_adapters, scale and dev_status are shared.
 *
 * Errors: both parts are checked before anything is launched; the first
 * failing check's status is returned (decode first) and nothing runs.
 * LRKV_ERR_CUDA if the second stream or its events cannot be made.
 */
typedef struct lrkv_decode_batch {
  const void* q;
  int32_t num_queries;
  const int32_t* ctx_q_start;
  int32_t num_ctx;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* ctx_lens;
  int32_t max_ctx_len;
  int32_t max_q_per_ctx;
  void* out;
  void* workspace;
  size_t workspace_bytes;
} lrkv_decode_batch;

typedef struct lrkv_prefill_batch {
  const void* q;
  const int32_t* q_start;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_q_len;
  const int32_t* seq_lens;
  int32_t max_seq_len;
  const int32_t* adapter_ids;
  const int32_t* block_tables;
  int32_t max_blocks;
  void* out;
} lrkv_prefill_batch;

lrkv_status lrkv_attn_mixed(const lrkv_config* cfg, const lrkv_decode_batch* dec,
                            const lrkv_prefill_batch* pre, const void* base_pool, const void* lr_pool,
                            int64_t num_blocks, const void* B_K, const void* B_V, int32_t n_adapters,
                            float scale, int32_t* dev_status, lrkv_stream_t stream);

/*
 * lrkv_attn_decode_noalloc -- lrkv_attn_decode for callers that cannot
 * allocate device memory.
 *
 * The paper has no counterpart: this is a library convenience. Some callers
 * cannot call cudaMalloc (or any routine that allocates) where they run
 * decode, e.g. a runtime whose device memory is reserved once at start-up, or
 * a serving loop that forbids allocation; they cannot supply the workspace of
 * lrkv_attn_decode. This entry point takes the same arguments minus the
 * workspace and uses instead a fixed scratch array of
 * LRKV_NOALLOC_SCRATCH_BYTES held in the library's own device memory (every
 * GPU that loads the library keeps it until the process exits). It allocates
 * nothing.
 *
 * - Result: identical to lrkv_attn_decode with a workspace of its own.
 * - Limit: sizes for which lrkv_decode_workspace_bytes(...) exceeds
 *   LRKV_NOALLOC_SCRATCH_BYTES return LRKV_ERR_WORKSPACE before any launch.
 * - First call on a device: resolves the array's device address for that
 *   device (with that device current) and caches it; make that first call
 *   before any stream capture on the device. The cached address belongs to
 *   the device's current context: after cudaDeviceReset (or anything else
 *   that destroys the primary context) this entry point must not be called
 *   again in the same process, since the array may then live elsewhere.
 * - Sharing: every call on a device uses the same array. Nothing in it needs
 *   to start at zero (it holds split partials that are written before they
 *   are read), but calls whose kernels overlap on the GPU (on different
 *   streams, or from several threads) race on it and give wrong results;
 *   order them on one stream or with events.
 * Other arguments, errors and dev_status: as lrkv_attn_decode.
 */
#define LRKV_NOALLOC_SCRATCH_BYTES (16u << 20)
lrkv_status lrkv_attn_decode_noalloc(const lrkv_config* cfg, const void* q, int32_t num_queries,
                                     const int32_t* ctx_q_start, int32_t num_ctx,
                                     const int32_t* adapter_ids, const int32_t* block_tables,
                                     int32_t max_blocks, const int32_t* ctx_lens,
                                     int32_t max_ctx_len, int32_t max_q_per_ctx,
                                     const void* base_pool, const void* lr_pool,
                                     int64_t num_blocks, const void* B_K, const void* B_V,
                                     int32_t n_adapters, float scale, void* out,
                                     int32_t* dev_status, lrkv_stream_t stream);

/* Static string naming a status code. */
const char* lrkv_status_string(lrkv_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t lrkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LRKV_H_ */
