/*
 * pa.h -- C ABI of libpagedattn: attention over a paged KV cache on GB300
 * (sm_103a).
 *
 * The operations follow the pages this library is built from:
 *   - "KV Cache > The Idea" on the LLM inference engine work-log
 *     (shehab-ashraf.github.io/posts/llm-inference): each step appends the new
 *     tokens' K and V to the cache, then the new queries attend over the whole
 *     history;
 *   - "S20 - The Complete Engine", section "Core idea" (the engine's step()
 *     loop): each request's block_table maps its logical blocks to physical
 *     blocks that the block manager allocated;
 *   - the course README "Build an LLM Inference Engine From Scratch",
 *     curriculum rows "Memory & KV Cache" (PagedAttention, GQA) and
 *     "Batching & Scheduling" (chunked prefill, FlashAttention), and the
 *     claims "online softmax is exact; paged and split-K variants agree",
 *     "chunked prefill produces a bit-identical KV cache".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *   - Pointers are DEVICE pointers unless stated otherwise. The caller owns
 *     and allocates every buffer, including the workspace. The library
 *     allocates no memory and never synchronises the stream on these calls.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t passed
 *     as void*; NULL = the legacy default stream) of the CURRENT device.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (pa_bf16 = uint16_t).
 *   - KV cache layout: k_cache and v_cache are separate arrays, each
 *     [num_blocks][num_kv_heads][block_size][head_dim], contiguous. The
 *     (block, kv head) tile of one block is block_size*head_dim contiguous
 *     elements (4 KB at block_size 16, head_dim 128).
 *   - A slot is phys_block * block_size + offset_in_block.
 *   - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - context_lens[s] counts every token of sequence s that its queries may
 *     see, INCLUDING the step's own new tokens (written first by
 *     pa_reshape_and_cache). Query j of a sequence with q_len Lq sits at
 *     position context_len - Lq + j.
 *   - lse is the natural-log log-sum-exp of the scaled logits
 *     (scale * q.k) over the keys a query sees, fp32, one per (query, head).
 *   - Return value: PA_OK (0) or a negative pa_status. Host-side argument
 *     checks run before anything is enqueued; a failing call enqueues nothing.
 *     Values that live in device memory (slots, block ids, lengths) are
 *     range-checked by the kernels: an out-of-range value sets a bit of the
 *     device error word (read it with pa_debug_read_error) and the offending
 *     access is skipped or clamped, never performed -- the kernels do not
 *     trap. Results for the affected rows are then undefined.
 *
 * Built configuration: head_dim 128, block_size 16, and num_q_heads /
 * num_kv_heads = 2 for pa_decode (1..8 for pa_decode_varlen with
 * q tiles of 16 / group rows). Other shapes return PA_ERR_UNSUPPORTED.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pa_bf16;

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_ARG = -1,         /* null pointer, negative size, inconsistent shape */
  PA_ERR_UNSUPPORTED = -2, /* shape not built (head_dim, block_size, group) */
  PA_ERR_WORKSPACE = -3,   /* workspace missing, misaligned or too small */
  PA_ERR_CUDA = -4,        /* a CUDA runtime call (launch, attribute query) failed */
  PA_ERR_DEVICE = -5       /* device-side check failed (see pa_debug_read_error) */
} pa_status;

/* Bits of the device error word (pa_debug_read_error). */
#define PA_DEVERR_SLOT_RANGE 0x1u    /* slot_mapping[t] >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_RANGE 0x2u   /* a used block_tables entry outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_RANGE 0x4u /* context_len < 0 or > max_blocks_per_seq * block_size */
#define PA_DEVERR_QLEN_RANGE 0x8u    /* q_len < 0, q_len > context_len (causal, or context 0), or cu_seqlens_q inconsistent */
#define PA_DEVERR_PIPE_TIMEOUT 0x10u /* an asynchronous copy did not land within its time limit */
#define PA_DEVERR_PLAN_OVERFLOW 0x20u /* work list larger than the launch was sized for */

/* Problem shape, passed by pointer (host memory) to every call. */
typedef struct pa_shape {
  int num_seqs;           /* S: sequences in the batch */
  int num_q_heads;        /* Hq */
  int num_kv_heads;       /* Hkv; Hq % Hkv == 0 */
  int head_dim;           /* D (built: 128) */
  int block_size;         /* BS, tokens per physical block (built: 16) */
  int max_blocks_per_seq; /* row length of block_tables */
  int64_t num_blocks;     /* physical blocks in each of k_cache / v_cache */
} pa_shape;

/*
 * pa_reshape_and_cache -- slot-mapped write of the step's new K/V rows into
 * the block pool ("KV Cache > The Idea": the new K and V are appended to the
 * cache; the course README's chunked-prefill claim: writing in chunks gives a
 * bit-identical cache).
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim] bf16, contiguous
 *   slot_mapping  [num_tokens] int64; slot < 0 means "skip this token"
 *   k_cache, v_cache  the pool, layout above; written in place
 *   shape         uses num_kv_heads, head_dim, block_size, num_blocks
 *
 * For every t with slot_mapping[t] >= 0 it copies the bytes of k[t][h][:]
 * to k_cache[slot / BS][h][slot % BS][:] (V alike). A pure byte copy: the
 * result is bit-exact. Two tokens with the same slot in one call race
 * (undefined which one lands). A slot >= num_blocks*block_size is skipped
 * and sets PA_DEVERR_SLOT_RANGE. num_tokens == 0 is a no-op.
 */
int pa_reshape_and_cache(const pa_bf16* k, const pa_bf16* v, const int64_t* slot_mapping,
                         int64_t num_tokens, pa_bf16* k_cache, pa_bf16* v_cache,
                         const pa_shape* shape, void* stream);

/*
 * pa_decode -- one query token per sequence (q_len 1) attending over its
 * paged context: block-table gather, GQA sharing of each K/V tile by the
 * group's query heads, online softmax, and split-K over long contexts with a
 * log-sum-exp merge ("online softmax is exact; paged and split-K variants
 * agree").
 *
 *   q             [S][Hq][D] bf16
 *   k_cache, v_cache  pool (read only)
 *   block_tables  [S][max_blocks_per_seq] int32; entries past a sequence's
 *                 ceil(context_len / BS) blocks are never read
 *   context_lens  [S] int32, 0 <= c <= max_blocks_per_seq * BS. c == 0 gives
 *                 out = 0 and lse = -inf for that sequence.
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(D))
 *   out           [S][Hq][D] bf16 (round to nearest even from fp32)
 *   lse           [S][Hq] fp32, natural log; may be NULL if not wanted
 *   num_splits    0  = balanced: the library cuts the batch's total K/V tile
 *                      count into equal contiguous ranges, one per resident
 *                      warp, and merges the pieces of sequences that were cut;
 *                 1  = no split: one warp per (sequence, KV head);
 *                 P >= 2 = every (sequence, KV head) is cut into P near-equal
 *                      block ranges (partitions; P <= 1024); each partition's
 *                      normalised output and log-sum-exp are merged with the
 *                      pa_splitk_reduce formula (empty partitions weigh
 *                      nothing). The partitions' tiles are spread over the
 *                      resident warps like num_splits 0 does with sequences.
 *   workspace     device scratch of at least pa_decode_workspace_size(...)
 *                 bytes, 256-byte aligned; may be NULL when that size is 0.
 *                 Its contents need no initialisation and are clobbered.
 */
int pa_decode(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale,
              pa_bf16* out, float* lse, const pa_shape* shape, int num_splits,
              void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace pa_decode needs for this shape and num_splits on the
 * current device (0 when num_splits == 1). */
size_t pa_decode_workspace_size(const pa_shape* shape, int num_splits);

/*
 * pa_append_decode -- one decode step of one attention layer in one call:
 * pa_reshape_and_cache(k_new, v_new, slot_mapping, num_new_tokens, ...)
 * followed by pa_decode(..., num_splits = 0, ...) ("KV Cache > The Idea":
 * append the new K/V, then attend over the whole history). Same arguments,
 * layouts, results and workspace (pa_decode_workspace_size(shape, 0)) as the
 * two calls. The decode grid is queued as a programmatic dependent of the
 * cache-write grid and prepares its work (reading context_lens and
 * block_tables) while the write runs, then streams every tile of the pool
 * except the last block of each (sequence, KV head) at once; a last block is
 * copied only after the write has finished. So: each new row must land in
 * the block that holds its sequence's last position (context_lens[s] - 1:
 * the decode step's own token), and context_lens and block_tables must not
 * alias k_new, v_new, slot_mapping or the pool.
 */
int pa_append_decode(const pa_bf16* k_new, const pa_bf16* v_new, const int64_t* slot_mapping,
                     int64_t num_new_tokens, const pa_bf16* q, pa_bf16* k_cache,
                     pa_bf16* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                     float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_static_scratch -- pa_decode with num_splits == 0 (balanced split)
 * that allocates nothing and takes no workspace. The source pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory themselves -- a plugin inside another runtime that owns every device
 * allocation, or a serving loop whose memory is planned once up front (where a
 * cudaMalloc would also synchronise the device).
 *
 * Arguments, layouts and results are those of pa_decode. The split scratch is
 * a fixed 8 MiB array inside the library (static device memory that every GPU
 * loading the library holds until the process exits). A shape whose balanced
 * split needs more than 8 MiB on the current device returns PA_ERR_WORKSPACE
 * (use pa_decode with a workspace instead); the need is 2 partial slots x 2
 * heads x 129 fp32 per resident warp of the decode grid: 3.6 MiB on a 152-SM
 * GB300, for any batch. The first call in each CUDA context looks up the
 * array's device address (cudaGetSymbolAddress) with that context current;
 * make that first call before any stream capture. All calls share the one
 * array and its contents carry over between calls (nothing in it needs to
 * start at zero): calls that may overlap on the GPU -- on different streams,
 * or from different host threads -- race on it and must be serialised by the
 * caller.
 */
int pa_decode_static_scratch(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                             void* stream);

/*
 * pa_decode_varlen -- several query tokens per sequence over the same paged
 * pool: speculative-decoding verify (1 + k draft tokens, causal within the
 * query window; "S20 - The Complete Engine", step 3 PROPOSE and step 5
 * verify) and chunked prefill (a chunk of queries at an offset whose earlier
 * tokens are already cached; course README, "chunked prefill"). QK^T and PV
 * run on the tensor cores. Sequences with q_len < 32 (verify windows, short
 * chunks) go through warp-level MMA tiles of 16 rows = (16 / G) query tokens x
 * G query heads of one KV head; when max_q_len >= 32 and 128 % G == 0,
 * sequences with q_len >= 32 go through a second kernel on the fifth-
 * generation tensor cores (tcgen05, accumulators in tensor memory) in tiles
 * of 128 rows x 128 keys. Both kernels are launched on `stream`, in order;
 * the results do not depend on which kernel a sequence went through beyond
 * floating-point rounding.
 *
 *   q             [num_q_tokens][Hq][D] bf16; sequence s owns rows
 *                 cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1
 *   cu_seqlens_q  [S+1] int32, cu_seqlens_q[0] == 0,
 *                 cu_seqlens_q[S] == num_q_tokens, non-decreasing
 *   max_q_len     an upper bound of the q_lens (host value, sizes the launch)
 *   causal        1: query j sees keys 0 .. c - Lq + j (needs Lq <= c);
 *                 0: it sees 0 .. c - 1 (any Lq when c > 0)
 *   out, lse      [num_q_tokens][Hq][D] bf16, [num_q_tokens][Hq] fp32 (lse may
 *                 be NULL)
 *   workspace     at least pa_decode_varlen_workspace_size(...) bytes,
 *                 256-byte aligned; clobbered.
 * Work is balanced like pa_decode with num_splits == 0. A sequence with
 * q_len 0 produces no rows.
 */
int pa_decode_varlen(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens,
                     const int32_t* cu_seqlens_q, int64_t num_q_tokens, int max_q_len,
                     int causal, float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                     void* workspace, size_t workspace_bytes, void* stream);

size_t pa_decode_varlen_workspace_size(const pa_shape* shape, int64_t num_q_tokens,
                                       int max_q_len);

/*
 * INT8 KV cache (course README, curriculum row "Memory & KV Cache":
 * quantization; "What to build in what order": quantization when memory or
 * bandwidth binds; the "INT8 KV" configuration; claim "s08": grouping keeps
 * outliers in check and dequantisation must be fused or it moves more bytes
 * than fp16). A second pool format that halves the bytes of the decode stream:
 *
 *   k_cache, v_cache  bytes, [num_blocks][num_kv_heads][PA_INT8_TILE_BYTES]:
 *                     one tile per (block, KV head) = the block_size rows'
 *                     codes, int8 [block_size][head_dim] (2048 bytes), then
 *                     the same rows' fp32 scales [block_size] (64 bytes); one
 *                     scale per (token, KV head) row of head_dim values.
 *                     A tile is one contiguous 2112-byte run (a multiple of 16).
 *
 * Row quantisation (symmetric, group = one head row): amax = max_d |x_d|;
 * if amax == 0 every code is 0 and the scale 0; otherwise
 * inv = fl(127 / amax), code_d = clamp(rint(fl(x_d * inv)), -127, 127) with
 * rint rounding half to even, scale = fl(amax / 127), where fl() is one
 * IEEE fp32 operation rounded to nearest even. A row dequantises to
 * code_d * scale. Rows are written once, so a block's earlier rows never
 * change when later tokens arrive.
 */
#define PA_INT8_TILE_BYTES 2112

/*
 * pa_reshape_and_cache_int8 -- pa_reshape_and_cache into the int8 pool: for
 * every t with slot_mapping[t] >= 0, row k[t][h][:] is quantised as above
 * into the codes of row slot % BS of tile (slot / BS, h) of k_cache and its
 * scale into that tile's scale slot slot % BS (V alike). Pointers 16-byte
 * aligned (slot_mapping 8). Same slot rules and error bits as
 * pa_reshape_and_cache. bf16 inputs that are subnormal are read as zero (the
 * kernels flush fp32 subnormals).
 */
int pa_reshape_and_cache_int8(const pa_bf16* k, const pa_bf16* v, const int64_t* slot_mapping,
                              int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                              const pa_shape* shape, void* stream);

/*
 * pa_decode_int8 -- pa_decode over the int8 pool, dequantisation fused: each
 * score is the int8 row dot product times the row's K scale, and each
 * softmax weight is multiplied by the row's V scale before it meets the
 * int8 V row. Same arguments, splits, outputs and workspace rules as
 * pa_decode (workspace from pa_decode_int8_workspace_size); k_cache and
 * v_cache 16-byte aligned. The result is attention over the dequantised
 * rows: q and the codes enter the products exactly and all sums are fp32;
 * each softmax weight times its row's V scale is rounded to f16 relative to
 * the largest such product of its head in the 16-token block (relative error
 * 2^-11, as when P is rounded to 16 bits); the log-sum-exp comes from fp32
 * sums.
 */
int pa_decode_int8(const pa_bf16* q, const uint8_t* k_cache, const uint8_t* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens, float scale,
                   pa_bf16* out, float* lse, const pa_shape* shape, int num_splits,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for pa_decode_int8 with this shape and split choice. */
size_t pa_decode_int8_workspace_size(const pa_shape* shape, int num_splits);

/*
 * FP8 KV cache (course pages, "The curriculum": the Machine layer names
 * bf16/fp8 and the Memory & KV Cache layer quantization). The same tile
 * layout as the int8 pool (PA_INT8_TILE_BYTES per (block, KV head): the
 * block_size rows' codes, then their fp32 scales), with each code an OCP
 * FP8 E4M3 byte: sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, 0x7F / 0xFF = NaN, largest finite value 448.
 *
 * Row quantisation (group = one head row): amax = max_d |x_d|; if amax == 0
 * every code is 0 and the scale 0; otherwise inv = fl(448 / amax),
 * code_d = the E4M3 value nearest to fl(x_d * inv) (ties to the code with
 * an even last mantissa bit; beyond +-448 it saturates to +-448),
 * scale = fl(amax / 448). The writer never stores a NaN code. A row
 * dequantises to value(code_d) * scale.
 */

/*
 * pa_reshape_and_cache_fp8 -- pa_reshape_and_cache_int8 with E4M3 codes
 * (quantised as above). Same layout, alignment, slot rules and error bits;
 * bf16 subnormal inputs are read as zero.
 */
int pa_reshape_and_cache_fp8(const pa_bf16* k, const pa_bf16* v, const int64_t* slot_mapping,
                             int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                             const pa_shape* shape, void* stream);

/*
 * pa_decode_fp8 -- pa_decode over the FP8 pool, dequantisation fused: each
 * score is the decoded row's dot product times the row's K scale, and each
 * softmax weight is multiplied by the row's V scale before it meets the
 * decoded V row. Rows past a sequence's context are never read into the
 * result (they may hold anything, NaN codes included). Same arguments,
 * splits, outputs and workspace rules as pa_decode (workspace from
 * pa_decode_fp8_workspace_size); k_cache and v_cache 16-byte aligned. The
 * result is attention over the dequantised rows, with the precision stated
 * for pa_decode_int8.
 */
int pa_decode_fp8(const pa_bf16* q, const uint8_t* k_cache, const uint8_t* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  pa_bf16* out, float* lse, const pa_shape* shape, int num_splits,
                  void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for pa_decode_fp8 with this shape and split choice. */
size_t pa_decode_fp8_workspace_size(const pa_shape* shape, int num_splits);

/*
 * pa_decode_cascade -- pa_decode (q_len 1, balanced) for a batch in which
 * groups of sequences share the physical blocks of a prompt prefix (prefix
 * caching: course README, "What to build in what order"; "S20 - The Complete
 * Engine", "The conflicts": reference-counted shared blocks). Same result as
 * pa_decode on the same q, pool, block_tables and context_lens (to fp32
 * rounding): attention splits into the shared prefix, attended once per group
 * by all its members together (non-causal multi-query tile on the tcgen05
 * path, so the prefix's K/V are read once per group), and each sequence's own
 * suffix (balanced decode), merged with the split-K formula.
 *
 *   seq_group      [S] int32: the group of sequence s, or -1
 *   num_groups     G (host)
 *   cu_group       [G+1] int32, cu_group[0] = 0: group g's members are
 *                  group_members[cu_group[g] .. cu_group[g+1]-1]
 *   group_members  [num_members] int32 sequence ids, increasing within a
 *                  group, each sequence in at most one group
 *   prefix_lens    [G] int32 prefix tokens of each group: > 0, a multiple of
 *                  block_size, <= every member's context_len and <=
 *                  max_prefix_len. Every member's first prefix_lens[g] /
 *                  block_size block_tables entries are the same physical
 *                  blocks (the library reads them from the first member).
 *   num_members, max_group_size (>= every group's size), max_prefix_len
 *                  (a multiple of block_size): host bounds that size the launch
 *   workspace      pa_decode_cascade_workspace_size(...) bytes, 256-byte
 *                  aligned, clobbered.
 * A description that breaks these rules sets PA_DEVERR_QLEN_RANGE or
 * PA_DEVERR_CONTEXT_RANGE; the output is then unspecified. Built for
 * num_q_heads == 2 * num_kv_heads (as pa_decode).
 *
 * pa_decode_cascade chooses between the cascade and plain pa_decode
 * (PA_CASCADE_AUTO below): the cascade's extra phases (gathering the members'
 * queries, the prefix tile, two merges) pay only when the prefix reads it
 * saves are large, so when the bound of those bytes, (num_members -
 * num_groups) x max_prefix_len x num_kv_heads x head_dim x 4, is below
 * 256 MiB per 64 members (at least 64) -- the crossover measured on GB300 --
 * the call runs pa_decode (num_splits 0) on the same arguments instead, and
 * the group description is not read.
 */
int pa_decode_cascade(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      const int32_t* seq_group, int num_groups, const int32_t* cu_group,
                      const int32_t* group_members, const int32_t* prefix_lens,
                      int num_members, int max_group_size, int max_prefix_len, float scale,
                      pa_bf16* out, float* lse, const pa_shape* shape, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Policies of pa_decode_cascade_ex. */
#define PA_CASCADE_AUTO 0   /* the cascade if its saved prefix bytes pay for it (see above) */
#define PA_CASCADE_ALWAYS 1 /* always the cascade */
#define PA_CASCADE_PLAIN 2  /* always plain pa_decode (the description is not read) */

/* pa_decode_cascade with the choice made by the caller (policy, above). */
int pa_decode_cascade_ex(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens,
                         const int32_t* seq_group, int num_groups, const int32_t* cu_group,
                         const int32_t* group_members, const int32_t* prefix_lens,
                         int num_members, int max_group_size, int max_prefix_len, float scale,
                         pa_bf16* out, float* lse, const pa_shape* shape, int policy,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for pa_decode_cascade and pa_decode_cascade_ex under any
 * policy (0 if the arguments are invalid). */
size_t pa_decode_cascade_workspace_size(const pa_shape* shape, int num_groups, int num_members,
                                        int max_group_size, int max_prefix_len);

/*
 * pa_splitk_reduce -- merge of split-K partial softmax results (course
 * README, "online softmax is exact; paged and split-K variants agree").
 * For each (row, head):
 *   M = max_i lse_i,  LSE = M + ln sum_i exp(lse_i - M),
 *   out = sum_i exp(lse_i - LSE) * o_i,  lse_out = LSE.
 * Partials with lse_i = -inf are empty and weigh 0; a row whose partials are
 * all empty gives out = 0 and lse_out = -inf.
 *
 *   part_out  [num_rows][num_heads][num_splits][head_dim] fp32 (each o_i is
 *             already normalised by its own softmax sum)
 *   part_lse  [num_rows][num_heads][num_splits] fp32, natural log
 *   out       [num_rows][num_heads][head_dim] bf16
 *   lse       [num_rows][num_heads] fp32, may be NULL
 * head_dim must be a multiple of 4 and at most 1024; num_splits >= 1.
 */
int pa_splitk_reduce(const float* part_out, const float* part_lse, int64_t num_rows,
                     int num_heads, int num_splits, int head_dim, pa_bf16* out, float* lse,
                     void* stream);

/* Text for a pa_status value (static storage). */
const char* pa_status_string(int status);

/*
 * pa_debug_read_error -- synchronises `stream`, returns the device error word
 * (an OR of PA_DEVERR_* bits, 0 if nothing was flagged) accumulated by every
 * kernel of this library on the current device since the last read, and
 * clears it. Returns PA_ERR_CUDA (negative) if the synchronisation or the
 * copy fails. Not for the hot path: it blocks the host.
 */
int pa_debug_read_error(void* stream);

/*
 * pa_debug_inject_missing_copy -- failure-detection test hook. The next
 * decode launch (pa_decode, pa_append_decode, pa_decode_int8, pa_decode_fp8 or
 * pa_decode_static_scratch) on this host thread leaves out the copy of flat
 * tile `flat_tile` of its work list (0 = the first (sequence 0, KV head 0,
 * block 0) tile), so the warp that waits for it runs into its bounded wait
 * (2 s), sets PA_DEVERR_PIPE_TIMEOUT and returns; the kernel exits, nothing
 * traps and the context stays usable (that call's output is unspecified).
 * A negative value clears a pending injection. Returns PA_OK.
 */
int pa_debug_inject_missing_copy(int flat_tile);

/* Library version string, e.g. "pagedattn 0.1 sm_103a". */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
