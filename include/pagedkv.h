/*
 * pagedkv.h -- C ABI of the paged-KV decode attention library (libpagedkv.so),
 * written for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the problem the paged-KV pages state:
 *   - inferd README, "Paged KV" phase (block allocator + page table) and the
 *     "Paged KV equivalence" result: each sequence's K/V live in fixed-size
 *     physical blocks addressed through a per-sequence block table, and
 *     attention through the table equals dense attention.
 *   - lfm25-inference README, "Paged GQA/XQA Decode Attention: zero-allocation
 *     paged KV caching with Split-K reduction", "--page-size 16", and the
 *     runtime principles "KV pages are managed by the engine", "temporary
 *     device memory is reused through bounded pools", "precision and page size
 *     are startup policies".
 *
 * Conventions for every entry point
 *   - All pointers named *_cache, q, out, k_new, v_new, slot_mapping,
 *     block_tables, context_lens, q_lens, *_scales, workspace, device_error
 *     are DEVICE pointers on the current CUDA device.  The caller owns every
 *     buffer; the library allocates nothing and keeps no state besides cached
 *     device attributes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no entry point synchronises
 *     except pkv_read_device_error.
 *   - Host-side argument checks run before anything is launched; a non-OK
 *     status means nothing was enqueued (except PKV_ERR_CUDA, which reports a
 *     failed launch).
 *   - Indices the host cannot see (block ids, slots, lengths) are checked on
 *     the device: an out-of-range value sets a device error word (see
 *     pkv_read_device_error) and the access is skipped; the kernels never
 *     trap.  Outputs of such a call are unspecified.
 *
 * Cache layout (fixed per cache).  K and V are each
 *     [num_blocks][num_kv_heads][page]
 * where a page holds the block_size = 16 tokens of one block for one kv-head,
 * laid out as 16-byte chunks:
 *     page = [16 / 8][head_dim / C][8][C],   C = 16 / element bytes
 * (C = 8 for bf16, 16 for fp8): two groups of 8 tokens; inside a group, one
 * 16-byte chunk of the head dimension after another; inside a chunk, the 8
 * tokens of the group, each contributing C consecutive elements.  Element
 * (token off, dim d) of a page sits at element index
 *     ((off / 8) * (head_dim / C) + d / C) * 8 * C + (off % 8) * C + d % C.
 * Each 8x16-byte core block of a page is one contiguous 128-byte unit, so a
 * page copied to shared memory unchanged is directly a tensor-core operand.
 * A token slot is  slot = block * 16 + off.
 *
 * FP8 cache (kv_dtype = PKV_KV_FP8_E4M3): OCP E4M3 ("fn": bias 7, no
 * infinities, max finite 448) with one fp32 scale per (block, kv-head) for K
 * and one for V, k_scales / v_scales = [num_blocks][num_kv_heads].  Stored
 * code = e4m3_rne_satfinite( (float)x / scale ) (IEEE fp32 division);
 * dequantised value = code value * scale.  Scales are inputs (the caller
 * computes them, e.g. absmax / 448 per block).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
    PKV_ERR_UNSUPPORTED = 2,   /* head_dim / block_size / dtype / group size not built */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or too small */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE_INDEX = 5,  /* device error word: bad block id / slot / length / value range */
    PKV_ERR_TIMEOUT = 6,       /* device error word: a bounded wait gave up */
    PKV_ERR_NO_BLOCKS = 7,     /* block manager: no free block and none evictable */
    PKV_ERR_UNKNOWN_SEQ = 8    /* block manager: no sequence with that id (or it exists already) */
} pkv_status;

typedef enum pkv_kv_dtype { PKV_KV_BF16 = 0, PKV_KV_FP8_E4M3 = 1 } pkv_kv_dtype;

/* Device error word values (bit flags, OR-ed together by the kernels). */
#define PKV_DEVERR_BLOCK_ID 1   /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_LENGTH 2     /* q_len > context_len, or a negative length */
#define PKV_DEVERR_SLOT 4       /* slot >= num_blocks * 16 in an append */
#define PKV_DEVERR_TIMEOUT 8    /* a bounded wait inside a kernel expired */
#define PKV_DEVERR_RANGE 16     /* pkv_paged_prefill: a finite V value of magnitude >= 65536;
                                   pkv_paged_attention, FP8 cache on the tensor cores: a V scale
                                   above 255 */

/* One paged cache ("startup policy": fixed for its lifetime). */
typedef struct pkv_cache {
    int64_t num_blocks;        /* physical blocks in the pool */
    int32_t block_size;        /* must be 16 */
    int32_t num_kv_heads;      /* Hkv >= 1 */
    int32_t head_dim;          /* 64 or 128 */
    int32_t kv_dtype;          /* pkv_kv_dtype */
    void* k_cache;             /* device, layout above, 16-byte aligned */
    void* v_cache;
    const float* k_scales;     /* device [num_blocks][Hkv] fp32; NULL for bf16 */
    const float* v_scales;
} pkv_cache;

/*
 * paged_kv_append -- write one step's new K/V rows into their block slots
 * (lfm25-inference file list, kernels/kv_cache.cu; scheduler/slots.rs).
 *
 *   k_new, v_new   device bf16 [num_tokens][Hkv][head_dim], row-major, 16-byte aligned
 *   slot_mapping   device int64 [num_tokens]; slot = block * 16 + offset.
 *                  A negative slot skips the token (padding).  A slot at or beyond
 *                  num_blocks * 16 is skipped and sets PKV_DEVERR_SLOT.
 *                  Two tokens with the same slot in one call: undefined.
 *   device_error   optional device int32 error word (NULL: errors are not reported)
 *
 * bf16 cache: the bf16 bits are copied.  FP8 cache: each value is divided by
 * its (block, kv-head) scale in IEEE fp32 and encoded to E4M3 with round to
 * nearest even and saturation to +-448 (NaN stays NaN).
 * num_tokens = 0 is a no-op.
 *
 * Launch (programmatic dependent launch): the kernel lets the next kernel on
 * the stream launch at once, and reads slot_mapping, k_new and v_new (its
 * threads' first chunks) before waiting for the previous kernel on the
 * stream; the cache and the scales are touched only after that wait.  So a
 * kernel that lets its dependents start early must not write those three
 * inputs (none of this library's kernels writes them).
 */
PKV_API pkv_status pkv_paged_kv_append(const pkv_cache* cache, const void* k_new, const void* v_new,
                                       const int64_t* slot_mapping, int64_t num_tokens,
                                       int32_t* device_error, void* stream);

/*
 * paged_kv_append with rotary position embedding fused in, and optionally
 * FP8 scales chosen from the values (lfm25-inference file list:
 * kernels/rope.cu, kernels/kv_cache.cu; the pages fix neither the rotation's
 * form nor a scale rule -- these are the library's readings).
 *
 *   positions      device int32 [num_tokens]: each new token's position in its
 *                  sequence.  NULL: no rotation (a plain append, which can
 *                  still choose FP8 scales).
 *   rope_theta     the rotation base (e.g. 10000, 1e6); > 0 with positions.
 *                  Rotate-half form: for i < head_dim / 2 and angle
 *                  a = position * rope_theta^(-2i / head_dim),
 *                  y_i = x_i cos a - x_{i+D/2} sin a, y_{i+D/2} = x_{i+D/2} cos a + x_i sin a,
 *                  evaluated in fp64 and rounded once to bf16.  K is rotated
 *                  before it is stored; V is stored as given.
 *   q, num_q_heads optional device bf16 [num_tokens][num_q_heads][head_dim]: the
 *                  same tokens' query rows, rotated in place (NULL: none).
 *   fp8_scales_from_values   FP8 caches only (else PKV_ERR_INVALID_ARG): for every
 *                  (block, kv-head) whose offset-0 slot this call writes (a block
 *                  the call starts), the scale becomes the largest |value| among
 *                  this call's (rotated) values in that block and head, NaN
 *                  ignored, divided by 448 in IEEE fp32 (1.0 if that maximum is 0),
 *                  and the values are encoded with it; the cache's k_scales /
 *                  v_scales arrays are written.  A block continued by a later call
 *                  keeps its scale (values beyond it saturate).  0: the scales are
 *                  inputs, as for pkv_paged_kv_append.
 * Other arguments and the slot rules as for pkv_paged_kv_append.  Unlike it,
 * the last of its launches lets the next kernel on the stream launch only
 * once it has completed: it rotates q in place, and an attention that
 * follows reads q before its own dependency wait.  Supported
 * up to 32 kv-heads (else PKV_ERR_UNSUPPORTED).  Launches one CTA per token
 * (plus two short kernels when FP8 scales are chosen here).
 */
PKV_API pkv_status pkv_paged_kv_append_rope(const pkv_cache* cache, const void* k_new, const void* v_new,
                                            const int64_t* slot_mapping, int64_t num_tokens, const int32_t* positions,
                                            float rope_theta, void* q, int32_t num_q_heads,
                                            int32_t fp8_scales_from_values, int32_t* device_error, void* stream);

/*
 * Workspace for pkv_paged_attention, in bytes.  The workspace holds the
 * device error word, one merge ticket per (sequence, kv-head) and the split
 * partial results.  It must be zeroed once before first use
 * (pkv_workspace_init); a call that completes leaves it ready for the next
 * call.  A call that reports PKV_ERR_TIMEOUT (pkv_read_device_error) may have
 * left merge tickets set: zero the workspace again before reusing it.
 * num_ctas = 0 means the library's default grid for the current device.
 * The size does not depend on the cache's dtype: it covers the larger of
 * the bf16 and FP8 plans (an FP8 cache splits each kv-head's query heads
 * into groups of at most 16 or 8 rows, one ticket each).
 */
PKV_API size_t pkv_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t max_q_len, int32_t num_ctas);

/* Zero a workspace (cudaMemsetAsync on `stream`). */
PKV_API pkv_status pkv_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_attention -- decode / causal-verify attention over the paged cache
 * (lfm25-inference "Paged GQA/XQA Decode Attention ... Split-K reduction";
 * inferd "paged attention" reference and its equivalence with dense
 * attention; the verify window of inferd's speculative decoding).
 *
 * For sequence b with context length L_b (it counts every resident token,
 * including the q_lens[b] tokens just appended) and query window Q_b:
 * query i (0 <= i < Q_b) of query head h attends to positions
 * j = 0 .. L_b - Q_b + i of kv-head g = h / (Hq / Hkv):
 *     out = sum_j softmax_j(scale * q . k_j) v_j,
 * accumulated in fp32 and rounded to bf16 (nearest even).
 *
 *   q, out         device bf16 [sum q_lens][Hq][head_dim], packed by sequence; they must hold
 *                  sum(q_lens) rows (the kernels trust this size)
 *                  (sequence b's rows start at q_lens[0] + ... + q_lens[b-1]).
 *   block_tables   device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(L_b / 16) are never read.
 *   context_lens,  device int32 [num_seqs]; 0 <= q_lens[b] <= context_lens[b].
 *   q_lens
 *   max_q_len      host-known upper bound of q_lens (1..16), picks the kernel
 *                  (FP8 caches run on the tensor cores with the GQA group split
 *                  into virtual groups of at most 16 query rows at head_dim
 *                  128, of 8 at head_dim 64 up to 8 tokens; head_dim 64 with
 *                  9..16 tokens on the CUDA cores).
 *   scale          softmax scale (e.g. 1/sqrt(head_dim)).
 *   num_ctas       grid size (0 = default); it sets how the batch's KV is
 *                  split, so results of different grids differ by rounding only.
 *   workspace      device, >= pkv_attention_workspace_size(...) bytes, zeroed
 *                  once by pkv_workspace_init; not shared by concurrent calls.
 *
 * Supported: block_size 16, head_dim 64 or 128, Hq % Hkv == 0 (any GQA
 * group G = Hq / Hkv), max_q_len <= 16, and max_blocks_per_seq * Hkv * S <
 * 2^20 (contexts below 2^24 / (Hkv * S) tokens) where S is the smallest
 * divisor of G with (G / S) * max_q_len <= 32; otherwise PKV_ERR_UNSUPPORTED,
 * nothing launched.  When G * max_q_len > 32 (a wide group verifying a
 * window), a kv-head's G query heads are processed as S consecutive groups
 * of G / S heads; each reads the kv-head's pages (the repeat reads mostly
 * hit L2).
 * Results are deterministic and depend only
 * on logical positions (not on which physical blocks hold them).
 *
 * FP8 caches on the tensor cores take P.V in fp16 (V's e4m3 codes are exact
 * in fp16; P carries the page's v scale): a v scale above 255 (values beyond
 * ~114,000 before encoding) sets PKV_DEVERR_RANGE and the affected outputs
 * are unspecified.
 *
 * NaN in the cache: a NaN stored in K makes every element of the rows that
 * see it NaN, and a NaN in V the matching dimension of those rows, as in the
 * definition.  One departure: inside a causal window (q_len > 1), a NaN in
 * the V row of a window token also reaches the window's earlier queries that
 * do not see that token (their zero weights multiply it in the same
 * tensor-core product), unless none of the tokens of that part of the
 * sequence is visible to them.
 *
 * Launch (programmatic dependent launch).  When the previous kernel on
 * `stream` lets its dependents start early -- pkv_paged_kv_append does -- this
 * kernel's set-up, which reads context_lens, q_lens, block_tables and q,
 * overlaps that kernel; its K/V reads and its workspace accesses wait until
 * that kernel has completed.  So a kernel that lets its dependents start
 * early must not write those four inputs.  This kernel lets the next kernel
 * on the stream launch at once; a kernel launched for programmatic
 * dependence must wait for its prerequisites (griddepcontrol.wait) before
 * reading `out` or the workspace.  Kernels launched the ordinary way see
 * the usual stream order.
 */
PKV_API pkv_status pkv_paged_attention(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, const int32_t* q_lens,
                                       int32_t num_seqs, int32_t max_q_len, float scale, void* out,
                                       void* workspace, size_t workspace_bytes, int32_t num_ctas,
                                       void* stream);

/*
 * Shared-prefix cascade: pkv_paged_attention for a batch whose sequences come
 * in groups that share their leading blocks (the turns of a conversation
 * reusing one system prompt through the radix tree: lfm25-inference README,
 * "Radix Tree Prefix Caching"; inferd backlog, prefix sharing).  Same result
 * as pkv_paged_attention over the same tables (up to the order of fp32 sums),
 * but each shared block is read and attended once for the whole group: a
 * first pass attends each group's prefix with all the group's query rows at
 * once and keeps a per-row state (normalised fp32 output and log-sum-exp);
 * a second pass attends every sequence's remaining pages and merges each row
 * with its prefix state before writing out.
 *
 *   group_starts       device int32 [num_groups + 1]: group g is sequences
 *                      [group_starts[g], group_starts[g + 1]); the groups cover
 *                      0 .. num_seqs - 1 in order (a sequence sharing nothing
 *                      is a group of its own with prefix 0).
 *   group_prefix_lens  device int32 [num_groups]: tokens of the shared prefix,
 *                      a multiple of 16; every sequence of the group holds the
 *                      same blocks in the first prefix/16 entries of its table,
 *                      and prefix <= context_len - q_len for each of them (the
 *                      query window lies after the prefix).  Violations set
 *                      PKV_DEVERR_LENGTH.
 *   max_group_q_len    host bound on the sum of q_lens over a group (<= 32).
 *   workspace          >= pkv_cascade_workspace_size(...) bytes, zeroed once
 *                      (pkv_workspace_init); it holds both passes' merge state
 *                      and the prefix states.
 * Other arguments as for pkv_paged_attention (default grid).  bf16 caches
 * only (FP8: PKV_ERR_UNSUPPORTED).  Two launches on `stream`.
 */
PKV_API size_t pkv_cascade_workspace_size(int32_t num_seqs, int32_t num_groups, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t max_q_len,
                                          int32_t max_group_q_len);
PKV_API pkv_status pkv_paged_attention_cascade(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
                                               int32_t max_q_len, const int32_t* group_starts,
                                               const int32_t* group_prefix_lens, int32_t num_groups,
                                               int32_t max_group_q_len, float scale, void* out, void* workspace,
                                               size_t workspace_bytes, void* stream);

/*
 * Paged chunked prefill: pkv_paged_attention for long query windows -- a
 * prompt processed in one call, or a chunk of it appended to a context that
 * already holds the earlier chunks (lfm25-inference README, ragged/segmented
 * prefill FlashAttention on tensor cores; inferd backlog, chunked prefill).
 * The same definition as pkv_paged_attention: query i (0 <= i < Q_b) of head
 * h sees positions 0 .. L_b - Q_b + i of kv-head h / G through the block
 * table, fp32 accumulation, bf16 output (nearest even).  Precision: q.k in
 * bf16 x bf16 -> fp32; the weights times V in fp16 x fp16 -> fp32 (the
 * weights rounded to fp16, 11 significant bits; V converted exactly, bf16
 * values carrying 8), so an output is off by at most about 2^-11 * max|v|
 * over the keys it sees, plus rounding of fp32 sums.  A finite V value of
 * magnitude >= 65536 (beyond fp16) sets PKV_DEVERR_RANGE and the outputs of
 * its CTA are unspecified.
 *
 *   q, out, block_tables, context_lens, q_lens, scale
 *                  as for pkv_paged_attention (q and out packed by sequence,
 *                  sum(q_lens) rows).
 *   max_q_len      host upper bound of q_lens (>= 1, no upper limit beyond
 *                  the grid size: num_seqs * Hkv * ceil(max_q_len * G / 256)
 *                  < 2^31 CTAs).
 *   device_error   optional device int32 error word (PKV_DEVERR_* bits: bad
 *                  block id, bad lengths, a V value out of range, a wait
 *                  that ran out); NULL: not reported.  No workspace.
 *
 * Supported: bf16 caches (FP8: PKV_ERR_UNSUPPORTED), head_dim 64 or 128, GQA
 * groups G = Hq / Hkv that divide 128.  One launch on `stream` (programmatic
 * dependent launch, as pkv_paged_attention; it reads nothing before the
 * previous kernel completes): one CTA per 256 query rows (256 / G positions x
 * the G heads) of one (sequence, kv-head).  Deterministic.  A NaN stored in
 * the V row of a window token also reaches the queries of the same CTA that
 * do not see it (their zero weights multiply it in the same tensor-core
 * product), as for pkv_paged_attention's causal windows.  The wait limit and
 * hold flag of pkv_debug_set_wait_limit apply to it too.
 */
PKV_API pkv_status pkv_paged_prefill(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, const int32_t* q_lens, int32_t num_seqs,
                                     int32_t max_q_len, float scale, void* out, int32_t* device_error,
                                     void* stream);

/*
 * pkv_paged_attention_noalloc -- pkv_paged_attention for callers that cannot
 * allocate device memory (the pages have no counterpart of this entry point).
 *
 * Some callers own no device allocator: a plugin or foreign-language host
 * that can only pass the tensors it already holds, or a serving loop whose
 * device memory budget is fixed at start-up and must not grow on the decode
 * path.  They cannot supply the attention workspace, so this variant keeps it
 * in a static device array of PKV_NOALLOC_SCRATCH_BYTES inside the library
 * (every GPU that loads the library holds that array until the process
 * exits).  The caller still passes all inputs and outputs; the arguments mean
 * what they mean for pkv_paged_attention.  It allocates nothing: no
 * cudaMalloc, cudaFree or allocating library call.
 *
 *   device_error   optional device int32 error word that receives the
 *                  PKV_DEVERR_* bits.  NULL: device-side errors (a bad block
 *                  id, a bad length, a wait that ran out) are not reported
 *                  at all and the output is unspecified.
 *
 * The first call on a device looks up the array's device address with that
 * device current and caches it; make that first call before any stream
 * capture, and do not reset the device (cudaDeviceReset) between calls: the
 * cached address would then be stale.  Each call clears the array's error word and merge tickets on
 * `stream` before launching.  All calls share the one array and it keeps the
 * last call's contents, so calls whose kernels overlap on the GPU (other
 * streams or other host threads on the same device) race: serialise them.
 * A call whose workspace would exceed PKV_NOALLOC_SCRATCH_BYTES (too many
 * sequences or CTAs) returns PKV_ERR_WORKSPACE and launches nothing.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
PKV_API pkv_status pkv_paged_attention_noalloc(const pkv_cache* cache, const void* q, int32_t num_q_heads,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, const int32_t* q_lens,
                                               int32_t num_seqs, int32_t max_q_len, float scale, void* out,
                                               int32_t num_ctas, int32_t* device_error, void* stream);

/*
 * Read and clear a device error word: either the first 4 bytes of an
 * attention workspace or an append's device_error.  Synchronises `stream`.
 * *code receives the PKV_DEVERR_* bits; the return value is PKV_OK when no bit
 * was set, PKV_ERR_TIMEOUT if the timeout bit was set, else
 * PKV_ERR_DEVICE_INDEX.  For tests and debugging, not the hot path.
 */
PKV_API pkv_status pkv_read_device_error(void* error_word, int32_t* code, void* stream);

/*
 * For tests of the device-side timeout path only (the pages have no
 * counterpart).  Every bounded wait inside the tensor-core attention kernel
 * (mbarrier phases, merge tickets) gives up after limit_ns nanoseconds
 * (0 restores the default, 2 s), sets PKV_DEVERR_TIMEOUT and winds the CTA
 * down.  A non-NULL hold_flag (device int32) makes the kernel wait for
 * *hold_flag != 0 before its first K/V copy: a flag that nothing sets makes
 * that wait run out.  The settings are process-wide and apply to every
 * later pkv_paged_attention(_noalloc) and pkv_paged_prefill launch (not to
 * the CUDA-core kernel, which has no waits) until they are set again; not for
 * concurrent use.
 */
PKV_API void pkv_debug_set_wait_limit(uint64_t limit_ns, const int32_t* hold_flag);

/* Static description of a status code. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Library version string. */
PKV_API const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
