/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged-KV attention library
 * (libpagedattn.so).
 *
 * Three operations make up the hot path of LLM serving attention over a
 * paged KV cache:
 *
 *   kv_write_paged               eager writeback of new K/V rows into their
 *                                pages ("Inside Ion", section "IonAttention
 *                                in One Paragraph": KV pages are written back
 *                                eagerly as they are produced).
 *   kv_write_paged_rope          the same with the Q/K RMS norm and rotary
 *                                embedding fused in.
 *   kv_write_paged_fp8,          writeback into, and decode over, an FP8
 *   attn_decode_paged_fp8        (e4m3) KV cache with per-KV-head scales.
 *   attn_decode_paged            one query row per sequence against its whole
 *                                paged history, split along the KV sequence
 *                                and merged with the log-sum-exp identity
 *                                ("The Stack Below the Stack, Part 2",
 *                                section 2.2 Flash-Decoding, steps 1-3).
 *   attn_decode_paged_append     writeback of each sequence's newest row and
 *                                the decode, in one kernel (and
 *                                attn_decode_multiquery_paged_append for
 *                                a block of new rows).
 *   attn_decode_multiquery_paged the same for a short block (2-8) of query
 *                                rows per sequence, causal inside the block
 *                                (speculative-decode verification).
 *   attn_prefill_varlen_causal   causal attention of variable-length query
 *                                blocks against their paged K/V, tiled with
 *                                the online softmax ("The Stack Below the
 *                                Stack, Part 2", section 2.1; "8. Kernels and
 *                                Attention Backends", section "Attention is an
 *                                I/O problem").  Decode rows may be mixed in as
 *                                entries with one query row.
 *
 * Common conventions
 * ------------------
 * Pointers named *_pool, q, out, k_new, v_new, block_table, seq_lens,
 * cu_seqlens_*, lse, workspace and status are pointers the GPU accesses:
 * device memory, or page-locked host memory where "Memory" below allows it;
 * the caller owns every buffer (nothing is allocated by the library).  All calls are
 * asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream),
 * perform no host synchronisation and allocate nothing, so they may be
 * captured in a CUDA graph.
 *
 * Back-to-back launches: the writeback kernels let the kernel after them
 * start at once (programmatic dependent launch), and the decode kernels are
 * launched so that they may start early.  A decode call's kernel then reads
 * seq_lens, cu_seqlens_q and block_table while the kernel before it still
 * runs, and reads q and the pools only after that kernel has finished.  So
 * seq_lens, cu_seqlens_q and block_table must be final before a kernel that
 * lets its dependents start early (only the writebacks of this library do,
 * unless the caller's own kernels use programmatic dependent launch).
 *
 * Memory: the K/V pools, block_table, the workspace and every argument of
 * attn_prefill_varlen_causal must be device memory.  The small per-step
 * arguments of the decode and writeback calls (q, out, lse, k_new, v_new,
 * seq_lens, cu_seqlens_q, cu_seqlens_new; also k_new and v_new of the
 * *_append calls) may instead be page-locked host
 * memory (cudaHostAlloc / cudaHostRegister): the kernels read and write it
 * in place over the CPU-GPU link (NVLink-C2C on GB300), which for a decode
 * step's few hundred kilobytes costs less than staging copies on the copy
 * engine.
 *
 * Element types: K/V pools, q, out, k_new, v_new are bf16 (bfloat16: sign,
 * 8 exponent and 7 mantissa bits, 2 bytes); lse is float32; integer arrays
 * are int32.
 *
 * Layouts (row-major, contiguous):
 *   k_pool, v_pool : [num_pages][num_kv_heads][page_size][head_dim]
 *   block_table    : [batch][max_pages_per_seq]; entry p of row b is the
 *                    physical page holding tokens p*page_size ..
 *                    (p+1)*page_size-1 of sequence b.  Entries past the
 *                    sequence's last page are never read.
 *   seq_lens       : [batch]; total keys of each sequence, including the rows
 *                    being attended from / written in this call.
 *   q, out         : [rows][num_q_heads][head_dim]
 *   lse            : [rows][num_q_heads], natural-log log-sum-exp of the
 *                    scaled scores of each row (-inf for a row with no key).
 * Query head h attends KV head h / (num_q_heads / num_kv_heads).
 *
 * Supported shapes: head_dim 64 or 128; page_size a power of two from 16 to
 * 256; num_q_heads a multiple of num_kv_heads; num_q_heads / num_kv_heads
 * up to 128.  The pools, q, out, k_new and v_new must start on a 16-byte
 * boundary (PA_ERR_SHAPE otherwise: the kernels move 16-byte vectors, and
 * the prefill moves whole 16-row page blocks with bulk tensor copies); a
 * workspace must start on a 256-byte boundary (PA_ERR_WORKSPACE otherwise).
 *
 * Errors: a negative return value is a pa_status detected on the host
 * before anything is launched (nothing was enqueued).  Errors found on the
 * device (a block_table entry outside [0, num_pages), an inconsistent
 * length, or -- in the prefill kernel of attn_prefill_varlen_causal, the only
 * kernel that waits on mbarriers -- a wait on a TMA copy or a tensor-core
 * operation that ran past its time limit) are written, first one wins, to the
 * optional device word `status` (int32, caller-zeroed); the kernels skip
 * the offending access instead of faulting, and the affected outputs are
 * unspecified.  Read `status` after synchronising the stream.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = -1,       /* a required pointer is NULL                          */
    PA_ERR_SHAPE = -2,      /* unsupported or inconsistent sizes                   */
    PA_ERR_WORKSPACE = -3,  /* workspace missing or smaller than required          */
    PA_ERR_CUDA = -4,       /* a CUDA runtime/driver call or the launch failed     */
    PA_ERR_TIMEOUT = -5,    /* device: a prefill-kernel wait ran past its limit    */
    PA_ERR_BAD_PAGE = -6,   /* device: block_table entry outside [0, num_pages)    */
    PA_ERR_BAD_LEN = -7,    /* device: seq_len / row count inconsistent            */
    PA_ERR_ARCH = -8,       /* the current device is not an sm_103 GPU             */
    PA_ERR_SCRATCH_LIMIT = -9 /* needs more scratch than attn_decode_paged_noalloc holds */
} pa_status;

/* Version of this ABI (bumped on any signature change). */
int pa_abi_version(void);

/* Static, NUL-terminated description of a pa_status value. */
const char* pa_status_string(int status);

/*
 * Workspace bytes attn_decode_paged needs for these sizes on the current
 * device.  The workspace holds each sequence's first work unit (batch + 1
 * int32) and the split partials (normalised partial outputs and their
 * log-sum-exps).  A call writes every part before reading it, so the
 * workspace needs no initialisation and may serve calls of any size that
 * fits.  Two calls that may run concurrently need separate workspaces.
 */
size_t pa_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim);

/*
 * Decode: out[b][h][:] = softmax(scale * q[b][h] . K_b^T) V_b over the
 * seq_lens[b] keys of sequence b, with K_b/V_b gathered through
 * block_table[b] from KV head h / (Hq/Hkv).
 *   out        bf16 [batch][num_q_heads][head_dim]           (written)
 *   lse        float [batch][num_q_heads] or NULL             (written)
 *   q          bf16 [batch][num_q_heads][head_dim]
 *   max_seq_len  host upper bound of seq_lens (sizes the launch only)
 * A sequence with seq_lens[b] == 0 gets out = 0 and lse = -inf.
 */
int attn_decode_paged(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                      int num_pages, const int32_t* block_table, int max_pages_per_seq,
                      const int32_t* seq_lens, int batch, int max_seq_len, int page_size,
                      int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                      void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Decode with the writeback of the newest rows in the same kernel ("Inside
 * Ion", section "IonAttention in One Paragraph": KV pages are written back
 * eagerly as they are produced): the result of kv_write_paged (one new row
 * per sequence, at position seq_lens[b] - 1) followed by attn_decode_paged,
 * in one call.  The decode stages each sequence's newest K/V row from
 * k_new / v_new instead of its pool slot, and one warp per (sequence, KV
 * head) writes the row into that slot (bit-exact copy).
 *   k_pool, v_pool  written at the new rows' slots (block_table must map
 *                   position seq_lens[b] - 1 to an allocated page)
 *   k_new, v_new    bf16 [batch][num_kv_heads][head_dim]
 * Other arguments, workspace and results as attn_decode_paged.  bf16 pools
 * only (the FP8 cache keeps kv_write_paged_fp8 + attn_decode_paged_fp8).
 */
int attn_decode_paged_append(void* out, float* lse, const void* q, void* k_pool, void* v_pool,
                             const void* k_new, const void* v_new, int num_pages, const int32_t* block_table,
                             int max_pages_per_seq, const int32_t* seq_lens, int batch, int max_seq_len,
                             int page_size, int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                             void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Workspace bytes attn_decode_multiquery_paged needs when no entry has more
 * than max_q_len (1..8) query rows; like the decode workspace it needs no
 * initialisation.  Returns 0 for unsupported sizes.
 */
size_t pa_decode_multiquery_workspace_bytes(int batch, int max_q_len, int num_q_heads, int num_kv_heads,
                                            int head_dim);

/*
 * Multi-query decode: a short block of q_len = cu_seqlens_q[b+1] -
 * cu_seqlens_q[b] query rows per sequence (1 <= q_len <= 8), e.g. the tokens
 * a draft model proposed, verified in one pass ("Inside Ion", section "What
 * Is Next": speculative decoding).  Row i of sequence b sits at position
 * seq_lens[b] - q_len + i and attends keys 0 .. that position (causal inside
 * the block, every earlier cached token visible), exactly as in
 * attn_prefill_varlen_causal; the work is split along the KV sequence and
 * merged as in attn_decode_paged, so the KV of a sequence is read from HBM
 * once for all its query rows and heads.
 *   out        bf16 [total_q][num_q_heads][head_dim]          (written)
 *   lse        float [total_q][num_q_heads] or NULL            (written)
 *   q          bf16 [total_q][num_q_heads][head_dim]
 *   cu_seqlens_q  int32 [batch+1], non-decreasing, cu_seqlens_q[batch] <= total_q
 *   max_q_len  host upper bound of q_len, 1..8 (PA_ERR_SHAPE otherwise); it
 *              sizes the workspace (pa_decode_multiquery_workspace_bytes)
 * An entry with q_len = 0 is skipped.  On the device, q_len > max_q_len,
 * cu_seqlens_q outside [0, total_q] or 0 < seq_lens[b] < q_len (for q_len > 1)
 * report PA_ERR_BAD_LEN; rows with no visible key get out = 0 and lse = -inf.
 */
int attn_decode_multiquery_paged(void* out, float* lse, const void* q, const void* k_pool,
                                 const void* v_pool, int num_pages, const int32_t* block_table,
                                 int max_pages_per_seq, const int32_t* cu_seqlens_q,
                                 const int32_t* seq_lens, int batch, int total_q, int max_q_len,
                                 int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                                 int head_dim, float softmax_scale, void* workspace,
                                 size_t workspace_bytes, int32_t* status, void* stream);

/*
 * attn_decode_multiquery_paged with the query tokens' own K/V rows written
 * back by the same kernel, as attn_decode_paged_append does for one row:
 * the result of kv_write_paged (cu_seqlens_new = cu_seqlens_q) followed by
 * attn_decode_multiquery_paged, in one call.
 *   k_new, v_new  bf16 [total_q][num_kv_heads][head_dim]: row cu_seqlens_q[b] + i
 *                 is token seq_lens[b] - q_len + i of sequence b
 * bf16 pools only.
 */
int attn_decode_multiquery_paged_append(void* out, float* lse, const void* q, void* k_pool, void* v_pool,
                                        const void* k_new, const void* v_new, int num_pages,
                                        const int32_t* block_table, int max_pages_per_seq,
                                        const int32_t* cu_seqlens_q, const int32_t* seq_lens, int batch,
                                        int total_q, int max_q_len, int max_seq_len, int page_size,
                                        int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                                        void* workspace, size_t workspace_bytes, int32_t* status,
                                        void* stream);

/*
 * Workspace bytes attn_prefill_varlen_causal needs (no initialisation, as
 * the decode workspace; it also holds the split partials of the entries
 * with at most 8 query rows, which the call serves on the split-K decode
 * path).
 */
size_t pa_prefill_workspace_bytes(int batch, int total_q, int num_q_heads, int num_kv_heads, int head_dim);

/*
 * Varlen causal prefill over paged K/V.  Rows cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1]-1 of q belong to sequence b; with
 * q_len = cu_seqlens_q[b+1] - cu_seqlens_q[b], row i sits at absolute
 * position seq_lens[b] - q_len + i and attends keys 0 .. that position
 * (bottom-right causal alignment: earlier cached tokens are all visible).
 * The K/V of the query rows themselves must already be in the pool (call
 * kv_write_paged first, on the same stream).  Entries with q_len <= 8 are
 * served exactly as attn_decode_multiquery_paged serves them (q_len = 1 is
 * ordinary decode), so one call serves a mixed prefill + decode step.
 *   out        bf16 [total_q][num_q_heads][head_dim]          (written)
 *   lse        float [total_q][num_q_heads] or NULL            (written)
 *   q          bf16 [total_q][num_q_heads][head_dim]
 *   cu_seqlens_q  int32 [batch+1], cu_seqlens_q[0] = 0, non-decreasing
 *   max_q_len, max_seq_len  host upper bounds (size the launch only)
 *   softmax_scale  must be finite and > 0 (PA_ERR_SHAPE otherwise)
 */
int attn_prefill_varlen_causal(void* out, float* lse, const void* q, const void* k_pool,
                               const void* v_pool, int num_pages, const int32_t* block_table,
                               int max_pages_per_seq, const int32_t* cu_seqlens_q,
                               const int32_t* seq_lens, int batch, int total_q, int max_q_len,
                               int max_seq_len, int page_size, int num_q_heads, int num_kv_heads,
                               int head_dim, float softmax_scale, void* workspace,
                               size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Eager KV writeback.  Rows cu_seqlens_new[b] .. cu_seqlens_new[b+1]-1 of
 * k_new/v_new are the newest n_b = cu_seqlens_new[b+1] - cu_seqlens_new[b]
 * tokens of sequence b, whose length AFTER the write is seq_lens[b]; row i
 * goes to position pos = seq_lens[b] - n_b + i, i.e. page
 * block_table[b][pos / page_size], slot pos % page_size, for every KV head.
 * A bit-exact copy; no other byte of the pools is touched.
 *   k_new, v_new  bf16 [total_new][num_kv_heads][head_dim]
 */
int kv_write_paged(void* k_pool, void* v_pool, int num_pages, const void* k_new, const void* v_new,
                   const int32_t* cu_seqlens_new, const int32_t* seq_lens,
                   const int32_t* block_table, int max_pages_per_seq, int batch, int total_new,
                   int page_size, int num_kv_heads, int head_dim, int32_t* status, void* stream);

/*
 * Fused Q/K normalisation, rotary embedding and KV writeback ("The Stack
 * Below the Stack, Part 2", section 2.1, kernel fusion: fused Q-norm,
 * KV-RoPE and K-insert).  Same placement as kv_write_paged: new row i of
 * sequence b goes to position pos = seq_lens[b] - n_b + i.  Before it is
 * written, each K head row is
 *     x <- x / sqrt(mean(x^2) + norm_eps) * k_norm_weight   (if k_norm_weight)
 *     (x[j], x[j + D/2]) <- rotated by pos * rope_base^(-2j/D)   (j < D/2)
 * in fp32 and rounded once to bf16 (round to nearest even); V rows are copied
 * bit for bit.  When q is not NULL its rows (bf16 [total_new][num_q_heads]
 * [head_dim], the queries of the same new tokens) get the same treatment in
 * place, with q_norm_weight.  The rotation pairs dimension j with j + D/2
 * (the "rotate-half" layout of Llama- and Qwen-family models).
 *   rope_base      > 1 and finite (PA_ERR_SHAPE otherwise)
 *   q_norm_weight, k_norm_weight  bf16 [head_dim] or NULL (no normalisation)
 *   norm_eps       >= 0 and finite
 * Angles are reduced exactly (64-bit fixed-point turns), so positions up to
 * 2^31 keep full fp32 accuracy.  A row whose block-table entry lies outside
 * the pool records PA_ERR_BAD_PAGE and writes no K/V; its query rows are
 * still normalised and rotated (they do not depend on the page).
 */
int kv_write_paged_rope(void* k_pool, void* v_pool, int num_pages, const void* k_new, const void* v_new,
                        void* q, int num_q_heads, const int32_t* cu_seqlens_new, const int32_t* seq_lens,
                        const int32_t* block_table, int max_pages_per_seq, int batch, int total_new,
                        int page_size, int num_kv_heads, int head_dim, float rope_base,
                        const void* q_norm_weight, const void* k_norm_weight, float norm_eps,
                        int32_t* status, void* stream);

/*
 * FP8 KV cache ("The Stack Below the Stack, Part 2", closing recipe: FP8 KV).
 * K and V elements are stored as e4m3 codes (1 byte; the OCP / CUDA E4M3
 * format: bias 7, 3 mantissa bits, largest finite value 448, no
 * infinities), which halves the bytes decode reads.  Element x of KV head g
 * is stored as the code nearest to x / scale[g] (fp32 quotient, round to
 * nearest even, saturating at +-448) and reads back as code * scale[g].
 * Layouts (uint8):
 *   k_pool  [num_pages][num_kv_heads][page_size][head_dim]   (as the bf16 pool)
 *   v_pool  [num_pages][num_kv_heads][head_dim][page_size]   (transposed inside
 *           each page block, so the keys of one value column are contiguous)
 *   k_scale, v_scale  float [num_kv_heads], device; must be > 0
 * One scale per KV head (not per page): pages are filled one token at a
 * time by the eager writeback, so a per-page scale would be fixed by the
 * page's first token.
 *
 * kv_write_paged_fp8: the quantising writeback, placement as kv_write_paged
 * (k_new, v_new bf16 [total_new][num_kv_heads][head_dim]).
 */
int kv_write_paged_fp8(void* k_pool, void* v_pool, int num_pages, const void* k_new, const void* v_new,
                       const float* k_scale, const float* v_scale, const int32_t* cu_seqlens_new,
                       const int32_t* seq_lens, const int32_t* block_table, int max_pages_per_seq, int batch,
                       int total_new, int page_size, int num_kv_heads, int head_dim, int32_t* status,
                       void* stream);

/*
 * attn_decode_paged over an FP8 cache: same arguments, results and workspace
 * (pa_decode_workspace_bytes) as attn_decode_paged, with the pools and
 * scales above.  Scores use q . (code * k_scale[g]) and the output
 * sum p * code * v_scale[g] / sum p, computed on fp16 tensor cores (every
 * e4m3 code is exact in fp16; q is rounded to fp16, so |q| must stay below
 * 65504) with fp32 accumulation.
 */
int attn_decode_paged_fp8(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                          const float* k_scale, const float* v_scale, int num_pages, const int32_t* block_table,
                          int max_pages_per_seq, const int32_t* seq_lens, int batch, int max_seq_len,
                          int page_size, int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                          void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Allocation-free variant of attn_decode_paged.  This entry point has no
 * counterpart in the paper; it exists for callers that cannot allocate
 * device memory -- code running inside an allocator or memory-pool
 * callback, plugins whose host framework owns every device allocation, or
 * paths that must never enter the driver's allocator -- and therefore
 * cannot provide the decode workspace.
 *
 * Same arguments and results as attn_decode_paged, minus the workspace: the
 * split-K scratch lives in a fixed 8 MiB device array inside the library,
 * which every GPU that loads the library holds until the process exits.
 * Problems whose workspace (pa_decode_workspace_bytes) exceeds 8 MiB are
 * rejected with PA_ERR_SCRATCH_LIMIT before anything is enqueued; roughly,
 * (batch * num_kv_heads * ceil(group / 64) + three times the SM count) * rows
 * must stay below about 16,000 at head_dim 128 (about 32,000 at head_dim 64),
 * where group = num_q_heads / num_kv_heads and rows = 16 for group <= 16,
 * 32 for group <= 32 and 64 above.
 *
 * No call allocates: no cudaMalloc, cudaFree or allocating library call.
 * The first call on each device (and the first after the device's context
 * was destroyed and created again, e.g. by cudaDeviceReset) looks up the
 * array's device address (cudaGetSymbolAddress) with that device current.
 * Because CUDA loads modules lazily, that first lookup (or the first launch of
 * any kernel of this library) is also where the driver loads the library's
 * device code and reserves the 8 MiB array, i.e. where the driver itself
 * allocates.  Make that first call -- or a warm-up call -- where driver
 * allocation is allowed and before any stream capture; later calls touch no
 * allocator.  All calls on a device share the one array and
 * it keeps the last call's contents:
 * calls whose execution may overlap on the GPU (different streams, or
 * concurrent graph branches) race on it and give wrong results.
 */
int attn_decode_paged_noalloc(void* out, float* lse, const void* q, const void* k_pool, const void* v_pool,
                              int num_pages, const int32_t* block_table, int max_pages_per_seq,
                              const int32_t* seq_lens, int batch, int max_seq_len, int page_size,
                              int num_q_heads, int num_kv_heads, int head_dim, float softmax_scale,
                              int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
