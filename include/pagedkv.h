/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode path.
 *
 * Three operations make up one decode step of PagedAttention:
 *
 *   pk_copy_blocks            copy-on-write clones of shared blocks
 *   pk_reshape_and_cache      append each new token's K/V to its slot
 *   pk_paged_attention_decode single-query attention through block tables
 *
 * plus helpers (workspace sizing, a block-table gather used to check the
 * table walk bit for bit, the device error word, status strings).
 *
 * Conventions common to every call
 * --------------------------------
 * Pointers.  Every tensor argument is a DEVICE pointer into memory the caller
 *   allocated and owns (cudaMalloc, a torch tensor, a pool).  The library keeps
 *   no pointer after a call returns and allocates no device memory.  All
 *   tensors are dense, row-major, with the shapes given below.
 * Types.  K/V/Q/new-token tensors are bf16 (IEEE binary32 truncated to its top
 *   16 bits, passed as raw 16-bit words).  block_tables and seq_lens are int32;
 *   slot_mapping and copy pairs are int64.
 * Cache layout.  k_cache and v_cache are [num_blocks, block_size, num_kv_heads,
 *   head_dim]: the tokens of a block side by side, the heads of a token side by
 *   side, the elements of a head side by side ("PagedAttention from First
 *   Principles", §7 "Inside the attention kernel"; "vLLM — PagedAttention",
 *   "Fused CUDA Kernels", conceptual kernel signature).
 * Streams.  Every call is enqueued on `stream` (NULL = the legacy default
 *   stream) and returns without waiting for the GPU, except
 *   pk_get_device_error, which synchronises `stream`.  No call reads device
 *   memory from the host, so the three step calls can be captured in a graph.
 * Alignment.  Device pointers must be 16-byte aligned (cudaMalloc and torch
 *   give 256); head_dim*2 bytes is then a multiple of 16 for every supported
 *   head_dim, so every row the kernels move is 16-byte aligned too.
 * Errors.  A call first checks its arguments on the host and returns a
 *   negative pk_status without launching anything if one is bad.  A failed
 *   launch returns PK_ERR_CUDA.  Bad DATA in device memory (a block id outside
 *   the pool, a slot past the pool, a length longer than the table) cannot be
 *   seen from the host: the kernels skip that access, never fault or trap, and
 *   OR a PK_DEVERR_* bit into a per-device error word that
 *   pk_get_device_error reads and clears.
 * Supported sizes.  head_dim in {64, 128}; block_size in {8, 16, 32};
 *   num_heads a multiple of num_kv_heads with G = num_heads / num_kv_heads in
 *   {1, 2, 4, 8, 16}; num_kv_heads >= 1.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *pk_stream_t;

enum pk_status {
    PK_OK = 0,
    PK_ERR_NULL = -1,          /* a required pointer is NULL */
    PK_ERR_SHAPE = -2,         /* sizes inconsistent or out of range */
    PK_ERR_UNSUPPORTED = -3,   /* head_dim, block_size or group size not supported */
    PK_ERR_WORKSPACE = -4,     /* workspace missing or smaller than required */
    PK_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
    PK_ERR_ALIGNMENT = -6,     /* a pointer is not 16-byte aligned */
    PK_ERR_NO_DEVICE = -7,     /* no usable CUDA device */
    /* Host block manager (pagedkv_block_manager.h) only: */
    PK_ERR_NO_BLOCKS = -8,     /* the pool has no free block left: the scheduler must preempt */
    PK_ERR_UNKNOWN_SEQUENCE = -9,  /* no sequence with that id */
    PK_ERR_SEQUENCE_EXISTS = -10,  /* a sequence with that id already exists */
    PK_ERR_HOST_MEMORY = -11   /* a host allocation failed */
};

enum pk_dtype { PK_BF16 = 0, PK_FP32 = 1 };

/* Bits of the device error word. */
#define PK_DEVERR_BLOCK_ID 0x1u /* a table entry below ceil(L/B) is outside [0, num_blocks) */
#define PK_DEVERR_SLOT     0x2u /* a slot_mapping entry is >= num_blocks * block_size */
#define PK_DEVERR_PAIR     0x4u /* a copy pair names a block outside [0, num_blocks) */
#define PK_DEVERR_SEQ_LEN  0x8u /* a seq_len is negative, exceeds max_seq_len or exceeds
                                   max_blocks_per_seq * block_size */
#define PK_DEVERR_TIMEOUT  0x10u /* a kernel gave up waiting on one of its own pipeline
                                    barriers (never expected; the results are invalid) */
#define PK_DEVERR_POINTER  0x20u /* a per-layer pointer of a *_layers call is NULL or not
                                    16-byte aligned (that layer was skipped) */

/* Human-readable name of a pk_status value; never NULL. */
const char *pk_status_string(int status);

/* ABI version: (major << 16) | minor. */
int pk_version(void);

/*
 * Bytes of workspace pk_paged_attention_decode (and
 * pk_paged_attention_multi_query) needs for these sizes; 0 when no sequence
 * can be split (max_seq_len <= 128) or the sizes are invalid.
 *
 * The workspace holds split-K partial results.  On the tensor-core kernel
 * (the default) a sequence longer than one 128-token tile may be cut across
 * CTAs of the persistent grid; each CTA has two 8,384-byte slots for the
 * parts it cuts (a header; per column the max and denominator; the
 * unnormalised output rows), so it needs 2 x 1,024 x 8,384 = 17,170,432
 * bytes whatever the sizes.  The CUDA-core kernel keeps (max, denominator,
 * output row) per (sequence, query head, 512-token partition) instead.  The
 * workspace is sized for the larger of the two, and for the worst case the
 * host can see (every sequence as long as max_seq_len), so the call never
 * reads seq_lens on the host.
 */
size_t pk_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int max_seq_len);

/*
 * Single-query decode attention over a paged KV cache.
 *
 * Defined by "vLLM — PagedAttention", Mathematical Formulation (Equation 4):
 * for sequence s of length L = seq_lens[s] and query head h,
 *
 *   out[s,h,:] = sum_j softmax_j(scale * q[s,h,:] . k_j) v_j,  j = 0 .. L-1,
 *
 * where token j lives in physical block block_tables[s, j / B] at offset j % B
 * ("PagedAttention from First Principles", §5: the kernel reads every block
 * through the table) and k_j, v_j are the rows of KV head h / G.  Table entries
 * at or beyond ceil(L/B) are never read, whatever they hold (§6: the sentinel
 * of unused table slots is never dereferenced).  L = 0 writes zeros.
 *
 *   out           [num_seqs, num_heads, head_dim], bf16 (out_dtype PK_BF16,
 *                 round-to-nearest-even of the fp32 result) or fp32 (PK_FP32)
 *   q             [num_seqs, num_heads, head_dim] bf16
 *   k_cache,
 *   v_cache       [num_blocks, block_size, num_kv_heads, head_dim] bf16
 *   block_tables  [num_seqs, max_blocks_per_seq] int32
 *   seq_lens      [num_seqs] int32, each in [0, max_seq_len]
 *   max_seq_len   host-side upper bound of seq_lens, used only to size the
 *                 split-K plan; must be <= max_blocks_per_seq * block_size.
 *                 A device length above it sets PK_DEVERR_SEQ_LEN and only its
 *                 first max_seq_len tokens are attended.
 *   scale         multiplies q.k before the softmax (1/sqrt(head_dim) for the
 *                 usual attention)
 *   workspace     device scratch of at least pk_decode_workspace_bytes(...)
 *                 bytes; its contents on entry do not matter.  Calls that share
 *                 one workspace must be ordered on the GPU (same stream).
 *
 * Long sequences are split into partitions processed in parallel and combined
 * by a log-sum-exp merge ("PagedAttention from First Principles", §17: the
 * partitioned kernel and its reduce step).  Results do not depend on the
 * physical placement of blocks and are deterministic run to run.
 */
int pk_paged_attention_decode(void *out, int out_dtype, const void *q,
                              const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *seq_lens, int max_seq_len,
                              int num_seqs, int num_heads, int num_kv_heads,
                              int head_dim, int num_blocks, int block_size,
                              float scale, void *workspace, size_t workspace_bytes,
                              pk_stream_t stream);

/*
 * The same decode attention as pk_paged_attention_decode, for callers that
 * cannot allocate device memory.  The pages have no counterpart of this call.
 *
 * Who needs it: code running inside a host program that owns all device
 * memory (a serving engine that reserved nearly all HBM for its KV pool at
 * start-up, so a later cudaMalloc fails), plugins that are handed tensors but
 * no allocator, and latency-critical loops that cannot afford cudaMalloc /
 * cudaFree, which may synchronise the device.  Such callers pass only the
 * inputs and the output; this call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *
 * Scratch: the partial results of sequences that span several CTAs go to a
 * fixed 2,682,880-byte array in the library's own device memory (a file-scope
 * __device__ array that every GPU loading the library holds until the
 * process exits): two 8,384-byte slots for each of at most 160 persistent
 * CTAs.  The call runs min(SM count, 160) CTAs; if that many slots did not
 * fit the array it would return PK_ERR_WORKSPACE.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 * Sharing: every call on a device uses the same array and leaves its contents
 * there.  Nothing in it has to start at zero (each CTA writes its own flag
 * before use), but calls that overlap on the GPU (several streams, or host
 * threads without ordering) race on it and give wrong results: order them.
 *
 * Arguments, layouts and errors are those of pk_paged_attention_decode
 * without the workspace.  The tensor-core kernel family is always used.
 */
int pk_paged_attention_decode_noalloc(void *out, int out_dtype, const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *seq_lens, int max_seq_len,
                                      int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int num_blocks, int block_size,
                                      float scale, pk_stream_t stream);

/*
 * Self-test of the kernels' bounded waits; the pages have no counterpart.
 *
 * Every wait of the tensor-core decode kernel on one of its own pipeline
 * barriers gives up after a time limit (1 s in normal calls), sets
 * PK_DEVERR_TIMEOUT, lets the CTA's own copies and MMAs land, frees its tensor
 * memory and returns, so a pipeline that stops never hangs the GPU.  This
 * call runs pk_paged_attention_decode on the tensor-core kernel with the
 * limit set to wait_limit_us and with CTA 0's copy producer stopping before
 * tile `stall_tile` of its range, so that CTA's waits on that tile's barriers
 * run out and take the give-up path.  Afterwards pk_get_device_error reports
 * PK_DEVERR_TIMEOUT and the output is invalid; the next call on the same
 * context and workspace is correct.
 *
 *   stall_tile     >= 1 (a tile of CTA 0's range; beyond its range nothing stalls)
 *   wait_limit_us  in [100, 1000000]
 *   everything else as for pk_paged_attention_decode.
 * Returns PK_ERR_SHAPE for a bad stall_tile or wait_limit_us.
 */
int pk_selftest_decode_wait_timeout(void *out, int out_dtype, const void *q,
                                    const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *seq_lens, int max_seq_len,
                                    int num_seqs, int num_heads, int num_kv_heads,
                                    int head_dim, int num_blocks, int block_size,
                                    float scale, void *workspace, size_t workspace_bytes,
                                    int stall_tile, unsigned int wait_limit_us,
                                    pk_stream_t stream);

/*
 * Self-test of the length check after the programmatic wait; the pages have
 * no counterpart.
 *
 * The tensor-core decode kernel is launched as a programmatic dependent of
 * the previous kernel in the stream.  With num_seqs <= 2048 it copies the
 * sequence lengths into shared memory and plans its range of the work before
 * that kernel has completed, then reads the lengths again after the wait and
 * plans again if any differs (the previous kernel may have written them).
 * This call runs pk_paged_attention_decode on the tensor-core kernel with the
 * first read taken from `stale_seq_lens` instead of `seq_lens`, so that the
 * second plan, from `seq_lens`, is the one used whenever the two differ.  The
 * result must equal that of pk_paged_attention_decode with the same inputs.
 *
 *   stale_seq_lens  [num_seqs] int32 DEVICE array, any values (lengths outside
 *                   [0, max_seq_len] included: only seq_lens is checked and
 *                   reported); unused when num_seqs > 2048
 *   everything else as for pk_paged_attention_decode.
 * Returns PK_ERR_NULL if stale_seq_lens is NULL.
 */
int pk_selftest_decode_stale_lengths(void *out, int out_dtype, const void *q,
                                     const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *seq_lens, int max_seq_len,
                                     int num_seqs, int num_heads, int num_kv_heads,
                                     int head_dim, int num_blocks, int block_size,
                                     float scale, const int32_t *stale_seq_lens,
                                     void *workspace, size_t workspace_bytes,
                                     pk_stream_t stream);

/*
 * Attention of SEVERAL new tokens per sequence over the paged cache, causal
 * among them: chunked prefill of a prompt ("PagedAttention from First
 * Principles", §12) and speculative-decoding verification, where the
 * verifier checks a few appended tokens in one pass (§14).  Sequence s owns
 * query rows cu_q_lens[s] .. cu_q_lens[s+1]-1: its q_s newest tokens, whose
 * K/V are already in the cache, so with L = seq_lens[s] query r sits at
 * position L - q_s + r and attends positions 0 .. L - q_s + r.  With one
 * query per sequence this is pk_paged_attention_decode.
 *
 *   out        [total_q, num_heads, head_dim], bf16 or fp32
 *   q          [total_q, num_heads, head_dim] bf16
 *   cu_q_lens  [num_seqs + 1] int32 DEVICE array, cu_q_lens[0] = 0,
 *              non-decreasing, cu_q_lens[num_seqs] = total_q
 *   max_q_len  host-side bound of cu_q_lens[s+1] - cu_q_lens[s]
 *   everything else as for pk_paged_attention_decode (same workspace size).
 *
 * Tensor cores.  Narrow blocks (G * q <= 16 with q = max_q_len rounded up
 * to a power of two: e.g. G = 8, 2 tokens; speculative verification) use
 * one MMA column per (query token, query head) in the decode kernel; wider
 * blocks (prompt chunks) use a kernel whose CTAs each take two query tiles
 * of 128 rows (128 / G tokens x G heads each) of one sequence and KV head
 * over the sequence's key tiles; the workspace is then not used.  A sequence with more queries than tokens sets PK_DEVERR_SEQ_LEN
 * (its rows are then unspecified).
 */
int pk_paged_attention_multi_query(void *out, int out_dtype, const void *q, int total_q,
                                   const int32_t *cu_q_lens, int max_q_len, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables,
                                   int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                   int num_blocks, int block_size, float scale, void *workspace,
                                   size_t workspace_bytes, pk_stream_t stream);

/* Kernel family of pk_paged_attention_decode, process-wide. */
enum pk_decode_path {
    PK_PATH_AUTO = 0,                    /* tensor cores (per-head tiles) for every
                                            group size, CUDA cores for a batch too
                                            small to give each SM one 128-token tile */
    PK_PATH_CUDA_CORE = 1,               /* fp32 FMA on CUDA cores, one CTA per partition */
    PK_PATH_TENSOR_CORE = 2              /* tcgen05 MMA, persistent CTAs, tiles of
                                            128 tokens x 1 KV head */
};

/*
 * Select the decode kernel family for later calls (all devices); returns the
 * previous setting, or PK_ERR_UNSUPPORTED for an unknown value.  Both
 * families compute the same attention; they differ in how the score and
 * output contractions are executed.  The setting is process-wide: do not
 * change it while another host thread may be issuing decode calls (each call
 * reads it once, so a call racing with the change may use either family).
 */
int pk_set_decode_path(int path);

/*
 * Append new tokens' K/V to their cache slots ("vLLM — PagedAttention",
 * Fused CUDA Kernels (1), fused reshape and block write; "PagedAttention from
 * First Principles", §2: the cache is append-only).
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim] bf16
 *   slot_mapping  [num_tokens] int64: token t goes to block slot / block_size,
 *                 offset slot % block_size, all heads.  A negative slot is a
 *                 padding token and writes nothing.  A slot at or beyond
 *                 num_blocks * block_size sets PK_DEVERR_SLOT and writes nothing.
 *                 Two tokens with the same slot race (the caller never does this).
 *
 * num_tokens == 0 is a no-op.  Bit-exact: the cache rows become the input bits.
 */
int pk_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int num_blocks,
                         int block_size, pk_stream_t stream);

/*
 * Copy whole blocks, K and V, one launch for all pairs ("vLLM —
 * PagedAttention", Copy-on-Write Logic and Fused CUDA Kernels (3): batched
 * block copies for copy-on-write).
 *
 *   src_dst_pairs [num_pairs, 2] int64 device array of (src, dst) block ids.
 *                 No dst may appear twice and no dst may be the src of another
 *                 pair (a copy-on-write step never produces that); otherwise
 *                 the result is unspecified.  An id outside [0, num_blocks)
 *                 sets PK_DEVERR_PAIR and that pair is skipped.
 *
 * num_pairs == 0 is a no-op.  Bit-exact.
 */
int pk_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                   int num_pairs, int num_kv_heads, int head_dim, int num_blocks,
                   int block_size, pk_stream_t stream);

/*
 * Multi-layer variants: the same append / block copy on every layer of a
 * model in ONE launch.  A model keeps two cache tensors per layer
 * ("PagedAttention from First Principles", §5 "The PagedAttention
 * algorithm"), a logical block costs one physical block in every layer (§6
 * "The block table, byte by byte": 80 layers of Llama-3-70B), so the slots
 * of a step and the copy-on-write pairs are the same for all layers.
 *
 *   k_layers, v_layers   DEVICE array of num_layers DEVICE pointers, layer l's
 *                        new K (V) rows [num_tokens, num_kv_heads, head_dim] bf16
 *   k_cache_layers, v_cache_layers
 *                        DEVICE array of num_layers DEVICE pointers, layer l's
 *                        cache [num_blocks, block_size, num_kv_heads, head_dim]
 *   slot_mapping, src_dst_pairs, sizes: as in the one-layer calls, shared by
 *                        every layer.
 *
 * The pointer arrays are caller-owned device memory (8-byte aligned); the
 * host cannot read them, so a NULL or unaligned per-layer pointer is found on
 * the GPU: that layer is skipped and PK_DEVERR_POINTER is set.  Bad slots and
 * pairs are handled per layer as in the one-layer calls.  num_layers in
 * [1, 65535] (block copies: [1, 32767]); num_layers == 0 or no tokens / pairs
 * is a no-op.  Bit-exact.
 */
int pk_reshape_and_cache_layers(const void *const *k_layers, const void *const *v_layers,
                                void *const *k_cache_layers, void *const *v_cache_layers,
                                const int64_t *slot_mapping, int num_tokens, int num_layers,
                                int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                pk_stream_t stream);
int pk_copy_blocks_layers(void *const *k_cache_layers, void *const *v_cache_layers,
                          const int64_t *src_dst_pairs, int num_pairs, int num_layers,
                          int num_kv_heads, int head_dim, int num_blocks, int block_size,
                          pk_stream_t stream);

/*
 * Move blocks between two pools in one launch: for every pair (src, dst),
 * dst_k[dst] = src_k[src] and dst_v[dst] = src_v[src], whole blocks.  One pool
 * is typically the device pool and the other a pool in page-locked host memory
 * that the GPU can address (cudaHostAlloc, or a torch pin_memory tensor under
 * unified addressing): swapping a preempted request out copies its blocks to
 * host RAM and swapping it in copies them back ("PagedAttention from First
 * Principles", §15 "KV-cache offloading and disaggregated serving";
 * "PagedAttention Explained", preemption by swapping or recomputation; "How
 * vLLM and PagedAttention Actually Work", §10 Q3).  The pages note that many
 * small transfers use the CPU-GPU link poorly; here one kernel moves every
 * block of the batch, each warp streaming whole 512-byte runs of block rows
 * over the link, many CTAs keeping many reads in flight.
 *
 *   src_k, src_v  [src_num_blocks, block_size, num_kv_heads, head_dim] bf16
 *   dst_k, dst_v  [dst_num_blocks, block_size, num_kv_heads, head_dim] bf16
 *   pairs         [num_pairs, 2] int64 DEVICE array of (src block, dst block)
 *
 * A block id outside its pool sets PK_DEVERR_PAIR and that pair is skipped.
 * No dst may repeat and the two pools must not overlap; otherwise the result
 * is unspecified.  num_pairs == 0 is a no-op.  Bit-exact.
 */
int pk_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                   const int64_t *pairs, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int src_num_blocks, int dst_num_blocks, pk_stream_t stream);

/*
 * Gather every sequence's K/V through its block table into contiguous rows:
 * out_k[cu_seq_lens[s] + j] = k_cache[block_tables[s, j / B], j % B] for
 * j < seq_lens[s] (same for V).  This is the table walk of the attention kernel
 * on its own ("PagedAttention from First Principles", §5), exported so that it
 * can be checked bit for bit.
 *
 *   out_k, out_v  [total_tokens, num_kv_heads, head_dim] bf16
 *   cu_seq_lens   [num_seqs] int64 device array: first output row of each sequence
 *   max_seq_len   host-side bound of seq_lens (as for the attention call)
 *
 * A table entry outside the pool sets PK_DEVERR_BLOCK_ID and its rows are left
 * unwritten.
 */
int pk_gather_kv(void *out_k, void *out_v, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, int max_blocks_per_seq,
                 const int32_t *seq_lens, const int64_t *cu_seq_lens, int max_seq_len,
                 int num_seqs, int num_kv_heads, int head_dim, int num_blocks,
                 int block_size, pk_stream_t stream);

/*
 * Read and clear the error word of the current device.  Synchronises `stream`
 * first, so it reports every kernel enqueued before it on that stream.
 * *code_out receives the OR of the PK_DEVERR_* bits set since the last clear.
 */
int pk_get_device_error(unsigned int *code_out, pk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
