// Parameters and launchers of the paged decode-attention kernels.
#pragma once

#include "common.cuh"

namespace pk {

// Everything a decode kernel needs, by value.  Scores are kept in the base-2
// domain: s2 = (q . k) * scale * log2(e), weights are 2^(s2 - m).
struct DecodeParams {
    void *out;
    int out_fp32;
    const uint16_t *q;          // [N, H, D]
    const uint16_t *k_cache;    // [P, B, Hkv, D]
    const uint16_t *v_cache;
    const int32_t *block_tables;  // [N, MB]
    const int32_t *seq_lens;      // [N]
    int max_blocks_per_seq;
    int max_seq_len;
    int num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size;
    float scale_log2;
    // Split-K partials, indexed by u = (s * H + h) * np_cap + partition:
    // ws_m[u] running max (base 2), ws_l[u] denominator, ws_o[u * D + d]
    // unnormalised output.
    float *ws_m;
    float *ws_l;
    float *ws_o;
    int part_tokens;   // tokens per partition (multiple of 128)
    int np_cap;        // partitions reserved per (sequence, head)
    // Tensor-core path: two cut-segment slots per CTA.
    void *tc_slots;
    // Bounded waits: give up after this many ns (0 = the default, 1 s).
    uint64_t wait_limit_ns;
    // Self-test of the bounded waits: when > 0, CTA 0's producer issues no
    // copy from this tile of its range on, so its consumers' waits run out.
    int stall_tile;
    // The lengths the tensor-core kernel plans from before the programmatic
    // wait (NULL = seq_lens).  After the wait it reads seq_lens and redoes the
    // plan if they differ; the self-test of that check passes other values.
    const int32_t *lens_ahead;
    // Multi-query attention (tensor-core path): q is [total_q, H, D] and
    // sequence s owns query rows cu_q_lens[s] .. cu_q_lens[s+1]-1, its newest
    // tokens, causal among themselves; q_len is the padded number of query
    // tokens per sequence the kernel packs into the MMA columns.  NULL / 1
    // for single-token decode.
    const int32_t *cu_q_lens;
    int q_len;
    int total_q;       // rows of q (multi-query)
    unsigned int *err;
};

// Smallest partition any decode path uses; fixes the workspace bound.
constexpr int kMinPartTokens = 256;

inline size_t workspace_floats(int num_seqs, int num_heads, int head_dim, int np_cap) {
    return static_cast<size_t>(num_seqs) * num_heads * np_cap * (head_dim + 2);
}

// Tensor-core path (tcgen05): main kernel + merge of cut segments.
cudaError_t launch_decode_tensor_core(const DecodeParams &p, cudaStream_t stream);
// Multi-query attention on the tensor-core path (p.cu_q_lens set, p.q_len a
// power of two with G * q_len <= 16).
cudaError_t launch_multi_query_tensor_core(const DecodeParams &p, cudaStream_t stream);
// Multi-query attention for wide query blocks (chunked prefill): 128 query
// rows (128 / G tokens x G heads) per CTA over the paged keys; no workspace.
cudaError_t launch_prefill_tensor_core(const DecodeParams &p, int max_q_len, cudaStream_t stream);
// Largest persistent grid of the tensor-core path.
constexpr int kTcMaxCtas = 1024;
// Workspace bytes the tensor-core path needs (independent of the sizes).
size_t tc_workspace_bytes();
// Bytes of one cut-segment slot of the tensor-core path (two per CTA).
size_t tc_slot_bytes();
// Tensor-core path with an explicit grid of `ctas` persistent CTAs; the
// slots at p.tc_slots must hold 2 * ctas slots.
cudaError_t launch_decode_tensor_core_grid(const DecodeParams &p, cudaStream_t stream, int ctas);

// CUDA-core path (any supported G).  Returns a cudaError_t.
cudaError_t launch_decode_cuda_core(const DecodeParams &p, cudaStream_t stream);
// Log-sum-exp merge of the partitions of split sequences.
cudaError_t launch_decode_merge(const DecodeParams &p, cudaStream_t stream);

}  // namespace pk
