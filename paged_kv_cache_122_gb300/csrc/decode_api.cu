// Host entry point of paged decode attention: argument checks, the split-K
// plan and the launches.
#include "decode.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>

namespace {

bool group_supported(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

// Partition size of the CUDA-core path.
constexpr int kCudaCorePartTokens = 512;

// Smallest group for which the automatic choice uses the tensor cores: all of
// them.  From G = 4 on, the scores of a 128-token tile are a [128 x D] x
// [D x G] contraction and fp32 FMA issue, not HBM, would bound the CUDA-core
// kernel; at G = 1 and 2 the tensor-core kernel still streams the pages
// faster (measured on a Llama-3-70B length mix with 8 KV heads, D = 128:
// 6.2 against 4.3 TB/s at G = 1, 6.2 against 4.1 at G = 2; equal at D = 64).
constexpr int kTensorCoreMinGroup = 1;

std::atomic<int> g_path{PK_PATH_AUTO};

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

extern "C" size_t pk_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                            int head_dim, int max_seq_len) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0) return 0;
    if (num_heads % num_kv_heads) return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    const int np_cap = ceil_div(max_seq_len, pk::kMinPartTokens);
    // Enough for either kernel family (the family can be switched at run time).
    const size_t cc = np_cap > 1 ? pk::workspace_floats(num_seqs, num_heads, head_dim, np_cap) * sizeof(float) : 0;
    const size_t tc = max_seq_len > 128 ? pk::tc_workspace_bytes() : 0;
    return std::max(cc, tc);
}

extern "C" int pk_set_decode_path(int path) {
    if (path != PK_PATH_AUTO && path != PK_PATH_CUDA_CORE && path != PK_PATH_TENSOR_CORE)
        return PK_ERR_UNSUPPORTED;
    return g_path.exchange(path);
}

namespace {

// The decode call; `stall_tile` and `wait_limit_ns` serve the self-test of
// the bounded waits (0 = off / the default limit) and `lens_ahead` the
// self-test of the length check after the programmatic wait (NULL = off);
// either forces the tensor-core kernel.
int decode_impl(void *out, int out_dtype, const void *q, const void *k_cache, const void *v_cache,
                const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                int num_seqs, int num_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
                float scale, void *workspace, size_t workspace_bytes, pk_stream_t stream, int stall_tile,
                uint64_t wait_limit_ns, const int32_t *lens_ahead) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0 ||
        max_blocks_per_seq < 0 || max_seq_len < 0 || block_size <= 0)
        return PK_ERR_SHAPE;
    if (num_heads % num_kv_heads) return PK_ERR_SHAPE;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return PK_ERR_SHAPE;
    if (out_dtype != PK_BF16 && out_dtype != PK_FP32) return PK_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PK_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PK_ERR_UNSUPPORTED;
    if (!group_supported(num_heads / num_kv_heads)) return PK_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PK_ERR_SHAPE;
    if (num_seqs > 65535 || num_kv_heads * 2 > 65535) return PK_ERR_SHAPE;
    if (num_seqs == 0) return PK_OK;
    if (!out || !q || !seq_lens || (max_seq_len > 0 && (!k_cache || !v_cache || !block_tables)))
        return PK_ERR_NULL;
    if (!pk::aligned16(out) || !pk::aligned16(q) || !pk::aligned16(k_cache) || !pk::aligned16(v_cache))
        return PK_ERR_ALIGNMENT;

    pk::DecodeParams p{};
    p.out = out;
    p.out_fp32 = out_dtype == PK_FP32;
    p.q = static_cast<const uint16_t *>(q);
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_seq_len = max_seq_len;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.scale_log2 = scale * pk::kLog2e;
    p.stall_tile = stall_tile;
    p.wait_limit_ns = wait_limit_ns;
    p.lens_ahead = lens_ahead;
    const int path = (stall_tile > 0 || lens_ahead) ? PK_PATH_TENSOR_CORE : g_path.load();
    const int G = num_heads / num_kv_heads;
    // A batch whose 128-token tiles could not give every SM even one (at most
    // num_seqs * Hkv * ceil(max_seq_len / 128) of them) is bound by launch
    // latency, where the CUDA-core kernel, without the persistent kernel's
    // set-up, answers sooner (4 short sequences: ~15 against ~18 us).
    const int64_t max_tiles = static_cast<int64_t>(num_seqs) * num_kv_heads * ceil_div(max_seq_len, 128);
    const bool tiny = max_tiles < pk::sm_count();
    const bool tensor_core = max_seq_len > 0 &&
        (path == PK_PATH_TENSOR_CORE || (path == PK_PATH_AUTO && G >= kTensorCoreMinGroup && !tiny));
    if (tensor_core) {
        // A sequence longer than one tile may span several CTAs: its parts need slots.
        const size_t need = pk::tc_workspace_bytes();
        if (max_seq_len > 128) {
            if (!workspace || workspace_bytes < need) return PK_ERR_WORKSPACE;
            if (!pk::aligned16(workspace)) return PK_ERR_ALIGNMENT;
            p.tc_slots = workspace;
        }
    } else {
        p.part_tokens = kCudaCorePartTokens;
        p.np_cap = std::max(1, ceil_div(max_seq_len, p.part_tokens));
        if (p.np_cap > 1) {
            const size_t need = pk::workspace_floats(num_seqs, num_heads, head_dim, p.np_cap) * sizeof(float);
            if (!workspace || workspace_bytes < need) return PK_ERR_WORKSPACE;
            if (!pk::aligned16(workspace)) return PK_ERR_ALIGNMENT;
            float *ws = static_cast<float *>(workspace);
            const size_t rows = static_cast<size_t>(num_seqs) * num_heads * p.np_cap;
            p.ws_o = ws;
            p.ws_m = ws + rows * head_dim;
            p.ws_l = p.ws_m + rows;
        }
    }

    p.err = pk::error_word_ptr();
    if (!p.err) return PK_ERR_NO_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (tensor_core) return pk::launch_decode_tensor_core(p, st) == cudaSuccess ? PK_OK : PK_ERR_CUDA;
    if (pk::launch_decode_cuda_core(p, st) != cudaSuccess) return PK_ERR_CUDA;
    if (pk::launch_decode_merge(p, st) != cudaSuccess) return PK_ERR_CUDA;
    return PK_OK;
}

}  // namespace

extern "C" int pk_paged_attention_decode(void *out, int out_dtype, const void *q,
                                         const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *seq_lens, int max_seq_len, int num_seqs,
                                         int num_heads, int num_kv_heads, int head_dim,
                                         int num_blocks, int block_size, float scale,
                                         void *workspace, size_t workspace_bytes,
                                         pk_stream_t stream) {
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                       workspace, workspace_bytes, stream, 0, 0, nullptr);
}

extern "C" int pk_selftest_decode_wait_timeout(void *out, int out_dtype, const void *q,
                                               const void *k_cache, const void *v_cache,
                                               const int32_t *block_tables, int max_blocks_per_seq,
                                               const int32_t *seq_lens, int max_seq_len, int num_seqs,
                                               int num_heads, int num_kv_heads, int head_dim,
                                               int num_blocks, int block_size, float scale,
                                               void *workspace, size_t workspace_bytes, int stall_tile,
                                               unsigned int wait_limit_us, pk_stream_t stream) {
    if (stall_tile < 1 || wait_limit_us < 100 || wait_limit_us > 1000000) return PK_ERR_SHAPE;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                       workspace, workspace_bytes, stream, stall_tile, static_cast<uint64_t>(wait_limit_us) * 1000u,
                       nullptr);
}

extern "C" int pk_selftest_decode_stale_lengths(void *out, int out_dtype, const void *q,
                                                const void *k_cache, const void *v_cache,
                                                const int32_t *block_tables, int max_blocks_per_seq,
                                                const int32_t *seq_lens, int max_seq_len, int num_seqs,
                                                int num_heads, int num_kv_heads, int head_dim,
                                                int num_blocks, int block_size, float scale,
                                                const int32_t *stale_seq_lens, void *workspace,
                                                size_t workspace_bytes, pk_stream_t stream) {
    if (!stale_seq_lens) return PK_ERR_NULL;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       max_seq_len, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                       workspace, workspace_bytes, stream, 0, 0, stale_seq_lens);
}

extern "C" int pk_paged_attention_multi_query(void *out, int out_dtype, const void *q, int total_q,
                                              const int32_t *cu_q_lens, int max_q_len, const void *k_cache,
                                              const void *v_cache, const int32_t *block_tables,
                                              int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                                              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                              int num_blocks, int block_size, float scale, void *workspace,
                                              size_t workspace_bytes, pk_stream_t stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0 || max_blocks_per_seq < 0 ||
        max_seq_len < 0 || block_size <= 0 || total_q < 0 || max_q_len < 0)
        return PK_ERR_SHAPE;
    if (num_heads % num_kv_heads) return PK_ERR_SHAPE;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return PK_ERR_SHAPE;
    if (out_dtype != PK_BF16 && out_dtype != PK_FP32) return PK_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PK_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PK_ERR_UNSUPPORTED;
    const int G = num_heads / num_kv_heads;
    if (!group_supported(G)) return PK_ERR_UNSUPPORTED;
    // Narrow query blocks (G x q <= 16, q padded to a power of two) run on the
    // decode kernel's 16 query columns; wider ones on the prefill kernel,
    // 128 query rows per CTA.
    int ql = 1;
    while (ql < max_q_len) ql <<= 1;
    const bool narrow = G * ql <= 16;
    if (!std::isfinite(scale)) return PK_ERR_SHAPE;
    if (num_seqs > 65535) return PK_ERR_SHAPE;
    if (num_seqs == 0 || total_q == 0) return PK_OK;
    if (!out || !q || !cu_q_lens || !seq_lens || (max_seq_len > 0 && (!k_cache || !v_cache || !block_tables)))
        return PK_ERR_NULL;
    if (!pk::aligned16(out) || !pk::aligned16(q) || !pk::aligned16(k_cache) || !pk::aligned16(v_cache))
        return PK_ERR_ALIGNMENT;

    pk::DecodeParams p{};
    p.out = out;
    p.out_fp32 = out_dtype == PK_FP32;
    p.q = static_cast<const uint16_t *>(q);
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_seq_len = max_seq_len;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.scale_log2 = scale * pk::kLog2e;
    p.cu_q_lens = cu_q_lens;
    p.q_len = ql;
    p.total_q = total_q;
    if (narrow && max_seq_len > 128) {
        if (!workspace || workspace_bytes < pk::tc_workspace_bytes()) return PK_ERR_WORKSPACE;
        if (!pk::aligned16(workspace)) return PK_ERR_ALIGNMENT;
        p.tc_slots = workspace;
    }
    p.err = pk::error_word_ptr();
    if (!p.err) return PK_ERR_NO_DEVICE;
    if (max_seq_len == 0) return PK_OK;   // every sequence is empty: no query can exist
    if (!narrow)
        return pk::launch_prefill_tensor_core(p, max_q_len, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? PK_OK : PK_ERR_CUDA;
    return pk::launch_multi_query_tensor_core(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PK_OK : PK_ERR_CUDA;
}
