// Cache writes, block copies and the table-walk gather.
//
// All three are byte movers: each thread moves 16-byte vectors, consecutive
// threads touch consecutive vectors, so every warp reads and writes whole
// 512-byte runs of a cache row.  The roofline is HBM bandwidth (bytes read +
// bytes written).
#include "common.cuh"

namespace {

constexpr int kThreads = 256;

// Launch as a programmatic dependent of the previous kernel in the stream
// (the kernels below wait for it before touching memory), so the launch
// overlaps that kernel's end.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// One 16-byte vector per thread over the flattened (token, vector) space.
// A token's K (or V) row, all heads, is contiguous both in the input
// [T, Hkv, D] and in the cache [P, B, Hkv, D] (flat slot = block * B + offset),
// so each token is a single contiguous row copy.
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int num_tokens,
                         int row_vecs, int64_t num_slots, unsigned int *err) {
    // A decode grid launched as this grid's programmatic dependent may start
    // its set-up now; it reads the cache only after this grid has completed.
    // This grid is itself a programmatic dependent of the previous kernel in
    // the stream: it reads and writes nothing before that kernel completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t t = i / row_vecs;
    const int e = static_cast<int>(i - t * row_vecs);
    if (t >= num_tokens) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;                         // padding token
    if (slot >= num_slots) {                      // outside the pool: skip, report
        if (e == 0) pk::set_error(err, PK_DEVERR_SLOT);
        return;
    }
    const uint4 kv = pk::ldg_stream(k + t * row_vecs + e);
    const uint4 vv = pk::ldg_stream(v + t * row_vecs + e);
    k_cache[slot * row_vecs + e] = kv;
    v_cache[slot * row_vecs + e] = vv;
}

// grid = (pairs, 2 [K, V], chunks of one block).  Plain loads: the pool is
// written by this kernel, so the read-only path is not used.
constexpr int kCopyVecsPerCta = kThreads * 4;

__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   const int64_t *__restrict__ pairs, int64_t block_vecs, int num_blocks,
                   unsigned int *err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // as in reshape_and_cache_kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int pair = blockIdx.x;
    const int64_t src = pairs[2 * pair];
    const int64_t dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) pk::set_error(err, PK_DEVERR_PAIR);
        return;
    }
    uint4 *c = blockIdx.y ? v_cache : k_cache;
    const uint4 *s = c + src * block_vecs;
    uint4 *d = c + dst * block_vecs;
    const int64_t lo = static_cast<int64_t>(blockIdx.z) * kCopyVecsPerCta;
    const int64_t hi = min(lo + kCopyVecsPerCta, block_vecs);
    uint4 buf[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t e = lo + u * kThreads + threadIdx.x;
        if (e < hi) buf[u] = s[e];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t e = lo + u * kThreads + threadIdx.x;
        if (e < hi) d[e] = buf[u];
    }
}

// Multi-layer variants: blockIdx.y selects the layer (copy: layer * 2 + K/V);
// each layer's pointers come from caller-owned device arrays and are checked
// here, where they can be read.
__device__ __forceinline__ bool usable(const void *ptr) {
    return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
}

__global__ void __launch_bounds__(kThreads)
reshape_and_cache_layers_kernel(const uint4 *const *k_layers, const uint4 *const *v_layers,
                                uint4 *const *k_cache_layers, uint4 *const *v_cache_layers,
                                const int64_t *__restrict__ slot_mapping, int num_tokens,
                                int row_vecs, int64_t num_slots, unsigned int *err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // as in reshape_and_cache_kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int layer = blockIdx.y;
    const uint4 *k = k_layers[layer];
    const uint4 *v = v_layers[layer];
    uint4 *kc = k_cache_layers[layer];
    uint4 *vc = v_cache_layers[layer];
    if (!usable(k) || !usable(v) || !usable(kc) || !usable(vc)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) pk::set_error(err, PK_DEVERR_POINTER);
        return;
    }
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t t = i / row_vecs;
    const int e = static_cast<int>(i - t * row_vecs);
    if (t >= num_tokens) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (e == 0) pk::set_error(err, PK_DEVERR_SLOT);
        return;
    }
    const uint4 kv = pk::ldg_stream(k + t * row_vecs + e);
    const uint4 vv = pk::ldg_stream(v + t * row_vecs + e);
    kc[slot * row_vecs + e] = kv;
    vc[slot * row_vecs + e] = vv;
}

__global__ void __launch_bounds__(kThreads)
copy_blocks_layers_kernel(uint4 *const *k_cache_layers, uint4 *const *v_cache_layers,
                          const int64_t *__restrict__ pairs, int64_t block_vecs, int num_blocks,
                          unsigned int *err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // as in reshape_and_cache_kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int pair = blockIdx.x;
    const int layer = blockIdx.y >> 1;
    uint4 *c = (blockIdx.y & 1) ? v_cache_layers[layer] : k_cache_layers[layer];
    if (!usable(c)) {
        if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0) pk::set_error(err, PK_DEVERR_POINTER);
        return;
    }
    const int64_t src = pairs[2 * pair];
    const int64_t dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) pk::set_error(err, PK_DEVERR_PAIR);
        return;
    }
    const uint4 *s = c + src * block_vecs;
    uint4 *d = c + dst * block_vecs;
    const int64_t lo = static_cast<int64_t>(blockIdx.z) * kCopyVecsPerCta;
    const int64_t hi = min(lo + kCopyVecsPerCta, block_vecs);
    uint4 buf[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t e = lo + u * kThreads + threadIdx.x;
        if (e < hi) buf[u] = s[e];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t e = lo + u * kThreads + threadIdx.x;
        if (e < hi) d[e] = buf[u];
    }
}

// grid = (pairs, 2 [K, V], chunks of one block): the block copy of
// copy_blocks_kernel between two pools (one of them usually host memory the
// GPU addresses over the CPU link).  Each thread keeps four 16-byte reads in
// flight before it writes.
__global__ void __launch_bounds__(kThreads)
swap_blocks_kernel(uint4 *__restrict__ dst_k, uint4 *__restrict__ dst_v, const uint4 *__restrict__ src_k,
                   const uint4 *__restrict__ src_v, const int64_t *__restrict__ pairs, int64_t block_vecs,
                   int src_blocks, int dst_blocks, unsigned int *err) {
    const int pair = blockIdx.x;
    const int64_t src = pairs[2 * pair];
    const int64_t dst = pairs[2 * pair + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) pk::set_error(err, PK_DEVERR_PAIR);
        return;
    }
    const uint4 *s = (blockIdx.y ? src_v : src_k) + src * block_vecs;
    uint4 *d = (blockIdx.y ? dst_v : dst_k) + dst * block_vecs;
    const int64_t lo = static_cast<int64_t>(blockIdx.z) * kCopyVecsPerCta;
    const int64_t hi = min(lo + kCopyVecsPerCta, block_vecs);
    uint4 buf[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t e = lo + u * kThreads + threadIdx.x;
        if (e < hi) buf[u] = s[e];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t e = lo + u * kThreads + threadIdx.x;
        if (e < hi) d[e] = buf[u];
    }
}

// grid = (num_seqs, token chunks of kGatherTokens).  Each CTA walks the table
// of one sequence for its chunk of positions.
constexpr int kGatherTokens = 32;

__global__ void __launch_bounds__(kThreads)
gather_kv_kernel(uint4 *__restrict__ out_k, uint4 *__restrict__ out_v,
                 const uint4 *__restrict__ k_cache, const uint4 *__restrict__ v_cache,
                 const int32_t *__restrict__ block_tables, int max_blocks_per_seq,
                 const int32_t *__restrict__ seq_lens, const int64_t *__restrict__ cu_seq_lens,
                 int max_seq_len, int row_vecs, int num_blocks, int block_size,
                 unsigned int *err) {
    const int s = blockIdx.x;
    int L = seq_lens[s];
    const int cap = min(max_seq_len, max_blocks_per_seq * block_size);
    if (L < 0 || L > cap) {
        if (blockIdx.y == 0 && threadIdx.x == 0) pk::set_error(err, PK_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : cap;
    }
    const int j0 = blockIdx.y * kGatherTokens;
    if (j0 >= L) return;
    const int nj = min(kGatherTokens, L - j0);
    const int64_t base = cu_seq_lens[s];
    const int32_t *row = block_tables + static_cast<int64_t>(s) * max_blocks_per_seq;
    for (int i = threadIdx.x; i < nj * row_vecs; i += kThreads) {
        const int jj = i / row_vecs;
        const int e = i - jj * row_vecs;
        const int j = j0 + jj;
        const int blk = row[j / block_size];
        if (blk < 0 || blk >= num_blocks) {
            if (e == 0) pk::set_error(err, PK_DEVERR_BLOCK_ID);
            continue;
        }
        const int64_t src = (static_cast<int64_t>(blk) * block_size + j % block_size) * row_vecs + e;
        const int64_t dst = (base + j) * row_vecs + e;
        out_k[dst] = pk::ldg_stream(k_cache + src);
        out_v[dst] = pk::ldg_stream(v_cache + src);
    }
}

bool supported_geometry(int num_kv_heads, int head_dim, int block_size) {
    return num_kv_heads >= 1 && (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || block_size == 16 || block_size == 32);
}

}  // namespace

extern "C" int pk_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                                    const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                    int head_dim, int num_blocks, int block_size,
                                    pk_stream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0)
        return PK_ERR_SHAPE;
    if (!supported_geometry(num_kv_heads, head_dim, block_size)) return PK_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PK_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PK_ERR_NULL;
    if (!pk::aligned16(k) || !pk::aligned16(v) || !pk::aligned16(k_cache) || !pk::aligned16(v_cache))
        return PK_ERR_ALIGNMENT;
    const int row_vecs = num_kv_heads * head_dim / 8;
    const int64_t total = static_cast<int64_t>(num_tokens) * row_vecs;
    const int64_t grid = (total + kThreads - 1) / kThreads;
    if (grid > 0x7fffffff) return PK_ERR_SHAPE;
    unsigned int *err = pk::error_word_ptr();
    if (!err) return PK_ERR_NO_DEVICE;
    const cudaError_t e = launch_dependent(
        reshape_and_cache_kernel, dim3(static_cast<unsigned>(grid)), reinterpret_cast<cudaStream_t>(stream),
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), slot_mapping, num_tokens, row_vecs,
        static_cast<int64_t>(num_blocks) * block_size, err);
    return e == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

extern "C" int pk_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                              int num_pairs, int num_kv_heads, int head_dim, int num_blocks,
                              int block_size, pk_stream_t stream) {
    if (num_pairs < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0)
        return PK_ERR_SHAPE;
    if (!supported_geometry(num_kv_heads, head_dim, block_size)) return PK_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PK_OK;
    if (!k_cache || !v_cache || !src_dst_pairs) return PK_ERR_NULL;
    if (!pk::aligned16(k_cache) || !pk::aligned16(v_cache)) return PK_ERR_ALIGNMENT;
    const int64_t block_vecs = static_cast<int64_t>(block_size) * num_kv_heads * head_dim / 8;
    const int64_t chunks = (block_vecs + kCopyVecsPerCta - 1) / kCopyVecsPerCta;
    if (chunks > 65535) return PK_ERR_SHAPE;
    unsigned int *err = pk::error_word_ptr();
    if (!err) return PK_ERR_NO_DEVICE;
    dim3 grid(static_cast<unsigned>(num_pairs), 2, static_cast<unsigned>(chunks));
    const cudaError_t e =
        launch_dependent(copy_blocks_kernel, grid, reinterpret_cast<cudaStream_t>(stream),
                         static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), src_dst_pairs, block_vecs,
                         num_blocks, err);
    return e == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

namespace {
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
}  // namespace

extern "C" int pk_reshape_and_cache_layers(const void *const *k_layers, const void *const *v_layers,
                                           void *const *k_cache_layers, void *const *v_cache_layers,
                                           const int64_t *slot_mapping, int num_tokens, int num_layers,
                                           int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                           pk_stream_t stream) {
    if (num_tokens < 0 || num_layers < 0 || num_layers > 65535 || num_blocks < 0 || num_kv_heads <= 0 ||
        block_size <= 0)
        return PK_ERR_SHAPE;
    if (!supported_geometry(num_kv_heads, head_dim, block_size)) return PK_ERR_UNSUPPORTED;
    if (num_tokens == 0 || num_layers == 0) return PK_OK;
    if (!k_layers || !v_layers || !k_cache_layers || !v_cache_layers || !slot_mapping) return PK_ERR_NULL;
    if (!aligned8(k_layers) || !aligned8(v_layers) || !aligned8(k_cache_layers) || !aligned8(v_cache_layers))
        return PK_ERR_ALIGNMENT;
    const int row_vecs = num_kv_heads * head_dim / 8;
    const int64_t total = static_cast<int64_t>(num_tokens) * row_vecs;
    const int64_t grid = (total + kThreads - 1) / kThreads;
    if (grid > 0x7fffffff) return PK_ERR_SHAPE;
    unsigned int *err = pk::error_word_ptr();
    if (!err) return PK_ERR_NO_DEVICE;
    const cudaError_t e = launch_dependent(
        reshape_and_cache_layers_kernel, dim3(static_cast<unsigned>(grid), static_cast<unsigned>(num_layers)),
        reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *const *>(k_layers),
        reinterpret_cast<const uint4 *const *>(v_layers), reinterpret_cast<uint4 *const *>(k_cache_layers),
        reinterpret_cast<uint4 *const *>(v_cache_layers), slot_mapping, num_tokens, row_vecs,
        static_cast<int64_t>(num_blocks) * block_size, err);
    return e == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

extern "C" int pk_copy_blocks_layers(void *const *k_cache_layers, void *const *v_cache_layers,
                                     const int64_t *src_dst_pairs, int num_pairs, int num_layers,
                                     int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                     pk_stream_t stream) {
    if (num_pairs < 0 || num_layers < 0 || num_layers > 32767 || num_blocks < 0 || num_kv_heads <= 0 ||
        block_size <= 0)
        return PK_ERR_SHAPE;
    if (!supported_geometry(num_kv_heads, head_dim, block_size)) return PK_ERR_UNSUPPORTED;
    if (num_pairs == 0 || num_layers == 0) return PK_OK;
    if (!k_cache_layers || !v_cache_layers || !src_dst_pairs) return PK_ERR_NULL;
    if (!aligned8(k_cache_layers) || !aligned8(v_cache_layers)) return PK_ERR_ALIGNMENT;
    const int64_t block_vecs = static_cast<int64_t>(block_size) * num_kv_heads * head_dim / 8;
    const int64_t chunks = (block_vecs + kCopyVecsPerCta - 1) / kCopyVecsPerCta;
    if (chunks > 65535) return PK_ERR_SHAPE;
    unsigned int *err = pk::error_word_ptr();
    if (!err) return PK_ERR_NO_DEVICE;
    dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(2 * num_layers), static_cast<unsigned>(chunks));
    const cudaError_t e = launch_dependent(copy_blocks_layers_kernel, grid, reinterpret_cast<cudaStream_t>(stream),
                                           reinterpret_cast<uint4 *const *>(k_cache_layers),
                                           reinterpret_cast<uint4 *const *>(v_cache_layers), src_dst_pairs,
                                           block_vecs, num_blocks, err);
    return e == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

extern "C" int pk_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                              const int64_t *pairs, int num_pairs, int num_kv_heads, int head_dim,
                              int block_size, int src_num_blocks, int dst_num_blocks, pk_stream_t stream) {
    if (num_pairs < 0 || src_num_blocks < 0 || dst_num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0)
        return PK_ERR_SHAPE;
    if (!supported_geometry(num_kv_heads, head_dim, block_size)) return PK_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PK_OK;
    if (!dst_k || !dst_v || !src_k || !src_v || !pairs) return PK_ERR_NULL;
    if (!pk::aligned16(dst_k) || !pk::aligned16(dst_v) || !pk::aligned16(src_k) || !pk::aligned16(src_v))
        return PK_ERR_ALIGNMENT;
    const int64_t block_vecs = static_cast<int64_t>(block_size) * num_kv_heads * head_dim / 8;
    const int64_t chunks = (block_vecs + kCopyVecsPerCta - 1) / kCopyVecsPerCta;
    if (chunks > 65535) return PK_ERR_SHAPE;
    unsigned int *err = pk::error_word_ptr();
    if (!err) return PK_ERR_NO_DEVICE;
    dim3 grid(static_cast<unsigned>(num_pairs), 2, static_cast<unsigned>(chunks));
    swap_blocks_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(dst_k), static_cast<uint4 *>(dst_v), static_cast<const uint4 *>(src_k),
        static_cast<const uint4 *>(src_v), pairs, block_vecs, src_num_blocks, dst_num_blocks, err);
    return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

extern "C" int pk_gather_kv(void *out_k, void *out_v, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, const int64_t *cu_seq_lens, int max_seq_len,
                            int num_seqs, int num_kv_heads, int head_dim, int num_blocks,
                            int block_size, pk_stream_t stream) {
    if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_seq_len < 0)
        return PK_ERR_SHAPE;
    if (!supported_geometry(num_kv_heads, head_dim, block_size)) return PK_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return PK_ERR_SHAPE;
    if (num_seqs == 0 || max_seq_len == 0) return PK_OK;
    if (!out_k || !out_v || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_seq_lens)
        return PK_ERR_NULL;
    if (!pk::aligned16(out_k) || !pk::aligned16(out_v) || !pk::aligned16(k_cache) ||
        !pk::aligned16(v_cache))
        return PK_ERR_ALIGNMENT;
    const int chunks = (max_seq_len + kGatherTokens - 1) / kGatherTokens;
    if (chunks > 65535 || num_seqs > 0x7fffffff) return PK_ERR_SHAPE;
    unsigned int *err = pk::error_word_ptr();
    if (!err) return PK_ERR_NO_DEVICE;
    dim3 grid(static_cast<unsigned>(num_seqs), static_cast<unsigned>(chunks));
    gather_kv_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(out_k), static_cast<uint4 *>(out_v),
        static_cast<const uint4 *>(k_cache), static_cast<const uint4 *>(v_cache), block_tables,
        max_blocks_per_seq, seq_lens, cu_seq_lens, max_seq_len, num_kv_heads * head_dim / 8,
        num_blocks, block_size, err);
    return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}
