// Decode attention for callers that cannot allocate device memory.
//
// pk_paged_attention_decode asks the caller for a workspace.  Some callers
// cannot provide one: a host program may own all device memory (a serving
// engine that reserved nearly all HBM for its KV pool at start-up, so a later
// cudaMalloc fails), a plugin may be handed tensors but no allocator, and a
// latency-critical loop may not afford cudaMalloc / cudaFree, which can
// synchronise the device.  This entry point runs the same tensor-core kernel
// with its scratch in a fixed array of this library's own device memory and
// allocates nothing.
#include "decode.cuh"

#include <algorithm>
#include <cmath>
#include <mutex>

namespace {

// The scratch holds two cut-segment slots per persistent CTA, for up to
// kNoAllocMaxCtas CTAs (GB300 has 152 SMs).  Every GPU that loads the
// library holds this array until the process exits.
constexpr int kNoAllocMaxCtas = 160;
constexpr size_t kNoAllocSlotBytes = 8384;
constexpr size_t kScratchBytes = 2 * kNoAllocMaxCtas * kNoAllocSlotBytes;   // 2,682,880 bytes

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current.
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

bool group_ok(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

}  // namespace

extern "C" int pk_paged_attention_decode_noalloc(void *out, int out_dtype, const void *q,
                                                 const void *k_cache, const void *v_cache,
                                                 const int32_t *block_tables, int max_blocks_per_seq,
                                                 const int32_t *seq_lens, int max_seq_len, int num_seqs,
                                                 int num_heads, int num_kv_heads, int head_dim,
                                                 int num_blocks, int block_size, float scale,
                                                 pk_stream_t stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0 ||
        max_blocks_per_seq < 0 || max_seq_len < 0 || block_size <= 0)
        return PK_ERR_SHAPE;
    if (num_heads % num_kv_heads) return PK_ERR_SHAPE;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return PK_ERR_SHAPE;
    if (out_dtype != PK_BF16 && out_dtype != PK_FP32) return PK_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PK_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PK_ERR_UNSUPPORTED;
    if (!group_ok(num_heads / num_kv_heads)) return PK_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PK_ERR_SHAPE;
    if (num_seqs > 65535 || num_kv_heads * 2 > 65535) return PK_ERR_SHAPE;
    if (num_seqs == 0) return PK_OK;
    if (!out || !q || !seq_lens || (max_seq_len > 0 && (!k_cache || !v_cache || !block_tables)))
        return PK_ERR_NULL;
    if (!pk::aligned16(out) || !pk::aligned16(q) || !pk::aligned16(k_cache) || !pk::aligned16(v_cache))
        return PK_ERR_ALIGNMENT;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t out_bytes = static_cast<size_t>(num_seqs) * num_heads * head_dim * (out_dtype == PK_FP32 ? 4 : 2);
    if (max_seq_len == 0)   // every sequence is empty: the output is zeros
        return cudaMemsetAsync(out, 0, out_bytes, st) == cudaSuccess ? PK_OK : PK_ERR_CUDA;

    const int sms = pk::sm_count();
    if (sms <= 0) return PK_ERR_NO_DEVICE;
    const int ctas = std::min(sms, kNoAllocMaxCtas);
    // The slots of `ctas` CTAs must fit the fixed array; reject otherwise.
    if (pk::tc_slot_bytes() != kNoAllocSlotBytes || 2 * static_cast<size_t>(ctas) * pk::tc_slot_bytes() > kScratchBytes)
        return PK_ERR_WORKSPACE;

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
    if (max_seq_len > 128) {          // only sequences longer than one tile can be cut
        p.tc_slots = scratch_address();
        if (!p.tc_slots) return PK_ERR_CUDA;
    }
    p.err = pk::error_word_ptr();
    if (!p.err) return PK_ERR_NO_DEVICE;
    return pk::launch_decode_tensor_core_grid(p, st, ctas) == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}
