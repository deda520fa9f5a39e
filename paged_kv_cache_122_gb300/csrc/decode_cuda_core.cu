// Paged decode attention on CUDA cores, and the split-K log-sum-exp merge.
//
// This is the straightforward mapping of the pages' kernel description
// ("vLLM — PagedAttention", Fused CUDA Kernels (2): each warp reads one KV block
// through the block table, computes partial attention, and the partial results
// are reduced across warps) with the group of query heads that shares a KV
// head kept in one CTA, so each page is read from HBM once per group chunk.
//
// grid = (partitions, KV heads x group chunks, sequences), 128 threads.
// A CTA owns one partition (part_tokens tokens) of one sequence for GC query
// heads.  Warp w walks pages w, w+4, ... of the partition.  Inside a warp a
// token row of D bf16 is spread over D/8 lanes (one 16-byte load each), so a
// warp covers 32/(D/8) rows per step; dot products are reduced with xor
// shuffles, and each lane keeps an online-softmax state (running max m,
// denominator l, output slice acc) for the rows it visits.  States are merged
// across lanes, then across warps in shared memory.  A sequence with one
// partition writes its output; longer ones write (m, l, acc) partials for the
// merge kernel.
#include "decode.cuh"

namespace pk {
namespace {

constexpr int kWarps = 4;

template <int D, int GC>
__global__ void __launch_bounds__(kWarps * 32)
decode_cuda_core_kernel(const DecodeParams p) {
    constexpr int LPR = D / 8;      // lanes per token row
    constexpr int RPW = 32 / LPR;   // token rows per warp step
    const int part = blockIdx.x;
    const int G = p.num_heads / p.num_kv_heads;
    const int gchunks = G / GC;
    const int kvh = blockIdx.y / gchunks;
    const int h0 = kvh * G + (blockIdx.y % gchunks) * GC;
    const int s = blockIdx.z;

    int L = p.seq_lens[s];
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * p.block_size);
    if (L < 0 || L > cap) {
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_error(p.err, PK_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : cap;
    }
    const int np = (L + p.part_tokens - 1) / p.part_tokens;
    if (part >= max(np, 1)) return;
    const int t0 = part * p.part_tokens;
    const int t1 = min(L, t0 + p.part_tokens);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int dl = (lane % LPR) * 8;
    const int r = lane / LPR;

    float qf[GC][8];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        const uint4 u = ldg_stream(p.q + (static_cast<size_t>(s) * p.num_heads + h0 + g) * D + dl);
        unpack8(u, qf[g]);
    }
    float m[GC], l[GC], acc[GC][8];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] = 0.f;
    }

    const int B = p.block_size;
    const size_t tok_stride = static_cast<size_t>(p.num_kv_heads) * D;
    const int32_t *table = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
    const int pg_end = (t1 + B - 1) / B;
    for (int pg = t0 / B + warp; pg < pg_end; pg += kWarps) {
        const int phys = table[pg];
        if (phys < 0 || phys >= p.num_blocks) {          // warp-uniform
            if (lane == 0) set_error(p.err, PK_DEVERR_BLOCK_ID);
            continue;
        }
        const size_t base = static_cast<size_t>(phys) * B * tok_stride + static_cast<size_t>(kvh) * D + dl;
        const int nvalid = min(B, t1 - pg * B);
        for (int j = r; j < B; j += RPW) {                // same trip count in every lane
            const bool valid = j < nvalid;
            uint4 ku = make_uint4(0, 0, 0, 0), vu = make_uint4(0, 0, 0, 0);
            if (valid) {
                ku = ldg_stream(p.k_cache + base + j * tok_stride);
                vu = ldg_stream(p.v_cache + base + j * tok_stride);
            }
            float kf[8];
            unpack8(ku, kf);
            float sc[GC];
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                float a = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) a = fmaf(qf[g][i], kf[i], a);
                sc[g] = a;
            }
#pragma unroll
            for (int off = LPR / 2; off >= 1; off >>= 1) {
#pragma unroll
                for (int g = 0; g < GC; ++g) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], off);
            }
            if (valid) {
                float vf[8];
                unpack8(vu, vf);
#pragma unroll
                for (int g = 0; g < GC; ++g) {
                    const float s2 = sc[g] * p.scale_log2;
                    const float mn = fmaxf(m[g], s2);
                    const float a = rescale(m[g], mn);
                    const float e = fast_exp2(s2 - mn);
                    l[g] = l[g] * a + e;
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(acc[g][i], a, e * vf[i]);
                    m[g] = mn;
                }
            }
        }
    }

    // Merge the row groups of a warp (lanes that share a d-slice).
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
            const float mn = fmaxf(m[g], mo);
            const float a = rescale(m[g], mn), b = rescale(mo, mn);
            l[g] = l[g] * a + lo * b;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[g][i], off);
                acc[g][i] = acc[g][i] * a + ao * b;
            }
            m[g] = mn;
        }
    }

    __shared__ float sm_m[kWarps][GC], sm_l[kWarps][GC];
    __shared__ __align__(16) float sm_acc[kWarps][GC][D];
    if (r == 0) {
#pragma unroll
        for (int g = 0; g < GC; ++g) {
#pragma unroll
            for (int i = 0; i < 8; ++i) sm_acc[warp][g][dl + i] = acc[g][i];
            if (lane == 0) {
                sm_m[warp][g] = m[g];
                sm_l[warp][g] = l[g];
            }
        }
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < GC * D; idx += kWarps * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][g]);
        float den = 0.f, num = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float a = rescale(sm_m[w][g], M);
            den += a * sm_l[w][g];
            num += a * sm_acc[w][g][d];
        }
        const int h = h0 + g;
        if (np <= 1) {
            const float o = den > 0.f ? num / den : 0.f;
            const size_t oi = (static_cast<size_t>(s) * p.num_heads + h) * D + d;
            if (p.out_fp32) static_cast<float *>(p.out)[oi] = o;
            else static_cast<uint16_t *>(p.out)[oi] = static_cast<uint16_t>(pack_bf16x2(o, 0.f) & 0xffffu);
        } else {
            const size_t u = (static_cast<size_t>(s) * p.num_heads + h) * p.np_cap + part;
            p.ws_o[u * D + d] = num;
            if (d == 0) {
                p.ws_m[u] = M;
                p.ws_l[u] = den;
            }
        }
    }
}

// grid = (sequences, query heads), D threads.  Combines the partitions of a
// split sequence: M = max_p m_p, w_p = 2^(m_p - M),
// out = sum_p w_p acc_p / sum_p w_p l_p.
template <int D>
__global__ void __launch_bounds__(D)
decode_merge_kernel(const DecodeParams p) {
    const int s = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
    int L = p.seq_lens[s];
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * p.block_size);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int np = (L + p.part_tokens - 1) / p.part_tokens;
    if (np <= 1) return;
    const size_t u0 = (static_cast<size_t>(s) * p.num_heads + h) * p.np_cap;
    float M = -INFINITY;
    for (int i = 0; i < np; ++i) M = fmaxf(M, p.ws_m[u0 + i]);
    float den = 0.f, num = 0.f;
    for (int i = 0; i < np; ++i) {
        const float a = rescale(p.ws_m[u0 + i], M);
        den += a * p.ws_l[u0 + i];
        num += a * p.ws_o[(u0 + i) * D + d];
    }
    const float o = den > 0.f ? num / den : 0.f;
    const size_t oi = (static_cast<size_t>(s) * p.num_heads + h) * D + d;
    if (p.out_fp32) static_cast<float *>(p.out)[oi] = o;
    else static_cast<uint16_t *>(p.out)[oi] = static_cast<uint16_t>(pack_bf16x2(o, 0.f) & 0xffffu);
}

template <int D>
cudaError_t launch_cc_d(const DecodeParams &p, cudaStream_t stream) {
    const int G = p.num_heads / p.num_kv_heads;
    const int GC = G >= 8 ? 8 : G;
    dim3 grid(p.np_cap, p.num_kv_heads * (G / GC), p.num_seqs);
    switch (GC) {
        case 1: decode_cuda_core_kernel<D, 1><<<grid, kWarps * 32, 0, stream>>>(p); break;
        case 2: decode_cuda_core_kernel<D, 2><<<grid, kWarps * 32, 0, stream>>>(p); break;
        case 4: decode_cuda_core_kernel<D, 4><<<grid, kWarps * 32, 0, stream>>>(p); break;
        case 8: decode_cuda_core_kernel<D, 8><<<grid, kWarps * 32, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_cuda_core(const DecodeParams &p, cudaStream_t stream) {
    return p.head_dim == 64 ? launch_cc_d<64>(p, stream) : launch_cc_d<128>(p, stream);
}

cudaError_t launch_decode_merge(const DecodeParams &p, cudaStream_t stream) {
    if (p.np_cap <= 1) return cudaSuccess;
    dim3 grid(p.num_seqs, p.num_heads);
    if (p.head_dim == 64) decode_merge_kernel<64><<<grid, 64, 0, stream>>>(p);
    else decode_merge_kernel<128><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pk
