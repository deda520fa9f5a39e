// Paged decode attention on the 5th-generation tensor cores (tcgen05), for a
// GQA group wide enough to make the score computation a dense contraction.
//
// What it computes is the block-wise attention of "vLLM — PagedAttention"
// (Mathematical Formulation, Equation 4): keys and values are fetched block by
// block through the block table and combined with an online softmax
// ("PagedAttention from First Principles", §5); long sequences are split and
// their parts combined by a log-sum-exp merge (§17, the partitioned kernel and
// its reduce step).
//
// Work split.  The flattened space (sequence, KV head, 128-token tile) is cut
// into gridDim.x equal contiguous ranges, one per persistent CTA (one CTA per
// SM).  A CTA's range covers whole (sequence, head) segments, which it writes
// straight to the output, plus at most two cut segments at its ends, whose
// partial (max, denominator, unnormalised output) go to a workspace slot and
// are combined by the merge kernel.
//
// Per 128-token tile, inside a CTA (192 threads):
//   warp 0  producer: reads the tile's block-table entries (one lane per
//           page), checks them, and TMA-loads each page's K and V rows of this
//           KV head (two 128-byte-swizzled 64-column boxes each) plus the
//           group's 16 query rows into a 3-stage shared-memory ring;
//   warp 1  MMA issuer (one thread): S^T[128 x 16] = K[128 x D] Q^T[D x 16]
//           into TMEM, then, once the probabilities are written,
//           O^T[D x 16] = V^T[D x 128] P^T[128 x 16] into TMEM;
//   warps 2-5 (128 threads, thread <-> TMEM lane): read S^T (one token per
//           thread), mask invalid tokens, take the tile max per query head
//           (shuffles + shared memory), compute p = 2^(s - m) in fp32, round
//           to bf16 for the MMA, keep the running denominator, and fold each
//           tile's O^T into fp32 registers with the rescale factor
//           (thread <-> head-dim row).
// Query heads are padded to the MMA's N = 16; padded columns are ignored.
#include "decode.cuh"
#include "sm100.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace pk {
namespace {

using namespace sm100;

constexpr int kTile = 128;                                   // tokens per tile = MMA M of S^T
constexpr int kStages = 3;
constexpr int kNPad = 16;                                    // MMA N (query heads, padded)
constexpr int kThreads = 192;
constexpr uint32_t kChunkBytes = kTile * 128;                // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kKOff = 0;
constexpr uint32_t kVOff = 2 * kChunkBytes;
constexpr uint32_t kQOff = 4 * kChunkBytes;
constexpr uint32_t kQChunkBytes = kNPad * 128;
constexpr uint32_t kStageBytes = 4 * kChunkBytes + 2 * kQChunkBytes;
constexpr uint32_t kPBytes = kTile * kNPad * 2;
constexpr uint32_t kTmemCols = 64;                           // S^T x2 (16 cols), O^T x2 (16 cols)
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 32;
constexpr uint64_t kWaitLimitNs = 1000000000ull;             // 1 s: far beyond any legal wait

constexpr uint32_t kIdescQK = idesc_bf16(kTile, kNPad, 0, 0);   // A = K (K-major), B = Q (K-major)
constexpr uint32_t kIdescPV = idesc_bf16(128, kNPad, 1, 1);     // A = V^T (MN-major), B = P^T (MN-major)

struct Misc {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_full[2];
    uint64_t drain;
    int64_t scan[kThreads];
    int64_t total;
    int64_t rem0;
    int32_t s0;
    uint32_t tmem_base;
    int abort;
    int never;
    uint32_t mask[kStages][4];
    float red[2][4][kNPad];
    float lsum[4][kNPad];
};

constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 2 * kPBytes + sizeof(Misc);

// Workspace slot of a cut segment.
struct Slot {
    int32_t flag;          // slot 0 only: 1 = this CTA merges the segment
    int32_t s, h, pad;
    int64_t start_tile;    // flattened index of the segment's (s, h) tile 0
    int64_t total_tiles;
    int64_t pad2[4];
    float m[kNPad];
    float l[kNPad];
    float o[kNPad * 128];
};
constexpr size_t kMaxCtas = 1024;

__device__ __forceinline__ int clamp_len(const DecodeParams &p, int s, int cap) {
    const int raw = p.seq_lens[s];
    return raw < 0 ? 0 : (raw > cap ? cap : raw);
}

// Walks the flattened (sequence, KV head, tile) space in order.
struct Walk {
    int s, h, t, nt, L;
    __device__ __forceinline__ void load(const DecodeParams &p, int cap) {
        L = clamp_len(p, s, cap);
        nt = (L + kTile - 1) / kTile;
    }
    __device__ __forceinline__ void next(const DecodeParams &p, int cap) {
        if (++t < nt) return;
        t = 0;
        if (++h < p.num_kv_heads) return;
        h = 0;
        do {
            if (++s >= p.num_seqs) return;
            load(p, cap);
        } while (nt == 0);
    }
};

__device__ __forceinline__ int64_t range_begin(int64_t c, int64_t T, int64_t C) { return c * T / C; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void store_out(const DecodeParams &p, size_t idx, float v) {
    if (p.out_fp32) static_cast<float *>(p.out)[idx] = v;
    else static_cast<uint16_t *>(p.out)[idx] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= kNPad, "group");
    constexpr int NCH = D / 64;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *stage_ptr = smem;
    uint8_t *p_ptr = smem + kStages * kStageBytes;
    Misc *misc = reinterpret_cast<Misc *>(p_ptr + 2 * kPBytes);
    const uint32_t stage_addr = smem_u32(stage_ptr);
    const uint32_t p_addr = smem_u32(p_ptr);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, C = gridDim.x;
    const int N = p.num_seqs, Hkv = p.num_kv_heads, H = p.num_heads, B = p.block_size;
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * B);
    Slot *slots = static_cast<Slot *>(p.tc_slots);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&misc->full[i]), 1);
            mbar_init(smem_u32(&misc->empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&misc->s_full[i]), 1);
            mbar_init(smem_u32(&misc->p_full[i]), 1);
            mbar_init(smem_u32(&misc->o_full[i]), 1);
        }
        mbar_init(smem_u32(&misc->drain), 1);
        misc->abort = 0;
        misc->never = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 0 && slots) slots[2 * c].flag = 0;
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
    }

    // ---- this CTA's range of the flattened tile space ----------------------
    const int per = (N + kThreads - 1) / kThreads;
    const int s_lo = min(N, static_cast<int>(threadIdx.x) * per), s_hi = min(N, s_lo + per);
    int64_t mine = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        const int raw = p.seq_lens[s];
        if ((raw < 0 || raw > cap) && s % C == c) set_error(p.err, PK_DEVERR_SEQ_LEN);
        const int L = raw < 0 ? 0 : (raw > cap ? cap : raw);
        mine += static_cast<int64_t>((L + kTile - 1) / kTile) * Hkv;
    }
    misc->scan[threadIdx.x] = mine;
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t acc = 0;
        for (int i = 0; i < kThreads; ++i) {
            const int64_t v = misc->scan[i];
            misc->scan[i] = acc;
            acc += v;
        }
        misc->total = acc;
    }
    __syncthreads();
    const int64_t T = misc->total;
    const int64_t beg = range_begin(c, T, C), end = range_begin(c + 1, T, C);
    const int n_tiles = static_cast<int>(end - beg);
    if (n_tiles > 0) {
        int64_t acc = misc->scan[threadIdx.x];
        if (acc <= beg && beg < acc + mine) {
            for (int s = s_lo; s < s_hi; ++s) {
                const int64_t w = static_cast<int64_t>((clamp_len(p, s, cap) + kTile - 1) / kTile) * Hkv;
                if (beg < acc + w) {
                    misc->s0 = s;
                    misc->rem0 = beg - acc;
                    break;
                }
                acc += w;
            }
        }
    }
    // Empty sequences: zeros, written by CTA s % C.
    for (int s = c; s < N; s += C) {
        if (clamp_len(p, s, cap) != 0) continue;
        for (int i = threadIdx.x; i < H * D; i += kThreads) store_out(p, static_cast<size_t>(s) * H * D + i, 0.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;

    Walk w0{};
    if (n_tiles > 0) {
        w0.s = misc->s0;
        w0.load(p, cap);
        w0.h = static_cast<int>(misc->rem0 / w0.nt);
        w0.t = static_cast<int>(misc->rem0 % w0.nt);
    }

    if (warp == 0) {
        // ================= producer =================
        Walk w = w0;
        const int MB = p.max_blocks_per_seq;
        int issued = 0;
        for (int i = 0; i < n_tiles; ++i) {
            const int st = i % kStages;
            int got = 1;
            if (lane == 0)
                got = mbar_wait(smem_u32(&misc->empty[st]), ((i / kStages) & 1) ^ 1, &misc->abort, kWaitLimitNs);
            if (!__shfl_sync(0xffffffffu, got, 0)) {      // one decision for the whole warp
                if (lane == 0) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                }
                break;
            }
            const int tok0 = w.t * kTile;
            const int vlen = min(kTile, w.L - tok0);
            const int pages = (vlen + B - 1) / B;
            const int first_page = tok0 / B;
            int phys = -1;
            bool ok = false;
            if (lane < pages) {
                phys = p.block_tables[static_cast<size_t>(w.s) * MB + first_page + lane];
                ok = phys >= 0 && phys < p.num_blocks;
                if (!ok) set_error(p.err, PK_DEVERR_BLOCK_ID);
            }
            uint32_t bits = 0;
            const int r0 = lane * B;
            if (ok) {
                const int nrows = min(B, vlen - r0);
                bits = (nrows >= 32 ? 0xffffffffu : ((1u << nrows) - 1u)) << (r0 & 31);
            }
            const int word = r0 >> 5;
            const uint32_t m0 = __reduce_or_sync(0xffffffffu, word == 0 ? bits : 0u);
            const uint32_t m1 = __reduce_or_sync(0xffffffffu, word == 1 ? bits : 0u);
            const uint32_t m2 = __reduce_or_sync(0xffffffffu, word == 2 ? bits : 0u);
            const uint32_t m3 = __reduce_or_sync(0xffffffffu, word == 3 ? bits : 0u);
            const uint32_t nok = __popc(__ballot_sync(0xffffffffu, ok));
            const uint32_t full = smem_u32(&misc->full[st]);
            const uint32_t sbase = stage_addr + st * kStageBytes;
            if (lane == 0) {
                misc->mask[st][0] = m0;
                misc->mask[st][1] = m1;
                misc->mask[st][2] = m2;
                misc->mask[st][3] = m3;
                mbar_arrive_expect_tx(full, nok * B * 128u * NCH * 2u + kNPad * 128u * NCH);
            }
            __syncwarp();
            if (ok) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    tma_load_4d(sbase + kKOff + ch * kChunkBytes + r0 * 128, &tm_k, full, ch * 64, w.h, 0, phys);
                    tma_load_4d(sbase + kVOff + ch * kChunkBytes + r0 * 128, &tm_v, full, ch * 64, w.h, 0, phys);
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    tma_load_2d(sbase + kQOff + ch * kQChunkBytes, &tm_q, full, ch * 64, w.s * H + w.h * G);
            }
            ++issued;
            w.next(p, cap);
        }
        // On abort, let this warp's copies land before the CTA can exit.
        if (misc->abort && lane == 0) {
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(smem_u32(&misc->full[i % kStages]), (i / kStages) & 1, &misc->never, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            bool alive = true;
            auto pv = [&](int j) {
                const int pb = j & 1;
                if (!mbar_wait(smem_u32(&misc->p_full[pb]), (j >> 1) & 1, &misc->abort, kWaitLimitNs)) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                    alive = false;
                    return;
                }
                tc_fence_after();
                const uint32_t vbase = stage_addr + (j % kStages) * kStageBytes + kVOff;
                const uint32_t pbase = p_addr + pb * kPBytes;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t a = smem_desc(vbase + kk * 16 * 128, kChunkBytes, 1024, kLayoutSw128);
                    const uint64_t b = smem_desc(pbase + kk * 512, 256, 128, kLayoutNone);
                    mma_bf16(tmem + kTmemO + pb * kNPad, a, b, kIdescPV, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&misc->o_full[pb]));
                mma_commit(smem_u32(&misc->empty[j % kStages]));
            };
            int i = 0;
            for (; i < n_tiles && alive; ++i) {
                const int st = i % kStages;
                if (!mbar_wait(smem_u32(&misc->full[st]), (i / kStages) & 1, &misc->abort, kWaitLimitNs)) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                    alive = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sbase = stage_addr + st * kStageBytes;
                const int sb = i & 1;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * kQChunkBytes + (kk & 3) * 32;
                    const uint64_t a = smem_desc(sbase + kKOff + off, 16, 1024, kLayoutSw128);
                    const uint64_t b = smem_desc(sbase + kQOff + qoff, 16, 1024, kLayoutSw128);
                    mma_bf16(tmem + kTmemS + sb * kNPad, a, b, kIdescQK, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&misc->s_full[sb]));
                if (i > 0) pv(i - 1);
            }
            if (alive && n_tiles > 0) pv(n_tiles - 1);
            // Let every issued MMA finish before the CTA can release TMEM.
            mma_commit(smem_u32(&misc->drain));
            mbar_wait(smem_u32(&misc->drain), 0, &misc->never, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ================= softmax + correction (warps 2-5) =================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        float m_run[G], l_run[G], alpha_prev[G], o_acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
            alpha_prev[g] = 0.f;
            o_acc[g] = 0.f;
        }
        bool first_corr = true;
        int seg_t0 = 0, seg_i0 = 0;
        Walk w = w0;
        auto correct = [&](int j, const float (&a)[G]) -> bool {
            const int ob = j & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->o_full[ob]), (j >> 1) & 1, &misc->never,
                                                   kWaitLimitNs)))
                return false;
            tc_fence_after();
            float ov[16];
            tmem_ld16(lane_addr + kTmemO + ob * kNPad, ov);
#pragma unroll
            for (int g = 0; g < G; ++g) o_acc[g] = first_corr ? ov[g] : fmaf(o_acc[g], a[g], ov[g]);
            first_corr = false;
            return true;
        };
        for (int i = 0; i < n_tiles; ++i) {
            const bool seg_first = (i == 0) || (w.t == 0);
            const bool seg_last = (i == n_tiles - 1) || (w.t == w.nt - 1);
            if (seg_first) {
                seg_t0 = w.t;
                seg_i0 = i;
                first_corr = true;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_run[g] = -INFINITY;
                    l_run[g] = 0.f;
                }
            }
            const int st = i % kStages;
            const int sb = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->s_full[sb]), (i >> 1) & 1, &misc->never,
                                                   kWaitLimitNs))) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            float sv[16];
            tmem_ld16(lane_addr + kTmemS + sb * kNPad, sv);
            const bool valid = (misc->mask[st][row >> 5] >> (row & 31)) & 1u;
            float s2[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                s2[g] = valid ? sv[g] * p.scale_log2 : -INFINITY;
                const float mx = warp_max(s2[g]);
                if (lane == 0) misc->red[sb][quad][g] = mx;
            }
            named_bar_sync(1, 128);
            float alpha[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float t = fmaxf(fmaxf(misc->red[sb][0][g], misc->red[sb][1][g]),
                                      fmaxf(misc->red[sb][2][g], misc->red[sb][3][g]));
                const float mn = fmaxf(m_run[g], t);
                alpha[g] = m_run[g] == -INFINITY ? 0.f : fast_exp2(m_run[g] - mn);
                m_run[g] = mn;
            }
            float pr[kNPad];
#pragma unroll
            for (int g = 0; g < kNPad; ++g) pr[g] = 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) pr[g] = valid ? fast_exp2(s2[g] - m_run[g]) : 0.f;
            uint32_t packed[kNPad / 2];
#pragma unroll
            for (int gp = 0; gp < kNPad / 2; ++gp) packed[gp] = pack_bf16x2(pr[2 * gp], pr[2 * gp + 1]);
            // The denominator sums the bf16 weights the MMA actually applies.
#pragma unroll
            for (int g = 0; g < G; ++g)
                l_run[g] = fmaf(l_run[g], alpha[g], (g & 1) ? bf16_hi(packed[g >> 1]) : bf16_lo(packed[g >> 1]));
            if (!valid) {
                // The MMA multiplies every V row by its probability; rows of
                // masked tokens may hold stale or non-finite bits, so zero them.
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(stage_ptr + st * kStageBytes + kVOff + ch * kChunkBytes + row * 128);
#pragma unroll
                    for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0, 0, 0, 0);
                }
            }
            uint8_t *prow = p_ptr + sb * kPBytes + (row >> 3) * 256 + (row & 7) * 16;
            *reinterpret_cast<uint4 *>(prow) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4 *>(prow + 128) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(1, 128);
            if (threadIdx.x == 64) mbar_arrive(smem_u32(&misc->p_full[sb]));

            bool ok = true;
            if (!seg_first) ok = correct(i - 1, alpha_prev);
            if (ok && seg_last) ok = correct(i, alpha);
            if (!ok) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) alpha_prev[g] = alpha[g];

            if (seg_last) {
                // Denominator over the 128 threads.
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float v = warp_sum(l_run[g]);
                    if (lane == 0) misc->lsum[quad][g] = v;
                }
                named_bar_sync(1, 128);
                float l[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    l[g] = misc->lsum[0][g] + misc->lsum[1][g] + misc->lsum[2][g] + misc->lsum[3][g];
                const bool complete = seg_t0 == 0 && w.t == w.nt - 1;
                if (complete) {
                    if (row < D) {
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            store_out(p, (static_cast<size_t>(w.s) * H + w.h * G + g) * D + row,
                                      l[g] > 0.f ? o_acc[g] / l[g] : 0.f);
                    }
                } else {
                    const int slot_idx = seg_i0 == 0 ? 0 : 1;
                    Slot *sl = slots + 2 * c + slot_idx;
                    if (row < D) {
#pragma unroll
                        for (int g = 0; g < G; ++g) sl->o[g * D + row] = o_acc[g];
                    }
                    if (row == 0) {
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            sl->m[g] = m_run[g];
                            sl->l[g] = l[g];
                        }
                        sl->s = w.s;
                        sl->h = w.h;
                        sl->start_tile = beg + seg_i0 - seg_t0;
                        sl->total_tiles = T;
                        // Cut at its start and finished here: this CTA merges it.
                        if (slot_idx == 0) sl->flag = (seg_t0 > 0 && w.t == w.nt - 1) ? 1 : 0;
                    }
                }
            }
            w.next(p, cap);
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One CTA per main-kernel CTA c: if c's first segment was cut at its start
// and ends in c, combine the parts of that segment from every CTA it spans.
template <int D, int G>
__global__ void __launch_bounds__(128)
decode_tc_merge_kernel(const DecodeParams p, int C) {
    const Slot *slots = static_cast<const Slot *>(p.tc_slots);
    const int c = blockIdx.x;
    const Slot *mine = slots + 2 * c;
    if (mine->flag != 1) return;
    const int s = mine->s, h = mine->h;
    const int64_t start = mine->start_tile, T = mine->total_tiles;
    int ca = static_cast<int>(start * C / T);
    while (ca + 1 < C && range_begin(ca + 1, T, C) <= start) ++ca;
    // Contributors are the CTAs from ca to c with a non-empty range (when the
    // grid has more CTAs than tiles, some ranges are empty and hold no slot).
    float M[G];
#pragma unroll
    for (int g = 0; g < G; ++g) M[g] = -INFINITY;
    for (int cc = ca; cc <= c; ++cc) {
        if (range_begin(cc, T, C) == range_begin(cc + 1, T, C)) continue;
        const Slot *sl = slots + 2 * cc + (range_begin(cc, T, C) >= start ? 0 : 1);
#pragma unroll
        for (int g = 0; g < G; ++g) M[g] = fmaxf(M[g], sl->m[g]);
    }
    const int d = threadIdx.x;
    if (d >= D) return;
    float num[G], den[G];
#pragma unroll
    for (int g = 0; g < G; ++g) num[g] = den[g] = 0.f;
    for (int cc = ca; cc <= c; ++cc) {
        if (range_begin(cc, T, C) == range_begin(cc + 1, T, C)) continue;
        const Slot *sl = slots + 2 * cc + (range_begin(cc, T, C) >= start ? 0 : 1);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float a = rescale(sl->m[g], M[g]);
            den[g] = fmaf(a, sl->l[g], den[g]);
            num[g] = fmaf(a, sl->o[g * D + d], num[g]);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
        store_out(p, (static_cast<size_t>(s) * p.num_heads + h * G + g) * D + d,
                  den[g] > 0.f ? num[g] / den[g] : 0.f);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

bool encode_cache_map(CUtensorMap *m, const void *base, const DecodeParams &p) {
    auto enc = get_encoder();
    if (!enc) return false;
    const cuuint64_t D = p.head_dim, Hkv = p.num_kv_heads, B = p.block_size;
    const cuuint64_t P = p.num_blocks > 0 ? p.num_blocks : 1;
    cuuint64_t dims[4] = {D, Hkv, B, P};
    cuuint64_t strides[3] = {D * 2, Hkv * D * 2, B * Hkv * D * 2};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(B), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap *m, const DecodeParams &p) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.head_dim),
                          static_cast<cuuint64_t>(p.num_seqs) * p.num_heads};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.head_dim) * 2};
    cuuint32_t box[2] = {64, kNPad};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p.q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_dg(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const DecodeParams &p,
                      int C, cudaStream_t stream) {
    static bool attr_set = false;   // per instantiation; setting it twice is harmless
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    decode_tc_kernel<D, G><<<C, kThreads, kSmemBytes, stream>>>(mk, mv, mq, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!p.tc_slots) return cudaSuccess;   // no sequence longer than one tile: nothing is cut
    decode_tc_merge_kernel<D, G><<<C, 128, 0, stream>>>(p, C);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const DecodeParams &p,
                     int C, cudaStream_t stream) {
    switch (p.num_heads / p.num_kv_heads) {
        case 1: return launch_dg<D, 1>(mk, mv, mq, p, C, stream);
        case 2: return launch_dg<D, 2>(mk, mv, mq, p, C, stream);
        case 4: return launch_dg<D, 4>(mk, mv, mq, p, C, stream);
        case 8: return launch_dg<D, 8>(mk, mv, mq, p, C, stream);
        case 16: return launch_dg<D, 16>(mk, mv, mq, p, C, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t tc_workspace_bytes() { return 2 * kMaxCtas * sizeof(Slot); }

cudaError_t launch_decode_tensor_core(const DecodeParams &p, cudaStream_t stream) {
    CUtensorMap mk, mv, mq;
    if (!encode_cache_map(&mk, p.k_cache, p) || !encode_cache_map(&mv, p.v_cache, p) || !encode_q_map(&mq, p))
        return cudaErrorInvalidValue;
    int C = sm_count();
    if (C <= 0) return cudaErrorNoDevice;
    if (C > static_cast<int>(kMaxCtas)) C = static_cast<int>(kMaxCtas);
    return p.head_dim == 64 ? launch_d<64>(mk, mv, mq, p, C, stream) : launch_d<128>(mk, mv, mq, p, C, stream);
}

}  // namespace pk

namespace pk {

size_t tc_slot_bytes() { return sizeof(Slot); }

cudaError_t launch_decode_tensor_core_grid(const DecodeParams &p, cudaStream_t stream, int ctas) {
    CUtensorMap mk, mv, mq;
    if (ctas <= 0 || ctas > static_cast<int>(kMaxCtas)) return cudaErrorInvalidValue;
    if (!encode_cache_map(&mk, p.k_cache, p) || !encode_cache_map(&mv, p.v_cache, p) || !encode_q_map(&mq, p))
        return cudaErrorInvalidValue;
    return p.head_dim == 64 ? launch_d<64>(mk, mv, mq, p, ctas, stream) : launch_d<128>(mk, mv, mq, p, ctas, stream);
}

}  // namespace pk
