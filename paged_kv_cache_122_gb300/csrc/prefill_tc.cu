// Multi-query paged attention for WIDE query blocks (chunked prefill): many
// newest tokens of a sequence attend its paged cache, causal among
// themselves ("PagedAttention from First Principles", §12 chunked prefill:
// a chunk of a prompt is processed over the cache in one pass; the
// attention itself is the decode definition of "vLLM — PagedAttention",
// Mathematical Formulation, Equation 4, with the causal limit).
//
// Orientation.  The decode kernel puts keys on the MMA's M and at most 16
// query columns on N.  Here the queries are the dense side: a CTA owns 128
// query rows -- 128 / G consecutive query tokens x the G query heads of one
// KV head, row = token * G + head -- and streams the sequence's keys in
// 128-token tiles:
//   S[128 x 128]  = Q[128 x D] K_tile^T          (tcgen05, fp32 in TMEM)
//   O[128 x D]   += P[128 x 128] V_tile[128 x D]  (tcgen05, fp32 in TMEM)
// so one thread of the softmax warps owns one query row of S, P and O and
// needs no cross-thread reduction.
//
// Per CTA (192 threads):
//   warp 0    producer: the Q block once (one TMA box of 64 elements x G
//             heads x 128/G tokens per 64-column chunk), then per key tile
//             each page's K rows and V rows of this KV head into a 2-stage
//             ring (K and V complete separate barriers);
//   warp 1    MMA issuer (one thread): S of tile i, then P.V of tile i-1
//             with P read from tensor memory;
//   warps 2-5 softmax, thread <-> query row: row max against a reference
//             max that moves only when exceeded by more than 2^8 (then the
//             row's O and denominator are rescaled), p = 2^(s - m_ref) with
//             the causal and validity masks, bf16 P rows stored into TMEM
//             (double-buffered, so the softmax of tile i never waits for the
//             P.V of tile i-1 unless its O must be rescaled), and at the end
//             O / l stored.
#include "decode.cuh"
#include "sm100.cuh"
#include "tmem_wide.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

namespace pk {
namespace {

using namespace sm100;

constexpr int kRows = 128;                      // query rows per CTA = MMA M
constexpr int kKeys = 128;                      // keys per tile = MMA N of S
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr uint32_t kChunk = 128 * 128;          // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kKOff = 0;
constexpr uint32_t kVOff = 2 * kChunk;
constexpr uint32_t kStageBytes = 4 * kChunk;    // K and V of one key tile (D <= 128)
constexpr uint32_t kQBytes = 2 * kChunk;
constexpr uint32_t kTmemCols = 512;             // S x2 (128 cols each), O (<= 128 cols), P x2 (64 cols each)
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;                // bf16 P: two keys per 32-bit column
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kRescaleLog2 = 8.0f;

struct Misc {
    uint64_t full[kStages];     // K rows of a stage landed
    uint64_t vfull[kStages];    // V rows of a stage landed
    uint64_t empty[kStages];    // P.V of the stage's tile done
    uint64_t q_full;
    uint64_t s_full[2];         // S of a tile in TMEM (by tile parity)
    uint64_t p_full;            // P of a tile written (4 softmax warps)
    uint64_t pv_done[2];        // P.V of a tile done (by tile parity): its P buffer and O free
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int never;
    uint32_t mask[kStages][4];  // valid keys of a stage's tile
};

constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + kQBytes + sizeof(Misc);

__device__ __forceinline__ void store_row_out(const DecodeParams &p, size_t idx, float v) {
    if (p.out_fp32) static_cast<float *>(p.out)[idx] = v;
    else static_cast<uint16_t *>(p.out)[idx] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}

// grid: one CTA per (sequence, KV head, query block of 128 / G tokens),
// blockIdx.x = (s * Hkv + h) * qblocks + j; CTAs past a sequence's queries exit.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const DecodeParams p, int qblocks) {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= 16 && (G & (G - 1)) == 0, "group");
    constexpr int NCH = D / 64;
    constexpr int QT = kRows / G;                 // query tokens per CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = p.num_kv_heads, H = p.num_heads, B = p.block_size;
    const int j = blockIdx.x % qblocks;
    const int h = (blockIdx.x / qblocks) % Hkv;
    const int s = blockIdx.x / qblocks / Hkv;
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * B);
    // V of a tile in shared memory: one slot of v_page bytes per page, each
    // [half][row][64] (B is 8, 16 or 32).
    const uint32_t v_page = static_cast<uint32_t>(B) * 128u * NCH;
    const uint32_t v_half = static_cast<uint32_t>(B) * 128u;        // between the two 64-element halves
    const uint32_t v_group = B >= 16 ? 1024u : v_page;              // between groups of 8 keys
    int L = p.seq_lens[s];
    const int q0 = p.cu_q_lens[s];
    const int qn = p.cu_q_lens[s + 1] - q0;
    if (L < 0 || L > cap || qn < 0 || qn > max(L, 0)) {
        if (j == 0 && h == 0 && threadIdx.x == 0) set_error(p.err, PK_DEVERR_SEQ_LEN);
        return;
    }
    const int qt0 = j * QT;                       // first query token of this CTA
    if (qt0 >= qn) return;
    const int qt1 = min(qn, qt0 + QT);
    const int pos0 = L - qn;                      // position of the sequence's first query
    const int last_pos = pos0 + qt1 - 1;          // the last key any row of this CTA sees
    const int n_tiles = last_pos / kKeys + 1;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *stage_ptr = smem;
    uint8_t *q_ptr = smem + kStages * kStageBytes;
    Misc *misc = reinterpret_cast<Misc *>(q_ptr + kQBytes);
    const uint32_t stage_addr = smem_u32(stage_ptr);
    const uint32_t q_addr = smem_u32(q_ptr);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&misc->full[i]), 1);
            mbar_init(smem_u32(&misc->vfull[i]), 1);
            mbar_init(smem_u32(&misc->empty[i]), 1);
        }
        mbar_init(smem_u32(&misc->q_full), 1);
        mbar_init(smem_u32(&misc->s_full[0]), 1);
        mbar_init(smem_u32(&misc->s_full[1]), 1);
        mbar_init(smem_u32(&misc->p_full), 4);
        mbar_init(smem_u32(&misc->pv_done[0]), 1);
        mbar_init(smem_u32(&misc->pv_done[1]), 1);
        mbar_init(smem_u32(&misc->drain), 1);
        misc->abort = 0;
        misc->never = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;

    if (warp == 0) {
        // ================= producer =================
        const int MB = p.max_blocks_per_seq;
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const uint32_t qf = smem_u32(&misc->q_full);
            mbar_arrive_expect_tx(qf, kRows * 128u * NCH);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
                tma_load_3d(q_addr + ch * kChunk, &tm_q, qf, ch * 64, h * G, q0 + qt0);
        }
        // Block-table entries of a tile, one page per lane; the next tile's
        // are fetched while the current tile's copies are issued.
        auto fetch = [&](int t) -> int {
            const int tok = t * kKeys;
            const int pg = (min(kKeys, L - tok) + B - 1) / B;
            return lane < pg ? p.block_tables[static_cast<size_t>(s) * MB + tok / B + lane] : -1;
        };
        int phys_next = fetch(0);
        int issued = 0;
        for (int i = 0; i < n_tiles; ++i) {
            const int st = i % kStages;
            const int phys_raw = phys_next;
            int got = 1;
            if (lane == 0)
                got = mbar_wait(smem_u32(&misc->empty[st]), ((i / kStages) & 1) ^ 1, &misc->abort, kWaitLimitNs);
            if (!__shfl_sync(0xffffffffu, got, 0)) {
                if (lane == 0) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                }
                break;
            }
            const int tok0 = i * kKeys;
            const int vlen = min(kKeys, L - tok0);
            const int pages = (vlen + B - 1) / B;
            int phys = -1;
            bool ok = false;
            if (lane < pages) {
                phys = phys_raw;
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
            const uint32_t vfull = smem_u32(&misc->vfull[st]);
            const uint32_t sbase = stage_addr + st * kStageBytes;
            if (lane == 0) {
                misc->mask[st][0] = m0;
                misc->mask[st][1] = m1;
                misc->mask[st][2] = m2;
                misc->mask[st][3] = m3;
                mbar_arrive_expect_tx(full, nok * B * 128u * NCH);
                mbar_arrive_expect_tx(vfull, nok * B * 128u * NCH);
            }
            __syncwarp();
            if (ok) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    tma_load_4d(sbase + kKOff + ch * kChunk + r0 * 128, &tm_k, full, ch * 64, h, 0, phys);
                // V: one box per page, [half][row][64] at the page's slot.
                tma_load_5d(sbase + kVOff + r0 * 128 * NCH, &tm_v, vfull, 0, 0, 0, h, phys);
            }
            ++issued;
            if (i + 1 < n_tiles) phys_next = fetch(i + 1);
        }
        if (misc->abort && lane == 0) {
            mbar_wait(smem_u32(&misc->q_full), 0, &misc->never, kWaitLimitNs);
            for (int i = max(0, issued - kStages); i < issued; ++i) {
                mbar_wait(smem_u32(&misc->full[i % kStages]), (i / kStages) & 1, &misc->never, kWaitLimitNs);
                mbar_wait(smem_u32(&misc->vfull[i % kStages]), (i / kStages) & 1, &misc->never, kWaitLimitNs);
            }
        }
    }
    else if (warp == 1) {
        // ================= MMA issuer =================
        // S of tile i is issued before P.V of tile i-1, so the scores of the
        // next tile are computed while the softmax works on the current one.
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(kRows, kKeys, 0, 0);   // A = Q, B = K, both K-major
            constexpr uint32_t kIdescO = idesc_bf16(kRows, D, 0, 1);       // A = P (TMEM), B = V (MN-major)
            bool alive = mbar_wait(smem_u32(&misc->q_full), 0, &misc->abort, kWaitLimitNs);
            auto pv = [&](int t) {
                alive = alive && mbar_wait(smem_u32(&misc->p_full), t & 1, &misc->abort, kWaitLimitNs) &&
                        mbar_wait(smem_u32(&misc->vfull[t % kStages]), (t / kStages) & 1, &misc->abort,
                                  kWaitLimitNs);
                if (!alive) return;
                tc_fence_after();
                const uint32_t vbase = stage_addr + (t % kStages) * kStageBytes + kVOff;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    // Keys 16kk .. 16kk+15: page (16kk / B) at its slot, row 16kk % B.
                    const uint32_t t0 = kk * 16;
                    const uint64_t b = smem_desc(vbase + (t0 / B) * v_page + (t0 % B) * 128, v_half, v_group,
                                                 kLayoutSw128);
                    mma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + (t & 1) * 64 + kk * 8, b, kIdescO,
                                    (t > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&misc->pv_done[t & 1]));
                mma_commit(smem_u32(&misc->empty[t % kStages]));
            };
            for (int i = 0; i < n_tiles && alive; ++i) {
                const int st = i % kStages;
                alive = mbar_wait(smem_u32(&misc->full[st]), (i / kStages) & 1, &misc->abort, kWaitLimitNs);
                if (!alive) break;
                tc_fence_after();
                const uint32_t kbase = stage_addr + st * kStageBytes + kKOff;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                    const uint64_t a = smem_desc(q_addr + off, 16, 1024, kLayoutSw128);
                    const uint64_t b = smem_desc(kbase + off, 16, 1024, kLayoutSw128);
                    mma_bf16(tmem + kTmemS + (i & 1) * kKeys, a, b, kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&misc->s_full[i & 1]));
                if (i > 0) pv(i - 1);
            }
            if (alive) pv(n_tiles - 1);
            if (!alive) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
            }
            // Let every issued MMA finish before the CTA can release TMEM.
            mma_commit(smem_u32(&misc->drain));
            mbar_wait(smem_u32(&misc->drain), 0, &misc->never, kWaitLimitNs);
        }
        __syncwarp();
    }
    else {
        // ================= softmax (warps 2-5): thread <-> query row =================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const int rr = row / G;                         // query token of this row (rows are token * G + head)
        const int qp = pos0 + qt0 + rr;                 // its position: it sees keys 0 .. qp
        float m_ref = -INFINITY, l_run = 0.f;
        bool alive = true;
        for (int i = 0; i < n_tiles; ++i) {
            const int st = i % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->s_full[i & 1]), (i >> 1) & 1, &misc->never,
                                                   kWaitLimitNs))) {
                alive = false;
                break;
            }
            tc_fence_after();
            uint32_t msk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) msk[c] = misc->mask[st][c];
            const int kbase = i * kKeys;
            const uint32_t sbase = lane_addr + kTmemS + (i & 1) * kKeys;
            // The row's 128 scores of this tile into registers (two loads in
            // flight, one wait).
            uint32_t sa[64], sb[64];
            tmemw::ld64(sbase, sa);
            tmemw::ld64(sbase + 64, sb);
            // This tile's P buffer is free once P.V of tile i - 2 is done (long ago).
            if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[i & 1]), ((i - 2) >> 1) & 1,
                                                             &misc->never, kWaitLimitNs))) {
                alive = false;
                break;
            }
            tmemw::wait_ld(sa);
            tmemw::wait_ld(sb);
            tc_fence_after();
            const uint32_t pbase = lane_addr + kTmemP + (i & 1) * 64;
            auto score = [&](int k) -> float { return __uint_as_float(k < 64 ? sa[k] : sb[k - 64]); };
            // Key k of the tile is visible to this row if its page was
            // loaded and it is not after the row's own position.
            const int lim = qp - kbase;
            auto visible = [&](int k) -> bool { return ((msk[k >> 5] >> (k & 31)) & 1u) && k <= lim; };
            // Tiles every key of which this row sees skip the masks
            // (warp-uniform: the tensor-memory moves below are warp-collective).
            const bool easy = __all_sync(0xffffffffu, kKeys - 1 <= lim &&
                                                          (msk[0] & msk[1] & msk[2] & msk[3]) == 0xffffffffu);
            const float c = p.scale_log2;
            // The tile's row max of c * s over the visible keys, from the raw
            // scores (c >= 0: the max, c < 0: the min; rounding is monotone,
            // so the product of the extreme equals the extreme of the
            // products).  Eight independent chains; a masked key is NaN,
            // which fmaxf / fminf skip.
            float ext[8];
            auto gather = [&](auto easy_tag) {
                constexpr bool kEasy = decltype(easy_tag)::value;
#pragma unroll
                for (int e = 0; e < 8; ++e) ext[e] = kEasy ? score(e) : (visible(e) ? score(e) : __int_as_float(0x7fffffff));
#pragma unroll
                for (int k = 8; k < kKeys; ++k) {
                    const float v = kEasy ? score(k) : (visible(k) ? score(k) : __int_as_float(0x7fffffff));
                    ext[k & 7] = c >= 0.f ? fmaxf(ext[k & 7], v) : fminf(ext[k & 7], v);
                }
            };
            if (easy) gather(std::true_type{});
            else gather(std::false_type{});
            float e4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) e4[e] = c >= 0.f ? fmaxf(ext[e], ext[e + 4]) : fminf(ext[e], ext[e + 4]);
            const float e2a = c >= 0.f ? fmaxf(e4[0], e4[2]) : fminf(e4[0], e4[2]);
            const float e2b = c >= 0.f ? fmaxf(e4[1], e4[3]) : fminf(e4[1], e4[3]);
            const float ex = c >= 0.f ? fmaxf(e2a, e2b) : fminf(e2a, e2b);
            // No visible key (NaN): no candidate for the reference max.
            const float tmax = ex == ex ? ex * c : -INFINITY;
            const bool need = tmax > m_ref + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
                // Move this row's reference max and rescale its O and
                // denominator (rare after the first tile).
                const float mn = need ? tmax : m_ref;
                const float a = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - mn);
                // O holds tiles up to i - 1: wait for that P.V (the only wait on it).
                if (i > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[(i - 1) & 1]),
                                                                ((i - 1) >> 1) & 1, &misc->never, kWaitLimitNs))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                if (i > 0) {
#pragma unroll
                    for (int cc = 0; cc < D / 8; ++cc) {
                        float ov[8];
                        tmem_ld<8>(lane_addr + kTmemO + cc * 8, ov);
#pragma unroll
                        for (int k = 0; k < 8; ++k) ov[k] *= a;
                        tmem_st8(lane_addr + kTmemO + cc * 8, ov);
                    }
                }
                l_run *= a;
                m_ref = mn;
            }
            // p = 2^(c * s - m_ref) as bf16 pairs into this tile's P columns of
            // TMEM (the P.V MMA's A operand); the denominator sums the bf16
            // weights the MMA actually applies, in four chains.
            const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            auto emit = [&](auto easy_tag) {
                constexpr bool kEasy = decltype(easy_tag)::value;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t packed[16];
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const int kk = cc * 32 + k;
                        float p0 = fast_exp2(fmaf(score(kk), c, nm));
                        float p1 = fast_exp2(fmaf(score(kk + 1), c, nm));
                        if constexpr (!kEasy) {
                            p0 = visible(kk) ? p0 : 0.f;
                            p1 = visible(kk + 1) ? p1 : 0.f;
                        }
                        const uint32_t w = pack_bf16x2(p0, p1);
                        packed[k / 2] = w;
                        ls[(k / 2) & 3] += bf16_lo(w) + bf16_hi(w);
                    }
                    tmem_st16(pbase + cc * 16, packed);   // keys 32cc .. 32cc+31 of this row
                }
            };
            if (easy) emit(std::true_type{});
            else emit(std::false_type{});
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // V rows of keys outside the sequence or behind a bad table entry
            // may hold stale or non-finite bits; the MMA multiplies them by 0,
            // so zero them (thread <-> key row) once V has landed.
            const int wrow = row >> 5;                      // select, not an indexed load: msk stays in registers
            const uint32_t mrow = wrow == 0 ? msk[0] : wrow == 1 ? msk[1] : wrow == 2 ? msk[2] : msk[3];
            const bool bad = !((mrow >> (row & 31)) & 1u);
            if (__any_sync(0xffffffffu, bad)) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->vfull[st]), (i / kStages) & 1, &misc->never,
                                                       kWaitLimitNs))) {
                    alive = false;
                    break;
                }
                if (bad) {
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        uint4 *vrow = reinterpret_cast<uint4 *>(stage_ptr + st * kStageBytes + kVOff + (row / B) * v_page +
                                                                ch * B * 128 + (row % B) * 128);
#pragma unroll
                        for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            tmem_wait_st();                 // P is in TMEM before the MMA may read it
            fence_proxy_async_smem();       // zeroed V rows are visible to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&misc->p_full));
        }
        if (alive && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[(n_tiles - 1) & 1]),
                                                         ((n_tiles - 1) >> 1) & 1,
                                                         &misc->never, kWaitLimitNs)))
            alive = false;
        if (!alive) {
            misc->abort = 1;
            set_error(p.err, PK_DEVERR_TIMEOUT);
        } else {
            tc_fence_after();
            // O / l of this row to out[q0 + qt0 + token, h * G + head, :].
            const bool store = qt0 + rr < qn;
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const size_t obase =
                (static_cast<size_t>(q0 + qt0 + rr) * H + h * G + (row & (G - 1))) * static_cast<size_t>(D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float ov[32];
                tmem_ld<32>(lane_addr + kTmemO + c * 32, ov);
                if (store) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) store_row_out(p, obase + c * 32 + k, ov[k] * inv);
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// A tiled map with the 128-byte swizzle the MMA descriptors expect.
bool encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
            const cuuint32_t *box) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_dg(const DecodeParams &p, int max_q_len, cudaStream_t stream) {
    const cuuint64_t Dd = p.head_dim, Hkv = p.num_kv_heads, B = p.block_size;
    const cuuint64_t P = p.num_blocks > 0 ? p.num_blocks : 1;
    const cuuint64_t cdims[4] = {Dd, Hkv, B, P};
    const cuuint64_t cstr[3] = {Dd * 2, Hkv * Dd * 2, B * Hkv * Dd * 2};
    const cuuint32_t cbox[4] = {64, 1, static_cast<cuuint32_t>(B), 1};
    // V: one box per (page, head) with all B rows of both halves, [half][row][64].
    const cuuint64_t vdims[5] = {64, B, Dd / 64, Hkv, P};
    const cuuint64_t vstr[4] = {Hkv * Dd * 2, 128, Dd * 2, B * Hkv * Dd * 2};
    const cuuint32_t vbox[5] = {64, static_cast<cuuint32_t>(B), static_cast<cuuint32_t>(Dd / 64), 1, 1};
    const cuuint64_t qdims[3] = {Dd, static_cast<cuuint64_t>(p.num_heads), static_cast<cuuint64_t>(p.total_q)};
    const cuuint64_t qstr[2] = {Dd * 2, Dd * p.num_heads * 2};
    const cuuint32_t qbox[3] = {64, G, kRows / G};
    CUtensorMap mk, mv, mq;
    if (!encode(&mk, p.k_cache, 4, cdims, cstr, cbox) || !encode(&mv, p.v_cache, 5, vdims, vstr, vbox) ||
        !encode(&mq, p.q, 3, qdims, qstr, qbox))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int qblocks = (max_q_len + kRows / G - 1) / (kRows / G);
    const int64_t grid = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * qblocks;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    prefill_tc_kernel<D, G><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(mk, mv, mq, p, qblocks);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeParams &p, int max_q_len, cudaStream_t stream) {
    switch (p.num_heads / p.num_kv_heads) {
        case 1: return launch_dg<D, 1>(p, max_q_len, stream);
        case 2: return launch_dg<D, 2>(p, max_q_len, stream);
        case 4: return launch_dg<D, 4>(p, max_q_len, stream);
        case 8: return launch_dg<D, 8>(p, max_q_len, stream);
        case 16: return launch_dg<D, 16>(p, max_q_len, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_tensor_core(const DecodeParams &p, int max_q_len, cudaStream_t stream) {
    if (!p.cu_q_lens || max_q_len <= 0) return cudaErrorInvalidValue;
    return p.head_dim == 64 ? launch_d<64>(p, max_q_len, stream) : launch_d<128>(p, max_q_len, stream);
}

}  // namespace pk
