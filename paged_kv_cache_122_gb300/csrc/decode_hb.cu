// Paged decode attention on tcgen05 with head-batched tiles (8 KV heads).
//
// Same definition as the per-head tensor-core kernel (block-wise softmax
// attention through the block table: "vLLM — PagedAttention", Mathematical
// Formulation, Equation 4; online softmax: "PagedAttention from First
// Principles", §5; partitioned long sequences with a reduce step: §17), with
// a different tiling that reads every block row whole:
//
// * A tile is 16 tokens of one sequence for ALL 8 KV heads: 128 MMA rows,
//   row = head * 16 + token.  One TMA box per 64-column chunk per tensor
//   (through a tensor map whose token and head dimensions are swapped) reads
//   16 consecutive 2 KiB token rows of a block: K and V are streamed in whole
//   DRAM rows instead of 256-byte pieces of eight different rows.
// * Scores S^T[128 x NQ] = K_tile[128 x D] Q^T[D x NQ] for all NQ = H query
//   heads of the sequence in one MMA per 16-wide k-step; a row (kv head h,
//   token t) uses only the G columns of its own group.
// * Probabilities are written per KV head (16 tokens x 16 padded columns)
//   and O^T[D x 16] += V_h^T[D x 16] P_h^T[16 x 16] runs once per head, so O
//   for the whole sequence (128 columns) accumulates in TMEM across tiles.
// * Softmax uses a reference max per query head that only moves when a score
//   exceeds it by more than 2^8 (then O and the denominators are rescaled by
//   2^(m_old - m_new)); between moves p = 2^(s - m_ref) <= 2^8, so each tile
//   costs one barrier with an OR-vote and no reductions.  The result is the
//   same softmax: numerator and denominator share the reference.
// * Work split: the flattened (sequence, tile) space is cut into gridDim.x
//   equal ranges, one per persistent CTA.  Each CTA first processes its last
//   segment, then the rest from the start, so both of its possibly cut
//   segments finish early.  A cut segment's parts go to workspace slots; the
//   part that finishes last (epoch-tagged ticket in the workspace) merges them
//   with the log-sum-exp rule.  No second kernel.
//
// Warp roles (352 threads): 0 K/V TMA producer, 1 MMA issuer, 2-5 softmax
// (thread <-> tile row), 6-9 epilogue (thread <-> head-dim row): reads O^T from
// TMEM at the end of each segment, normalises and stores, or writes a part and
// merges; 10 query loader (one buffer, refilled per sequence once the last
// score MMA of the previous one is done; the next sequence's rows are
// prefetched into L2 meanwhile).  O is double-buffered in TMEM by segment, so
// the epilogue of one sequence overlaps the next.
#include "decode.cuh"
#include "sm100.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>

namespace pk {
namespace {

using namespace sm100;

constexpr int kHkv = 8;                     // KV heads per tile
constexpr int kTok = 16;                    // tokens per tile
constexpr int kRows = kHkv * kTok;          // 128 = MMA M
constexpr int kStages = 3;
constexpr int kThreads = 352;
constexpr uint32_t kChunk = kRows * 128;    // 16 KiB: 128 rows x 64 bf16
constexpr uint32_t kKOff = 0;
constexpr uint32_t kVOff = 2 * kChunk;
constexpr uint32_t kStageBytes = 4 * kChunk;
constexpr int kMaxH = 64;                   // query heads per sequence (G <= 8)
constexpr uint32_t kQChunk = kMaxH * 128;
constexpr uint32_t kQBytes = 2 * kQChunk;
constexpr uint32_t kPHead = 512;            // one head's P^T: 16 tokens x 16 columns, bf16
constexpr uint32_t kPBytes = kHkv * kPHead;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;              // 2 buffers x NQ (<= 64) columns
constexpr uint32_t kTmemO = 128;            // 2 buffers x 128 columns (8 heads x 16)
constexpr float kRescaleLog2 = 8.0f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kMaxCtas = 1024;

struct Misc {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t q_full, q_empty;
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t pv_done[2];
    uint64_t seg_o[2];
    uint64_t seg_l[2];
    uint64_t o_free[2];
    uint64_t drain;
    int64_t scan[kThreads];
    int64_t total;
    int64_t rem_beg, rem_last;
    int32_t s_beg, s_last;
    uint32_t tmem_base;
    int abort;
    int never;
    int merge_flag;
    int vlen[kStages];
    float alpha[kMaxH];
    float seg_m[2][kMaxH];
    float seg_l_val[2][kMaxH];
};
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + kQBytes + 2 * kPBytes + sizeof(Misc);

struct Slot {
    int32_t s, pad;
    int64_t start, nt;
    int64_t pad2[5];
    float m[kMaxH];
    float l[kMaxH];
    float o[kMaxH * 128];
};

__device__ __forceinline__ int clamp_len(const DecodeParams &p, int s, int cap) {
    const int raw = p.seq_lens[s];
    return raw < 0 ? 0 : (raw > cap ? cap : raw);
}

struct Walk {
    int s, t, nt, L;
    __device__ __forceinline__ void load(const DecodeParams &p, int cap) {
        L = clamp_len(p, s, cap);
        nt = (L + kTok - 1) / kTok;
    }
    __device__ __forceinline__ void next(const DecodeParams &p, int cap) {
        if (++t < nt) return;
        t = 0;
        do {
            if (++s >= p.num_seqs) return;
            load(p, cap);
        } while (nt == 0);
    }
};

__device__ __forceinline__ int64_t range_begin(int64_t c, int64_t T, int64_t C) { return c * T / C; }
__device__ __forceinline__ int cta_of(int64_t idx, int64_t T, int C) {
    int c = static_cast<int>(idx * C / T);
    while (c + 1 < C && range_begin(c + 1, T, C) <= idx) ++c;
    return c;
}

__device__ __forceinline__ void store_out(const DecodeParams &p, size_t idx, float v) {
    if (p.out_fp32) static_cast<float *>(p.out)[idx] = v;
    else static_cast<uint16_t *>(p.out)[idx] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}

// The CTA's tiles in processing order: first [S_last, end) (its last
// segment), then [beg, S_last).  Every role walks the same sequence.
struct Order {
    int n, n_a;
    int64_t beg, s_last_start;       // global index of the first tile of each sub-range
    int s_a, t_a, s_b, t_b;
    __device__ __forceinline__ int64_t global(int i) const {
        return i < n_a ? s_last_start + i : beg + (i - n_a);
    }
    __device__ __forceinline__ void start(Walk &w, int i, const DecodeParams &p, int cap) const {
        w.s = i == 0 ? s_a : s_b;
        w.load(p, cap);
        w.t = i == 0 ? t_a : t_b;
    }
};

template <int G>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[G < 2 ? 2 : G]) {
    tmem_ld<(G < 2 ? 2 : G)>(taddr, v);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
decode_hb_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group");
    constexpr int NCH = D / 64;
    constexpr int H = kHkv * G;
    constexpr int NQ = H < 16 ? 16 : H;                 // MMA N of the score product
    constexpr int GL = G < 2 ? 2 : G;                   // TMEM load width per head
    constexpr uint32_t kIdescQK = idesc_bf16(kRows, NQ, 0, 0);
    constexpr uint32_t kIdescPV = idesc_bf16(128, 16, 1, 1);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *stage_ptr = smem;
    uint8_t *q_ptr = smem + kStages * kStageBytes;
    uint8_t *p_ptr = q_ptr + kQBytes;
    Misc *misc = reinterpret_cast<Misc *>(p_ptr + 2 * kPBytes);
    const uint32_t stage_addr = smem_u32(stage_ptr);
    const uint32_t q_addr = smem_u32(q_ptr);
    const uint32_t p_addr = smem_u32(p_ptr);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, C = gridDim.x;
    const int N = p.num_seqs, B = p.block_size;
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * B);
    Slot *slots = static_cast<Slot *>(p.tc_slots);
    unsigned long long *tickets =
        slots ? reinterpret_cast<unsigned long long *>(slots + 2 * kMaxCtas) : nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&misc->full[i]), 1);
            mbar_init(smem_u32(&misc->empty[i]), 1);
        }
        mbar_init(smem_u32(&misc->q_full), 1);
        mbar_init(smem_u32(&misc->q_empty), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&misc->s_full[i]), 1);
            mbar_init(smem_u32(&misc->p_full[i]), 4);
            mbar_init(smem_u32(&misc->pv_done[i]), 1);
            mbar_init(smem_u32(&misc->seg_o[i]), 1);
            mbar_init(smem_u32(&misc->seg_l[i]), 4);
            mbar_init(smem_u32(&misc->o_free[i]), 4);
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
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
    }
    // P^T buffers: the padded columns (and padded query heads) stay zero.
    for (uint32_t i = threadIdx.x; i < 2 * kPBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(p_ptr)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();

    // ---- range of the flattened (sequence, tile) space ---------------------
    const int per = (N + kThreads - 1) / kThreads;
    const int s_lo = min(N, static_cast<int>(threadIdx.x) * per), s_hi = min(N, s_lo + per);
    int64_t mine = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        const int raw = p.seq_lens[s];
        if ((raw < 0 || raw > cap) && s % C == c) set_error(p.err, PK_DEVERR_SEQ_LEN);
        const int L = raw < 0 ? 0 : (raw > cap ? cap : raw);
        mine += (L + kTok - 1) / kTok;
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
        const int64_t acc0 = misc->scan[threadIdx.x];
        // Sequence and offset of tile `beg` and of tile `end - 1`.
        for (int which = 0; which < 2; ++which) {
            const int64_t target = which == 0 ? beg : end - 1;
            if (acc0 <= target && target < acc0 + mine) {
                int64_t acc = acc0;
                for (int s = s_lo; s < s_hi; ++s) {
                    const int64_t nt = (clamp_len(p, s, cap) + kTok - 1) / kTok;
                    if (target < acc + nt) {
                        if (which == 0) {
                            misc->s_beg = s;
                            misc->rem_beg = target - acc;
                        } else {
                            misc->s_last = s;
                            misc->rem_last = target - acc;
                        }
                        break;
                    }
                    acc += nt;
                }
            }
        }
    }
    for (int s = c; s < N; s += C) {
        if (clamp_len(p, s, cap) != 0) continue;
        for (int i = threadIdx.x; i < H * D; i += kThreads) store_out(p, static_cast<size_t>(s) * H * D + i, 0.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;

    Order ord{};
    ord.n = n_tiles;
    ord.beg = beg;
    if (n_tiles > 0) {
        const int64_t last_seg_start = (end - 1) - misc->rem_last;      // global index of its tile 0
        ord.s_last_start = last_seg_start > beg ? last_seg_start : beg;
        ord.n_a = static_cast<int>(end - ord.s_last_start);
        ord.s_a = misc->s_last;
        ord.t_a = static_cast<int>(ord.s_last_start - last_seg_start);
        ord.s_b = misc->s_beg;
        ord.t_b = static_cast<int>(misc->rem_beg);
    }

    if (warp == 0) {
        // ================= producer =================
        // Block-table entries are read kLook tiles ahead (a register ring,
        // fully unrolled so it stays in registers), so their latency overlaps
        // the streaming of earlier tiles instead of preceding each TMA.
        if (lane == 0) {
            constexpr int kLook = 8;
            const int MB = p.max_blocks_per_seq;
            auto entry = [&](const Walk &x) {
                return p.block_tables[static_cast<size_t>(x.s) * MB + (x.t * kTok) / B];
            };
            auto step = [&](Walk &x, int &idx) {
                ++idx;
                if (idx == ord.n_a) ord.start(x, idx, p, cap);
                else x.next(p, cap);
            };
            Walk w{}, wa{};
            int ia = 0;
            int ring[kLook];
            if (n_tiles > 0) ord.start(wa, 0, p, cap);
#pragma unroll
            for (int k = 0; k < kLook; ++k) {
                if (ia < n_tiles) {
                    ring[k] = entry(wa);
                    step(wa, ia);
                }
            }
            int issued = 0;
            bool stop = false;
            for (int base = 0; base < n_tiles && !stop; base += kLook) {
#pragma unroll
                for (int k = 0; k < kLook; ++k) {
                    const int i = base + k;
                    if (i >= n_tiles) break;
                    if (i == 0 || i == ord.n_a) ord.start(w, i, p, cap);
                    const int phys = ring[k];
                    if (ia < n_tiles) {                        // tile i + kLook
                        ring[k] = entry(wa);
                        step(wa, ia);
                    }
                    const int st = i % kStages;
                    if (!mbar_wait(smem_u32(&misc->empty[st]), ((i / kStages) & 1) ^ 1, &misc->abort, kWaitLimitNs)) {
                        misc->abort = 1;
                        set_error(p.err, PK_DEVERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                    const int tok0 = w.t * kTok;
                    const int vlen = min(kTok, w.L - tok0);
                    const bool ok = phys >= 0 && phys < p.num_blocks;
                    if (!ok) set_error(p.err, PK_DEVERR_BLOCK_ID);
                    misc->vlen[st] = ok ? vlen : 0;
                    const uint32_t full = smem_u32(&misc->full[st]);
                    const uint32_t sbase = stage_addr + st * kStageBytes;
                    mbar_arrive_expect_tx(full, ok ? 2u * NCH * kChunk : 0u);
                    if (ok) {
#pragma unroll
                        for (int ch = 0; ch < NCH; ++ch) {
                            tma_load_4d(sbase + kKOff + ch * kChunk, &tm_k, full, ch * 64, tok0 % B, 0, phys);
                            tma_load_4d(sbase + kVOff + ch * kChunk, &tm_v, full, ch * 64, tok0 % B, 0, phys);
                        }
                    }
                    ++issued;
                    w.next(p, cap);
                }
            }
            if (misc->abort) {
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(smem_u32(&misc->full[i % kStages]), (i / kStages) & 1, &misc->never, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            bool alive = true;
            auto fail = [&]() {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                alive = false;
            };
            auto pv = [&](int j, int sg, bool first, bool last) {
                if (!mbar_wait(smem_u32(&misc->p_full[j & 1]), (j >> 1) & 1, &misc->abort, kWaitLimitNs)) return fail();
                const int ob = sg & 1;
                if (first && !mbar_wait(smem_u32(&misc->o_free[ob]), ((sg >> 1) & 1) ^ 1, &misc->abort, kWaitLimitNs))
                    return fail();
                tc_fence_after();
                const uint32_t vbase = stage_addr + (j % kStages) * kStageBytes + kVOff;
                const uint32_t pbase = p_addr + (j & 1) * kPBytes;
#pragma unroll
                for (int hh = 0; hh < kHkv; ++hh) {
                    const uint64_t a = smem_desc(vbase + hh * kTok * 128, kChunk, 1024, kLayoutSw128);
                    const uint64_t b = smem_desc(pbase + hh * kPHead, 256, 128, kLayoutNone);
                    mma_bf16(tmem + kTmemO + ob * 128 + hh * 16, a, b, kIdescPV, first ? 0u : 1u);
                }
                mma_commit(smem_u32(&misc->pv_done[j & 1]));
                mma_commit(smem_u32(&misc->empty[j % kStages]));
                if (last) mma_commit(smem_u32(&misc->seg_o[ob]));
            };
            Walk w{};
            int seg = -1;
            int prev_seg = 0;
            bool prev_first = false, prev_last = false, pending = false;
            for (int i = 0; i < n_tiles && alive; ++i) {
                if (i == 0 || i == ord.n_a) ord.start(w, i, p, cap);
                const bool seg_first = i == 0 || i == ord.n_a || w.t == 0;
                const bool seg_last = i == ord.n_a - 1 || i == n_tiles - 1 || w.t == w.nt - 1;
                if (seg_first) {
                    // The previous tile's P.V does not need the new query rows.
                    if (pending) {
                        pv(i - 1, prev_seg, prev_first, prev_last);
                        pending = false;
                        if (!alive) break;
                    }
                    ++seg;
                    if (!mbar_wait(smem_u32(&misc->q_full), seg & 1, &misc->abort, kWaitLimitNs)) {
                        fail();
                        break;
                    }
                }
                const int st = i % kStages;
                if (!mbar_wait(smem_u32(&misc->full[st]), (i / kStages) & 1, &misc->abort, kWaitLimitNs)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t sbase = stage_addr + st * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * kQChunk + (kk & 3) * 32;
                    const uint64_t a = smem_desc(sbase + kKOff + off, 16, 1024, kLayoutSw128);
                    const uint64_t b = smem_desc(q_addr + qoff, 16, 1024, kLayoutSw128);
                    mma_bf16(tmem + kTmemS + (i & 1) * NQ, a, b, kIdescQK, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&misc->s_full[i & 1]));
                if (seg_last) mma_commit(smem_u32(&misc->q_empty));
                if (pending) pv(i - 1, prev_seg, prev_first, prev_last);
                pending = true;
                prev_seg = seg;
                prev_first = seg_first;
                prev_last = seg_last;
                w.next(p, cap);
            }
            if (alive && pending) pv(n_tiles - 1, prev_seg, prev_first, prev_last);
            mma_commit(smem_u32(&misc->drain));
            mbar_wait(smem_u32(&misc->drain), 0, &misc->never, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ================= softmax (warps 2-5): thread <-> tile row =================
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int h = r >> 4, t = r & 15;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        float m_ref[G], l_run[G];
        Walk w{};
        int seg = -1;
        for (int i = 0; i < n_tiles; ++i) {
            if (i == 0 || i == ord.n_a) ord.start(w, i, p, cap);
            const bool seg_first = i == 0 || i == ord.n_a || w.t == 0;
            const bool seg_last = i == ord.n_a - 1 || i == n_tiles - 1 || w.t == w.nt - 1;
            if (seg_first) {
                ++seg;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    m_ref[g] = -INFINITY;
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
            // The stage's phase for this tile is complete; waiting on it makes
            // the producer's per-stage length visible here.
            mbar_wait(smem_u32(&misc->full[st]), (i / kStages) & 1, &misc->never, kWaitLimitNs);
            tc_fence_after();
            float sv[2 * G < 2 ? 2 : 2 * G];
            tmem_ld<(2 * G < 2 ? 2 : 2 * G)>(lane_addr + kTmemS + sb * NQ + 2 * quad * G, sv);
            const bool valid = t < misc->vlen[st];
            float s2[G];
            bool need = false;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float raw = (h & 1) ? sv[G + g] : sv[g];     // this row's group of columns
                s2[g] = valid ? raw * p.scale_log2 : -INFINITY;
                need |= s2[g] > m_ref[g] + kRescaleLog2;
            }
            if (named_bar_or(1, 128, need)) {
                // Rare: move the reference max of the heads that need it.
                const uint32_t votes = __ballot_sync(0xffffffffu, need);
                const bool head_needs = ((votes >> (lane & 16)) & 0xffffu) != 0;
                float a[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float mx = s2[g];
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    const float mn = head_needs ? fmaxf(m_ref[g], mx) : m_ref[g];
                    a[g] = m_ref[g] == -INFINITY ? 0.f : fast_exp2(m_ref[g] - mn);
                    l_run[g] *= a[g];
                    m_ref[g] = mn;
                }
                if (t == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g) misc->alpha[h * G + g] = a[g];
                }
                named_bar_sync(1, 128);
                if (!seg_first) {
                    // O so far (through tile i-1) is rescaled in TMEM: thread r
                    // acts on TMEM lane r (head-dim row r of O^T).
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[(i - 1) & 1]), ((i - 1) >> 1) & 1,
                                                           &misc->never, kWaitLimitNs))) {
                        misc->abort = 1;
                        set_error(p.err, PK_DEVERR_TIMEOUT);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t obase = lane_addr + kTmemO + (seg & 1) * 128;
#pragma unroll 1
                    for (int hh = 0; hh < kHkv; ++hh) {
                        bool moved = false;
#pragma unroll
                        for (int g = 0; g < G; ++g) moved |= misc->alpha[hh * G + g] != 1.f;
                        if (!moved) continue;                  // same for every thread
                        float ov[8];
                        tmem_ld<8>(obase + hh * 16, ov);
#pragma unroll
                        for (int g = 0; g < G; ++g) ov[g] *= misc->alpha[hh * G + g];
                        tmem_st8(obase + hh * 16, ov);
                    }
                }
            }
            float pr[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) pr[g] = 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) pr[g] = valid ? fast_exp2(s2[g] - m_ref[g]) : 0.f;
            uint32_t packed[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) packed[k] = pack_bf16x2(pr[2 * k], pr[2 * k + 1]);
#pragma unroll
            for (int g = 0; g < G; ++g)
                l_run[g] += (g & 1) ? bf16_hi(packed[g >> 1]) : bf16_lo(packed[g >> 1]);
            // P buffer sb is free once PV(i-2) has finished.
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[sb]), ((i >> 1) & 1) ^ 1, &misc->never,
                                                   kWaitLimitNs))) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
            if (!valid) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(stage_ptr + st * kStageBytes + kVOff + ch * kChunk + r * 128);
#pragma unroll
                    for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0, 0, 0, 0);
                }
            }
            *reinterpret_cast<uint4 *>(p_ptr + sb * kPBytes + h * kPHead + (t >> 3) * 256 + (t & 7) * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&misc->p_full[sb]));

            if (seg_last) {
                float lsum[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = l_run[g];
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    lsum[g] = v;
                }
                const int b = seg & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->o_free[b]), ((seg >> 1) & 1) ^ 1, &misc->never,
                                                       kWaitLimitNs))) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                    break;
                }
                if (t == 0) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        misc->seg_l_val[b][h * G + g] = lsum[g];
                        misc->seg_m[b][h * G + g] = m_ref[g];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&misc->seg_l[b]));
            }
            w.next(p, cap);
        }
        tc_fence_before();
    } else if (warp < 10) {
        // ================= epilogue (warps 6-9): thread <-> head-dim row =================
        const int quad = warp & 3;
        const int d = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        Walk w{};
        int seg = -1;
        int seg_t0 = 0;
        int64_t seg_gstart = 0;
        for (int i = 0; i < n_tiles; ++i) {
            if (i == 0 || i == ord.n_a) ord.start(w, i, p, cap);
            const bool seg_first = i == 0 || i == ord.n_a || w.t == 0;
            const bool seg_last = i == ord.n_a - 1 || i == n_tiles - 1 || w.t == w.nt - 1;
            if (seg_first) {
                ++seg;
                seg_t0 = w.t;
                seg_gstart = ord.global(i) - w.t;
            }
            if (seg_last) {
                const int b = seg & 1;
                const bool got = mbar_wait(smem_u32(&misc->seg_o[b]), (seg >> 1) & 1, &misc->never, kWaitLimitNs) &&
                                 mbar_wait(smem_u32(&misc->seg_l[b]), (seg >> 1) & 1, &misc->never, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got)) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const bool complete = seg_t0 == 0 && w.t == w.nt - 1;
                float res[kHkv][GL];
#pragma unroll
                for (int hh = 0; hh < kHkv; ++hh) ld_cols<G>(lane_addr + kTmemO + b * 128 + hh * 16, res[hh]);
                float mcopy = 0.f, lcopy = 0.f;
                if (complete) {
#pragma unroll
                    for (int hh = 0; hh < kHkv; ++hh)
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float l = misc->seg_l_val[b][hh * G + g];
                            res[hh][g] = l > 0.f ? res[hh][g] / l : 0.f;
                        }
                } else if (d < H) {
                    mcopy = misc->seg_m[b][d];
                    lcopy = misc->seg_l_val[b][d];
                }
                // TMEM buffer b and the per-segment values are no longer needed.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&misc->o_free[b]));
                const int s = w.s;
                if (complete) {
                    if (d < D) {
#pragma unroll
                        for (int hh = 0; hh < kHkv; ++hh)
#pragma unroll
                            for (int g = 0; g < G; ++g)
                                store_out(p, (static_cast<size_t>(s) * H + hh * G + g) * D + d, res[hh][g]);
                    }
                } else {
                    // A cut segment: write this part, then the last part to
                    // finish merges all of them.
                    const int slot_idx = beg >= seg_gstart ? 0 : 1;
                    Slot *sl = slots + 2 * c + slot_idx;
                    if (d < D) {
#pragma unroll
                        for (int hh = 0; hh < kHkv; ++hh)
#pragma unroll
                            for (int g = 0; g < G; ++g) sl->o[(hh * G + g) * D + d] = res[hh][g];
                    }
                    if (d < H) {
                        sl->m[d] = mcopy;
                        sl->l[d] = lcopy;
                    }
                    __threadfence();
                    named_bar_sync(2, 128);
                    if (d == 0) {
                        const int64_t seg_end = seg_gstart + w.nt;           // one past its last tile
                        const int ca = cta_of(seg_gstart, T, C), cb = cta_of(seg_end - 1, T, C);
                        unsigned parts = 0;
                        for (int cc = ca; cc <= cb; ++cc)
                            parts += range_begin(cc, T, C) < range_begin(cc + 1, T, C) ? 1u : 0u;
                        const unsigned long long ep = static_cast<unsigned long long>(p.epoch) << 32;
                        unsigned long long cur = 0;
                        unsigned mine_count = 0;
                        for (int tries = 0; tries < 4096; ++tries) {
                            const unsigned long long assumed = cur;
                            const unsigned cnt = (assumed >> 32) == p.epoch ? static_cast<unsigned>(assumed) : 0u;
                            cur = atomicCAS(tickets + ca, assumed, ep | (cnt + 1u));
                            if (cur == assumed) {
                                mine_count = cnt + 1u;
                                break;
                            }
                        }
                        if (mine_count == 0) set_error(p.err, PK_DEVERR_TIMEOUT);
                        misc->merge_flag = (mine_count == parts) ? 1 : 0;
                    }
                    named_bar_sync(2, 128);
                    if (misc->merge_flag) {
                        __threadfence();
                        const int64_t seg_end = seg_gstart + w.nt;
                        const int ca = cta_of(seg_gstart, T, C), cb = cta_of(seg_end - 1, T, C);
#pragma unroll 1
                        for (int n0 = 0; n0 < H; n0 += G) {
                            float M[G], num[G], den[G];
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                M[g] = -INFINITY;
                                num[g] = den[g] = 0.f;
                            }
                            for (int cc = ca; cc <= cb; ++cc) {
                                if (range_begin(cc, T, C) == range_begin(cc + 1, T, C)) continue;
                                const Slot *ps = slots + 2 * cc + (range_begin(cc, T, C) >= seg_gstart ? 0 : 1);
#pragma unroll
                                for (int g = 0; g < G; ++g) M[g] = fmaxf(M[g], __ldcg(&ps->m[n0 + g]));
                            }
                            for (int cc = ca; cc <= cb; ++cc) {
                                if (range_begin(cc, T, C) == range_begin(cc + 1, T, C)) continue;
                                const Slot *ps = slots + 2 * cc + (range_begin(cc, T, C) >= seg_gstart ? 0 : 1);
#pragma unroll
                                for (int g = 0; g < G; ++g) {
                                    const float a = rescale(__ldcg(&ps->m[n0 + g]), M[g]);
                                    den[g] = fmaf(a, __ldcg(&ps->l[n0 + g]), den[g]);
                                    if (d < D) num[g] = fmaf(a, __ldcg(&ps->o[(n0 + g) * D + d]), num[g]);
                                }
                            }
                            if (d < D) {
#pragma unroll
                                for (int g = 0; g < G; ++g)
                                    store_out(p, (static_cast<size_t>(s) * H + n0 + g) * D + d,
                                              den[g] > 0.f ? num[g] / den[g] : 0.f);
                            }
                        }
                    }
                }
            }
            w.next(p, cap);
        }
        tc_fence_before();
    }
    if (warp == 10 && lane == 0) {
        // ================= query loader =================
        Walk w{};
        int seg = -1;
        for (int i = 0; i < n_tiles; ++i) {
            if (i == 0 || i == ord.n_a) ord.start(w, i, p, cap);
            if (i == 0 || i == ord.n_a || w.t == 0) {
                ++seg;
                if (!mbar_wait(smem_u32(&misc->q_empty), (seg & 1) ^ 1, &misc->abort, kWaitLimitNs)) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                    break;
                }
                const uint32_t qf = smem_u32(&misc->q_full);
                mbar_arrive_expect_tx(qf, NCH * NQ * 128u);
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) tma_load_2d(q_addr + ch * kQChunk, &tm_q, qf, ch * 64, w.s * H);
                if (w.s + 1 < N) prefetch_l2(p.q + static_cast<size_t>(w.s + 1) * H * D, H * D * 2);
                if (i == 0 && ord.n_a < n_tiles) prefetch_l2(p.q + static_cast<size_t>(ord.s_b) * H * D, H * D * 2);
            }
            w.next(p, cap);
        }
        if (misc->abort) mbar_wait(smem_u32(&misc->q_full), seg & 1, &misc->never, kWaitLimitNs);
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Cache viewed as (d, token, head, block) so that one box of
// (64, 16 tokens, 8 heads) lands head-major: row = head * 16 + token.
bool encode_cache(CUtensorMap *m, const void *base, const DecodeParams &p) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t D = p.head_dim, Hkv = p.num_kv_heads, B = p.block_size;
    const cuuint64_t P = p.num_blocks > 0 ? p.num_blocks : 1;
    cuuint64_t dims[4] = {D, B, Hkv, P};
    cuuint64_t strides[3] = {Hkv * D * 2, D * 2, B * Hkv * D * 2};
    cuuint32_t box[4] = {64, kTok, kHkv, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q(CUtensorMap *m, const DecodeParams &p, int nq) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.head_dim), static_cast<cuuint64_t>(p.num_seqs) * p.num_heads};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.head_dim) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(nq)};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p.q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_dg(const DecodeParams &p, int C, cudaStream_t stream) {
    constexpr int H = kHkv * G;
    CUtensorMap mk, mv, mq;
    if (!encode_cache(&mk, p.k_cache, p) || !encode_cache(&mv, p.v_cache, p) || !encode_q(&mq, p, H < 16 ? 16 : H))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_hb_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    decode_hb_kernel<D, G><<<C, kThreads, kSmemBytes, stream>>>(mk, mv, mq, p);
    return cudaGetLastError();
}

std::atomic<uint32_t> g_epoch{0};

}  // namespace

bool hb_supported(int num_heads, int num_kv_heads, int head_dim, int block_size) {
    if (num_kv_heads != kHkv || num_heads % num_kv_heads) return false;
    const int G = num_heads / num_kv_heads;
    return (G == 1 || G == 2 || G == 4 || G == 8) && (head_dim == 64 || head_dim == 128) &&
           (block_size == 16 || block_size == 32);
}

size_t hb_workspace_bytes() { return 2 * kMaxCtas * sizeof(Slot) + kMaxCtas * sizeof(unsigned long long); }

uint32_t next_epoch() {
    uint32_t e = g_epoch.load();
    if (e == 0) {
        // Start from a value that differs between processes, so that stale
        // tickets left in reused memory never match.
        const uint32_t seed = static_cast<uint32_t>(
            std::chrono::steady_clock::now().time_since_epoch().count() * 2654435761u) | 1u;
        uint32_t zero = 0;
        g_epoch.compare_exchange_strong(zero, seed);
    }
    for (;;) {
        e = g_epoch.fetch_add(1);
        if (e != 0) return e;
    }
}

cudaError_t launch_decode_head_batched(const DecodeParams &p, cudaStream_t stream) {
    int C = sm_count();
    if (C <= 0) return cudaErrorNoDevice;
    if (C > kMaxCtas) C = kMaxCtas;
    DecodeParams q = p;
    q.epoch = next_epoch();
    const int G = p.num_heads / p.num_kv_heads;
    if (p.head_dim == 64) {
        switch (G) {
            case 1: return launch_dg<64, 1>(q, C, stream);
            case 2: return launch_dg<64, 2>(q, C, stream);
            case 4: return launch_dg<64, 4>(q, C, stream);
            case 8: return launch_dg<64, 8>(q, C, stream);
        }
    } else {
        switch (G) {
            case 1: return launch_dg<128, 1>(q, C, stream);
            case 2: return launch_dg<128, 2>(q, C, stream);
            case 4: return launch_dg<128, 4>(q, C, stream);
            case 8: return launch_dg<128, 8>(q, C, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pk
