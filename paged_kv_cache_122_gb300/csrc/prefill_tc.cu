// Multi-query paged attention for WIDE query blocks (chunked prefill): many
// newest tokens of a sequence attend its paged cache, causal among
// themselves ("PagedAttention from First Principles", §12 chunked prefill:
// a chunk of a prompt is processed over the cache in one pass; the
// attention itself is the decode definition of "vLLM — PagedAttention",
// Mathematical Formulation, Equation 4, with the causal limit).
//
// Orientation.  The decode kernel puts keys on the MMA's M and at most 16
// query columns on N.  Here the queries are the dense side: a query tile is
// 128 rows -- 128 / G consecutive query tokens x the G query heads of one
// KV head, row = token * G + head -- and the sequence's keys stream by in
// 128-key tiles:
//   S[128 x 128]  = Q[128 x D] K_tile^T          (tcgen05, fp32 in TMEM)
//   O[128 x D]   += P[128 x 128] V_tile[128 x D]  (tcgen05, fp32 in TMEM)
// so one softmax thread owns one query row of S, P and O and needs no
// cross-thread reduction.
//
// A CTA holds TWO query tiles, X = 0 and X = 1 (consecutive token blocks of
// the same sequence and KV head), which share every K and V tile: each
// page is fetched once per 256 query rows.  The two tiles' softmax warp
// groups alternate with the tensor core (while one group turns its S into
// P, the MMAs of the other tile run).  Tensor memory (512 columns) holds
// S_0, S_1, O_0, O_1; the bf16 P of a tile is written over the first 64
// columns of its own S (two keys per column), which the P.V MMA reads as
// its A operand; the next S of that tile is issued after that P.V, and
// tcgen05 MMAs of one thread execute in issue order.
//
// Per CTA (352 threads):
//   warp 0     producer: both Q tiles once, then per key tile the K rows
//              of each page (one box: 8-row blocks [half][8 rows][64])
//              into a K ring;
//   warp 10    producer: per key tile the V rows of each page (one box,
//              likewise) into a V ring;
//   warp 1     MMA issuer (one thread): per key tile i, P.V(i-1) then S(i)
//              for tile 0, then the same for tile 1;
//   warps 2-5  softmax of tile 0, warps 6-9 softmax of tile 1: row max
//              against a reference max that moves only when exceeded by
//              more than 2^8 (then the row's O and denominator are
//              rescaled), p = 2^(s - m_ref) with the causal and validity
//              masks, bf16 P into tensor memory, and at the end O / l
//              written out (a TMA store of the tile when it is full).
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

constexpr int kRows = 128;                      // query rows per tile = MMA M
constexpr int kKeys = 128;                      // keys per tile = MMA N of S
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kMaskRing = 4;                    // tile masks in flight (the K producer runs <= 3 tiles ahead)
constexpr int kThreads = 352;
constexpr uint32_t kChunk = 128 * 128;          // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kQBytes = 2 * kChunk;        // one query tile (D <= 128)
constexpr uint32_t kKBytes = 2 * kChunk;        // K of one key tile
constexpr uint32_t kVBytes = 2 * kChunk;        // V of one key tile
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = 2 * kQBytes;
constexpr uint32_t kVOff = kKOff + kKStages * kKBytes;
constexpr uint32_t kTmemCols = 512;             // S_0, S_1, O_0, O_1 (128 columns each)
constexpr uint32_t kTmemS = 0;                  // + X * 128; P_X over its first 64 columns
constexpr uint32_t kTmemO = 256;                // + X * 128
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kRescaleLog2 = 8.0f;

struct Misc {
    uint64_t kfull[kKStages];   // K rows of a tile landed
    uint64_t kempty[kKStages];  // both S of the tile done: K slot free
    uint64_t vfull[kVStages];   // V rows of a tile landed
    uint64_t vempty[kVStages];  // both P.V of the tile done: V slot free
    uint64_t q_full;
    uint64_t s_full[2];         // S of query tile X in TMEM
    uint64_t p_full[2];         // P of query tile X written (4 softmax warps)
    uint64_t pv_done[2];        // P.V of query tile X done
    uint64_t go;                // tile 0's group has finished key tile 0 (4 warps)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int never;
    uint32_t mask[kMaskRing][4];  // valid keys of a key tile (by tile index mod 4)
};

constexpr size_t kSmemBytes = 1024 + kVOff + kVStages * kVBytes + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void group_bar(uint32_t id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// Three-input max / min (NaN inputs are skipped, as by fmaxf / fminf).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// grid: one CTA per (sequence, KV head, pair of query tiles of 128 / G
// tokens each), blockIdx.x = (s * Hkv + h) * qblocks + j; CTAs past a
// sequence's queries exit.  tm_o (bf16 output only, o_tma != 0) stores
// full query tiles.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                  const DecodeParams p, int qblocks, int o_tma) {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= 16 && (G & (G - 1)) == 0, "group");
    constexpr int NCH = D / 64;
    constexpr int QT = kRows / G;                 // query tokens per tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = p.num_kv_heads, H = p.num_heads, B = p.block_size;
    const int j = blockIdx.x % qblocks;
    const int h = (blockIdx.x / qblocks) % Hkv;
    const int s = blockIdx.x / qblocks / Hkv;
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * B);
    // K and V of a key tile in shared memory: each page in one TMA box as
    // B / 8 blocks of 8 rows, each block [half][8 rows][64] -- so the 8-row
    // swizzle atoms of one 64-element half lie kAtomStride bytes apart
    // whatever the block size.
    constexpr uint32_t kAtomStride = 1024u * NCH;
    int L = p.seq_lens[s];
    const int q0 = p.cu_q_lens[s];
    const int qn = p.cu_q_lens[s + 1] - q0;
    if (L < 0 || L > cap || qn < 0 || qn > max(L, 0)) {
        if (j == 0 && h == 0 && threadIdx.x == 0) set_error(p.err, PK_DEVERR_SEQ_LEN);
        return;
    }
    const int qt0 = j * 2 * QT;                   // first query token of tile 0
    if (qt0 >= qn) return;
    const int pos0 = L - qn;                      // position of the sequence's first query
    // Key tiles each query tile needs (the last key it sees is that of its
    // last token); tile 1 may be empty.
    const int n0 = (pos0 + min(qn, qt0 + QT) - 1) / kKeys + 1;
    const int n1 = qt0 + QT < qn ? (pos0 + min(qn, qt0 + 2 * QT) - 1) / kKeys + 1 : 0;
    const int nT = max(n0, n1);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Misc *misc = reinterpret_cast<Misc *>(smem + kVOff + kVStages * kVBytes);
    const uint32_t base = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(smem_u32(&misc->kfull[i]), 1);
            mbar_init(smem_u32(&misc->kempty[i]), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(smem_u32(&misc->vfull[i]), 1);
            mbar_init(smem_u32(&misc->vempty[i]), 1);
        }
        mbar_init(smem_u32(&misc->q_full), 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&misc->s_full[x]), 1);
            mbar_init(smem_u32(&misc->p_full[x]), 4);
            mbar_init(smem_u32(&misc->pv_done[x]), 1);
        }
        mbar_init(smem_u32(&misc->go), 4);
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

    if (warp == 0 || warp == 10) {
        // ================= producers: warp 0 the queries and K, warp 10 V =================
        // (Two warps, so that the copies of K and of V are issued side by side.)
        const bool kprod = warp == 0;
        const int MB = p.max_blocks_per_seq;
        if (kprod && lane == 0) {
            prefetch_tmap(&tm_k);
            const uint32_t qf = smem_u32(&misc->q_full);
            const int tiles = n1 > 0 ? 2 : 1;
            mbar_arrive_expect_tx(qf, tiles * kRows * 128u * NCH);
            for (int x = 0; x < tiles; ++x) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    tma_load_3d(base + kQOff + x * kQBytes + ch * kChunk, &tm_q, qf, ch * 64, h * G,
                                q0 + qt0 + x * QT);
            }
        }
        if (!kprod && lane == 0) prefetch_tmap(&tm_v);
        // Block-table entries of a key tile, one page per lane; the next
        // tile's are fetched while the current tile's copies are issued.
        auto fetch = [&](int t) -> int {
            const int tok = t * kKeys;
            const int pg = (min(kKeys, L - tok) + B - 1) / B;
            return lane < pg ? p.block_tables[static_cast<size_t>(s) * MB + tok / B + lane] : -1;
        };
        const int nstages = kprod ? kKStages : kVStages;
        int phys_next = fetch(0);
        int issued = 0;
        for (int i = 0; i < nT; ++i) {
            const int st = i % nstages;
            const int phys_raw = phys_next;
            int got = 1;
            if (lane == 0)
                got = mbar_wait(smem_u32(kprod ? &misc->kempty[st] : &misc->vempty[st]), ((i / nstages) & 1) ^ 1,
                                &misc->abort, kWaitLimitNs);
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
                if (!ok && kprod) set_error(p.err, PK_DEVERR_BLOCK_ID);
            }
            const uint32_t nok = __popc(__ballot_sync(0xffffffffu, ok));
            const int r0 = lane * B;
            if (kprod) {
                uint32_t bits = 0;
                if (ok) {
                    const int nrows = min(B, vlen - r0);
                    bits = (nrows >= 32 ? 0xffffffffu : ((1u << nrows) - 1u)) << (r0 & 31);
                }
                const int word = r0 >> 5;
                const uint32_t m0 = __reduce_or_sync(0xffffffffu, word == 0 ? bits : 0u);
                const uint32_t m1 = __reduce_or_sync(0xffffffffu, word == 1 ? bits : 0u);
                const uint32_t m2 = __reduce_or_sync(0xffffffffu, word == 2 ? bits : 0u);
                const uint32_t m3 = __reduce_or_sync(0xffffffffu, word == 3 ? bits : 0u);
                const uint32_t kfull = smem_u32(&misc->kfull[st]);
                if (lane == 0) {
                    uint32_t *mk = misc->mask[i % kMaskRing];
                    mk[0] = m0;
                    mk[1] = m1;
                    mk[2] = m2;
                    mk[3] = m3;
                    mbar_arrive_expect_tx(kfull, nok * B * 128u * NCH);
                }
                __syncwarp();
                // One box per page, at the page's place in the tile.
                if (ok) tma_load_5d(base + kKOff + st * kKBytes + r0 * 128 * NCH, &tm_k, kfull, 0, 0, 0, phys * (B >> 3), h);
            } else {
                const uint32_t vfull = smem_u32(&misc->vfull[st]);
                if (lane == 0) mbar_arrive_expect_tx(vfull, nok * B * 128u * NCH);
                __syncwarp();
                // One box per page, at the page's place in the tile.
                if (ok) tma_load_5d(base + kVOff + st * kVBytes + r0 * 128 * NCH, &tm_v, vfull, 0, 0, 0, phys * (B >> 3), h);
            }
            ++issued;
            if (i + 1 < nT) phys_next = fetch(i + 1);
        }
        if (misc->abort && lane == 0) {
            // Let the copies in flight land before the CTA can exit.
            if (kprod) mbar_wait(smem_u32(&misc->q_full), 0, &misc->never, kWaitLimitNs);
            for (int i = max(0, issued - nstages); i < issued; ++i)
                mbar_wait(smem_u32(kprod ? &misc->kfull[i % nstages] : &misc->vfull[i % nstages]), (i / nstages) & 1,
                          &misc->never, kWaitLimitNs);
        }
    }
    else if (warp == 1) {
        // ================= MMA issuer =================
        // Key tile i: for query tile 0, P.V of tile i-1 (its P lies in the
        // columns S(i) overwrites, so it goes first) and then S(i); the same
        // for query tile 1.  Meanwhile the softmax of the other query tile
        // runs.
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(kRows, kKeys, 0, 0);   // A = Q, B = K, both K-major
            constexpr uint32_t kIdescO = idesc_bf16(kRows, D, 0, 1);       // A = P (TMEM), B = V (MN-major)
            bool alive = mbar_wait(smem_u32(&misc->q_full), 0, &misc->abort, kWaitLimitNs);
            for (int i = 0; i <= nT && alive; ++i) {
                for (int x = 0; x < 2; ++x) {
                    const int nx = x ? n1 : n0;
                    const uint32_t s_col = tmem + kTmemS + x * 128;
                    if (i >= 1 && i - 1 < nx) {
                        const int t = i - 1;
                        alive = mbar_wait(smem_u32(&misc->p_full[x]), t & 1, &misc->abort, kWaitLimitNs) &&
                                mbar_wait(smem_u32(&misc->vfull[t % kVStages]), (t / kVStages) & 1, &misc->abort,
                                          kWaitLimitNs);
                        if (!alive) break;
                        tc_fence_after();
                        const uint32_t vbase = base + kVOff + (t % kVStages) * kVBytes;
#pragma unroll
                        for (int kk = 0; kk < kKeys / 16; ++kk) {
                            // Keys 16kk .. 16kk+15: 8-row blocks 2kk and 2kk + 1;
                            // the two 64-element halves 1,024 bytes apart.
                            const uint64_t b = smem_desc(vbase + kk * 2 * kAtomStride, 1024, kAtomStride, kLayoutSw128);
                            mma_bf16_tmem_a(tmem + kTmemO + x * 128, s_col + kk * 8, b, kIdescO,
                                            (t > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&misc->pv_done[x]));
                    }
                    if (i < nx) {
                        alive = mbar_wait(smem_u32(&misc->kfull[i % kKStages]), (i / kKStages) & 1, &misc->abort,
                                          kWaitLimitNs);
                        if (!alive) break;
                        tc_fence_after();
                        const uint32_t kbase = base + kKOff + (i % kKStages) * kKBytes;
                        const uint32_t qbase = base + kQOff + x * kQBytes;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                            // K: the half (kk / 4) of each 8-row block, 1,024
                            // bytes in for the second; atoms kAtomStride apart.
                            const uint32_t koff = (kk >> 2) * 1024u + (kk & 3) * 32;
                            const uint64_t a = smem_desc(qbase + off, 16, 1024, kLayoutSw128);
                            const uint64_t b = smem_desc(kbase + koff, 16, kAtomStride, kLayoutSw128);
                            mma_bf16(s_col, a, b, kIdescS, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&misc->s_full[x]));
                    }
                }
                if (!alive) break;
                if (i >= 1) mma_commit(smem_u32(&misc->vempty[(i - 1) % kVStages]));   // both P.V of tile i-1
                if (i < nT) mma_commit(smem_u32(&misc->kempty[i % kKStages]));         // both S of tile i
            }
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
    else if (warp < 10) {
        // ================= softmax: warps 2-5 tile 0, 6-9 tile 1; thread <-> query row =================
        const int x = (warp - 2) >> 2;
        const int nx = x ? n1 : n0;
        const int quad = warp & 3;                      // TMEM lanes 32 * (warp % 4) ..
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t s_col = lane_addr + kTmemS + x * 128;
        const uint32_t o_col = lane_addr + kTmemO + x * 128;
        const int tok0 = qt0 + x * QT;                  // first query token of this tile
        const int rr = row / G;                         // query token of this row (rows are token * G + head)
        const int qp = pos0 + tok0 + rr;                // its position: it sees keys 0 .. qp
        float m_ref = -INFINITY, l_run = 0.f;
        bool alive = nx > 0;
        for (int i = 0; i < nx; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->s_full[x]), i & 1, &misc->abort, kWaitLimitNs))) {
                alive = false;
                break;
            }
            // Tile 1's group starts half a period behind tile 0's (it
            // begins key tile 0 once tile 0's group has finished it), so that
            // the MMAs of one group run while the other computes.  (A barrier
            // of its own: p_full[0] may have moved on by more than a phase.)
            if (x == 1 && i == 0 && n0 > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->go), 0, &misc->abort, kWaitLimitNs))) {
                alive = false;
                break;
            }
            tc_fence_after();
            // The row's 128 scores of this tile into registers for the max
            // (two loads in flight, one wait).
            uint32_t sa[64], sb[64];
            tmemw::ld64(s_col, sa);
            tmemw::ld64(s_col + 64, sb);
            uint32_t msk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) msk[c] = misc->mask[i % kMaskRing][c];
            tmemw::wait_ld(sa);
            tmemw::wait_ld(sb);
            const int kbase = i * kKeys;
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
            auto gather = [&](auto easy_tag, auto max_tag) {
                constexpr bool kEasy = decltype(easy_tag)::value;
                constexpr bool kMax = decltype(max_tag)::value;
                auto v = [&](int k) -> float {
                    return kEasy ? score(k) : (visible(k) ? score(k) : __int_as_float(0x7fffffff));
                };
                auto pick3 = [&](float a, float b, float d) { return kMax ? max3(a, b, d) : min3(a, b, d); };
#pragma unroll
                for (int e = 0; e < 8; ++e) ext[e] = v(e);
#pragma unroll
                for (int k = 8; k + 16 <= kKeys; k += 16) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) ext[e] = pick3(ext[e], v(k + e), v(k + 8 + e));
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) ext[e] = kMax ? fmaxf(ext[e], v(kKeys - 8 + e)) : fminf(ext[e], v(kKeys - 8 + e));
                const float e0 = pick3(ext[0], ext[1], ext[2]), e1 = pick3(ext[3], ext[4], ext[5]);
                return pick3(e0, e1, kMax ? fmaxf(ext[6], ext[7]) : fminf(ext[6], ext[7]));
            };
            const float ex = easy ? (c >= 0.f ? gather(std::true_type{}, std::true_type{})
                                             : gather(std::true_type{}, std::false_type{}))
                                  : (c >= 0.f ? gather(std::false_type{}, std::true_type{})
                                             : gather(std::false_type{}, std::false_type{}));
            // No visible key (NaN): no candidate for the reference max.
            const float tmax = ex == ex ? ex * c : -INFINITY;
            const bool need = tmax > m_ref + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
                // Move this row's reference max and rescale its O and
                // denominator (rare after the first tile).
                const float mn = need ? tmax : m_ref;
                const float a = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - mn);
                // O holds key tiles up to i - 1: wait for that P.V.
                if (i > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[x]), (i - 1) & 1,
                                                                &misc->abort, kWaitLimitNs))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                if (i > 0) {
#pragma unroll
                    for (int cc = 0; cc < D / 8; ++cc) {
                        float ov[8];
                        tmem_ld<8>(o_col + cc * 8, ov);
#pragma unroll
                        for (int k = 0; k < 8; ++k) ov[k] *= a;
                        tmem_st8(o_col + cc * 8, ov);
                    }
                }
                l_run *= a;
                m_ref = mn;
            }
            // p = 2^(c * s - m_ref) as bf16 pairs over the first 64 columns
            // of S (the P.V MMA's A operand); the denominator sums the bf16
            // weights the MMA actually applies, in four chains.  The scores
            // are read again, 32 columns at a time with the next load in
            // flight (fewer live registers than keeping all 128): P of
            // columns 32cc.. goes to columns 16cc.., already read.
            const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
            const uint64_t c2 = f2(c, c), nm2 = f2(nm, nm);
            uint64_t lacc[2] = {0ull, 0ull};           // (+0, +0) pairs
            auto emit = [&](auto easy_tag) {
                constexpr bool kEasy = decltype(easy_tag)::value;
                uint32_t cb[2][32];
                tmemw::ld32(s_col, cb[0]);
                tmemw::wait_ld(cb[0]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    if (cc < 3) tmemw::ld32(s_col + 32 * (cc + 1), cb[(cc + 1) & 1]);
                    uint32_t packed[16];
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const int kk = cc * 32 + k;
                        const uint64_t arg =
                            ffma2(f2(__uint_as_float(cb[cc & 1][k]), __uint_as_float(cb[cc & 1][k + 1])), c2, nm2);
                        float a0, a1;
                        f2_split(arg, a0, a1);
                        float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
                        if constexpr (!kEasy) {
                            p0 = visible(kk) ? p0 : 0.f;
                            p1 = visible(kk + 1) ? p1 : 0.f;
                        }
                        const uint32_t w = pack_bf16x2(p0, p1);
                        packed[k / 2] = w;
                        lacc[(k >> 1) & 1] = fadd2(lacc[(k >> 1) & 1], f2(bf16_lo(w), bf16_hi(w)));
                    }
                    tmem_st16(s_col + cc * 16, packed);   // keys 32cc .. 32cc+31 of this row
                    if (cc < 3) tmemw::wait_ld(cb[(cc + 1) & 1]);
                }
            };
            if (easy) emit(std::true_type{});
            else emit(std::false_type{});
            {
                float a0, a1, b0, b1;
                f2_split(lacc[0], a0, a1);
                f2_split(lacc[1], b0, b1);
                l_run += (a0 + a1) + (b0 + b1);
            }
            // V rows of keys outside the sequence or behind a bad table entry
            // may hold stale or non-finite bits; the MMA multiplies them by 0,
            // so zero them (thread <-> key row) once V has landed.  The group
            // of the first query tile that uses this key tile does it, before
            // its P.V is issued (the other tile's P.V follows).
            const int wrow = row >> 5;                      // select, not an indexed load: msk stays in registers
            const uint32_t mrow = wrow == 0 ? msk[0] : wrow == 1 ? msk[1] : wrow == 2 ? msk[2] : msk[3];
            const bool bad = !((mrow >> (row & 31)) & 1u) && (x == 0 || i >= n0);
            if (__any_sync(0xffffffffu, bad)) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->vfull[i % kVStages]), (i / kVStages) & 1,
                                                       &misc->abort, kWaitLimitNs))) {
                    alive = false;
                    break;
                }
                if (bad) {
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        uint4 *vrow = reinterpret_cast<uint4 *>(smem + kVOff + (i % kVStages) * kVBytes +
                                                                (row >> 3) * kAtomStride + ch * 1024 + (row & 7) * 128);
#pragma unroll
                        for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            tmem_wait_st();                 // P is in TMEM before the MMA may read it
            fence_proxy_async_smem();       // zeroed V rows are visible to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&misc->p_full[x]));
            if (x == 0 && i == 0 && lane == 0) mbar_arrive(smem_u32(&misc->go));
        }
        if (alive && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->pv_done[x]), (nx - 1) & 1, &misc->abort,
                                                         kWaitLimitNs)))
            alive = false;
        if (!alive && nx > 0) {
            misc->abort = 1;
            set_error(p.err, PK_DEVERR_TIMEOUT);
        }
        // One decision for the whole group (every warp reaches this barrier;
        // the TMA-store path below has another).
        if (!named_bar_or(1 + x, 128, !alive)) {
            tc_fence_after();
            // O / l of this row to out[q0 + tok0 + token, h * G + head, :].
            const int ntok = min(qn - tok0, QT);
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            if (o_tma && ntok == QT) {
                // A full tile: bf16 rows into this tile's Q buffer (free: its
                // last S is done) in the 128-byte-swizzled layout of the
                // output map's box, then one TMA store per 64 columns.
                uint8_t *obuf = smem + kQOff + x * kQBytes;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint32_t ov[64];
                    tmemw::ld64(o_col + ch * 64, ov);
                    tmemw::wait_ld(ov);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(ov[8 * jj + 0]) * inv, __uint_as_float(ov[8 * jj + 1]) * inv);
                        u.y = pack_bf16x2(__uint_as_float(ov[8 * jj + 2]) * inv, __uint_as_float(ov[8 * jj + 3]) * inv);
                        u.z = pack_bf16x2(__uint_as_float(ov[8 * jj + 4]) * inv, __uint_as_float(ov[8 * jj + 5]) * inv);
                        u.w = pack_bf16x2(__uint_as_float(ov[8 * jj + 6]) * inv, __uint_as_float(ov[8 * jj + 7]) * inv);
                        *reinterpret_cast<uint4 *>(obuf + ch * kChunk + row * 128 + ((jj ^ (row & 7)) << 4)) = u;
                    }
                }
                fence_proxy_async_smem();
                group_bar(1 + x);
                if (quad == 2 && lane == 0) {               // one thread of the group
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
                        tma_store_3d(&tm_o, base + kQOff + x * kQBytes + ch * kChunk, ch * 64, h * G, q0 + tok0);
                    bulk_commit();
                    bulk_wait_read();                       // the buffer stays until the copy has read it
                }
            } else {
                const bool store = rr < ntok;
                const size_t obase =
                    (static_cast<size_t>(q0 + tok0 + rr) * H + h * G + (row & (G - 1))) * static_cast<size_t>(D);
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint32_t ov[64];
                    tmemw::ld64(o_col + ch * 64, ov);
                    tmemw::wait_ld(ov);
                    if (!store) continue;
                    float f[64];
#pragma unroll
                    for (int k = 0; k < 64; ++k) f[k] = __uint_as_float(ov[k]) * inv;
                    // (Device pointers are 16-byte aligned: the call checks.)
                    if (p.out_fp32) {
                        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + obase + ch * 64);
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
                    } else {
                        uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + obase + ch * 64);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            o[k] = make_uint4(pack_bf16x2(f[8 * k], f[8 * k + 1]), pack_bf16x2(f[8 * k + 2], f[8 * k + 3]),
                                              pack_bf16x2(f[8 * k + 4], f[8 * k + 5]),
                                              pack_bf16x2(f[8 * k + 6], f[8 * k + 7]));
                    }
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

// A tiled bf16 map with the 128-byte swizzle the MMA descriptors expect.
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
    // K and V: one box per (page, KV head) holding its B rows as B / 8 blocks
    // of [half][8 rows][64] (dimensions: 64 elements; row within the block;
    // half, 128 bytes apart; 8-row block, page * B / 8 + block; KV head).
    const cuuint64_t pdims[5] = {64, 8, Dd / 64, P * (B / 8), Hkv};
    const cuuint64_t pstr[4] = {Hkv * Dd * 2, 128, 8 * Hkv * Dd * 2, Dd * 2};
    const cuuint32_t pbox[5] = {64, 8, static_cast<cuuint32_t>(Dd / 64), static_cast<cuuint32_t>(B / 8), 1};
    // Queries (and bf16 outputs) [total_q, H, D]: box (64 elements, G heads,
    // 128 / G tokens) = one query tile, row = token * G + head.
    const cuuint64_t qdims[3] = {Dd, static_cast<cuuint64_t>(p.num_heads), static_cast<cuuint64_t>(p.total_q)};
    const cuuint64_t qstr[2] = {Dd * 2, Dd * p.num_heads * 2};
    const cuuint32_t qbox[3] = {64, G, kRows / G};
    CUtensorMap mk, mv, mq, mo;
    if (!encode(&mk, p.k_cache, 5, pdims, pstr, pbox) || !encode(&mv, p.v_cache, 5, pdims, pstr, pbox) ||
        !encode(&mq, p.q, 3, qdims, qstr, qbox))
        return cudaErrorInvalidValue;
    // Full tiles of a bf16 output go out by TMA store; otherwise (fp32, or
    // an output the map does not accept) by plain stores.
    int o_tma = 0;
    if (!p.out_fp32 && encode(&mo, p.out, 3, qdims, qstr, qbox)) o_tma = 1;
    else mo = mq;
    {
        const cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(prefill_tc_kernel<D, G>),
                                                   static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
    }
    const int qblocks = (max_q_len + 2 * (kRows / G) - 1) / (2 * (kRows / G));
    const int64_t grid = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads * qblocks;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    prefill_tc_kernel<D, G><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(mk, mv, mq, mo, p, qblocks,
                                                                                           o_tma);
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
