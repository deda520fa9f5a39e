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
// into gridDim.x contiguous ranges of equal cost (tiles, tokens and
// (sequence, head) segments each weighted; see kTileCost), one per
// persistent CTA (one CTA per SM).  A CTA's range covers whole segments, which it writes straight to
// the output, plus at most two cut segments at its ends, whose partial (max,
// denominator, unnormalised output) go to a workspace slot and are combined
// by the merge kernel.
//
// Per 128-token tile, inside a CTA (192 threads):
//   warp 0  producer: reads the tile's block-table entries one tile ahead
//           (one lane per page), checks them, and TMA-loads each page's K rows
//           and then V rows of this KV head (one box each, landing as 8-row
//           blocks [half][8 rows][64] with the 128-byte swizzle) into a
//           3-stage shared-memory ring; K (with the
//           group's 16 query rows, loaded only when the stage does not hold
//           them already) and V complete separate barriers, so the scores
//           can start while V is still landing; the tile's position
//           (sequence, head, tile, tiles in segment) goes with the stage, so
//           the other roles never walk the sequence lengths themselves;
//   warp 1  MMA issuer (one thread, event loop): S^T[128 x 16] =
//           K[128 x D] Q^T[D x 16] into TMEM as soon as a tile's K is in, and
//           O^T[D x 16] += V^T[D x 128] P^T[128 x 16] into TMEM as soon as its
//           probabilities are written, so neither waits for the other; O of a
//           (sequence, head) segment accumulates in TMEM across its tiles;
//   warps 2-5 (128 threads, thread <-> TMEM lane): read S^T (one token per
//           thread), mask invalid tokens, compute p = 2^(s - m_ref) in fp32,
//           round to bf16 for the MMA and keep the denominator.  m_ref is a
//           reference max per query head that moves only when a score exceeds
//           it by more than 2^8 (then O in TMEM and the denominator are
//           rescaled); between moves a tile costs one OR-vote barrier.  A
//           segment's O is read out of TMEM one tile after its last P.V was
//           issued, normalised and stored (or written to a slot if cut).
// Launch: the decode grid is a programmatic dependent of the previous kernel
// in the stream: its set-up -- barriers, TMEM, and the plan of its range from
// the sequence lengths (read again after the wait; the plan is redone if one
// changed) -- overlaps that kernel's tail.  The merge grid is a programmatic
// dependent of the decode grid and lets the next decode grid start at once,
// so back-to-back calls overlap one call's set-up with the previous call's
// end.
// Query heads are padded to the MMA's N = 16; padded columns are ignored.
#include "decode.cuh"
#include "sm100.cuh"
#include "block_scan.cuh"

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
constexpr uint64_t kWaitLimitNs = 1000000000ull;             // 1 s: far beyond any legal wait (default)
constexpr int kLenCache = 2048;                              // lengths kept in shared memory up to this batch

constexpr uint32_t kIdescQK = idesc_bf16(kTile, kNPad, 0, 0);   // A = K (K-major), B = Q (K-major)
constexpr uint32_t kIdescPV = idesc_bf16(128, kNPad, 1, 1);     // A = V^T (MN-major), B = P^T (MN-major)

struct Misc {
    uint64_t full[kStages];       // K rows (and Q) of a stage landed
    uint64_t vfull[kStages];      // V rows of a stage landed
    uint64_t empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_full[2];       // P.V of a tile complete (per tile parity)
    uint64_t o_free[2];       // a segment's O buffer has been read out
    uint64_t drain;
    int64_t scan[kThreads / 32 + 1];   // warp totals of the prologue scans (tiles)
    int64_t scan_w[kThreads / 32 + 1]; // (costs)
    int64_t bnd[2];                    // first tile of this CTA's range and of the next one
    int64_t rem0;
    int32_t s0;
    int32_t first_cta;                 // the CTA in whose range this CTA's first segment starts
    uint32_t tmem_base;
    int abort;
    int never;
    uint32_t mask[kStages][4];
    int4 meta[kStages];            // (sequence, KV head, tile, tiles in segment) of a stage's tile
    int4 qmeta[kStages];           // (first query row, query tokens, first query position, 0) of it
    float red[4][kNPad];          // per-warp maxima when the reference max moves
    float lsum[4][kNPad];
    int lens[kLenCache];          // the raw sequence lengths, when num_seqs <= kLenCache
};

constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 2 * kPBytes + sizeof(Misc);

// Workspace slot of a cut segment's part: slot 0 of a CTA holds the part of
// its first segment, slot 1 the part of its last one.
struct Slot {
    int32_t flag;          // slot 0 only: 1 = the merge kernel's CTA c combines this segment
    int32_t s, h;
    int32_t first_cta;     // slot 0 only: the CTA in whose range the segment starts
    int64_t start_tile;    // flattened index of the segment's (s, h) tile 0
    int64_t total_tiles;
    int64_t range_beg;     // slot 0 only: first tile of this CTA's range
    int64_t pad2[3];
    float m[kNPad];        // reference max per column (base 2)
    float l[kNPad];        // denominator per column
    float o[kNPad * 128];  // unnormalised output, [column][O^T row]
};
constexpr size_t kMaxCtas = kTcMaxCtas;

// A 32-bit load that bypasses L1: L2 is coherent with writes of other
// grids, so a value read before the programmatic wait and read again after
// it cannot come back stale from L1.
__device__ __forceinline__ int ld_cg(const int *p) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// The sequence lengths, from the shared-memory copy when there is one;
// operator() clamps to [0, cap] (values outside are reported separately).
struct LenSrc {
    const int *cache;   // shared memory, or null
    const int *glob;
    int cap;
    __device__ __forceinline__ int raw(int s) const { return cache ? cache[s] : glob[s]; }
    __device__ __forceinline__ int operator()(int s) const {
        const int r = raw(s);
        return r < 0 ? 0 : (r > cap ? cap : r);
    }
};

// Walks the flattened (sequence, KV head group, tile) space in order.
struct Walk {
    int s, h, t, nt, L, nh, ns;      // nh: KV head groups per sequence; ns: sequences
    __device__ __forceinline__ void load(const LenSrc &len) {
        L = len(s);
        nt = (L + kTile - 1) / kTile;
    }
    __device__ __forceinline__ void next(const LenSrc &len) {
        if (++t < nt) return;
        t = 0;
        if (++h < nh) return;
        h = 0;
        do {
            if (++s >= ns) return;
            load(len);
        } while (nt == 0);
    }
};

// This CTA's range of the flattened tile space.  Tile x, whose cost interval
// starts at a_x (a segment's tile 0 at its start, tile t >= 1 at start +
// seg_cost + full * t, full the cost of a full tile), belongs to CTA k when
// P_k <= a_x < P_{k+1}, P_k = k * W / C, W the total cost.  Writes misc->bnd (the first tile of this range and of the next),
// misc->s0 / rem0 (where the range starts) and misc->first_cta (the CTA in
// whose range a segment cut at this range's start begins); returns the
// total tile count and, in *odd, whether some length is zero or outside
// [0, cap] (the same for every thread).  Every thread of the CTA calls it.
template <int kThreadsT, typename MiscT>
__device__ __forceinline__ int64_t plan_range(const LenSrc lens, MiscT *misc, int N, int Hkv, int c, int C,
                                           int64_t seg_cost, int tile_cost, int tok_cost, int *odd) {
    // A segment of L tokens in nt tiles costs seg_cost + tile_cost * nt -
    // tok_cost * L: a full tile costs full = tile_cost - tok_cost * kTile, and
    // only a segment's last tile can be partial, so tile t >= 1 starts at
    // seg_cost + full * t.
    const int64_t full = tile_cost - static_cast<int64_t>(tok_cost) * kTile;
    auto seg_total = [&](int64_t nt, int L) -> int64_t {
        return nt > 0 ? seg_cost + tile_cost * nt - static_cast<int64_t>(tok_cost) * L : 0;
    };
    const int per = (N + kThreadsT - 1) / kThreadsT;
    const int s_lo = min(N, static_cast<int>(threadIdx.x) * per), s_hi = min(N, s_lo + per);
    const int cap = lens.cap;
    int64_t mine = 0, mine_w = 0;
    int bad = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        const int raw = lens.raw(s);
        bad |= raw <= 0 || raw > cap;
        const int L = lens(s);
        const int64_t nt = (L + kTile - 1) / kTile;
        mine += nt * Hkv;
        mine_w += seg_total(nt, L) * Hkv;
    }
    int64_t T, W;
    const int64_t my_off = block_exclusive_scan<kThreadsT>(mine, misc->scan, &T);
    const int64_t my_off_w = block_exclusive_scan<kThreadsT>(mine_w, misc->scan_w, &W);
    for (int k = 0; k < 2; ++k) {
        const int64_t P = static_cast<int64_t>(c + k) * W / C;
        if (P >= W) {
            if (threadIdx.x == 0) misc->bnd[k] = T;
            continue;
        }
        if (my_off_w <= P && P < my_off_w + mine_w) {
            int64_t acc_t = my_off, acc_w = my_off_w;
            for (int s = s_lo; s < s_hi; ++s) {
                const int L = lens(s);
                const int64_t nt = (L + kTile - 1) / kTile;
                const int64_t segc = seg_total(nt, L);
                const int64_t cw = segc * Hkv;
                if (P < acc_w + cw) {
                    const int64_t q = P - acc_w;
                    int64_t h = q / segc;
                    const int64_t r = q - h * segc;
                    // The first tile of the segment that starts at or after r.
                    int64_t t = r == 0 ? 0 : (r - seg_cost + full - 1) / full;
                    if (r > 0 && t < 1) t = 1;
                    if (t >= nt) {
                        ++h;
                        t = 0;
                    }
                    misc->bnd[k] = acc_t + h * nt + t;
                    break;
                }
                acc_t += nt * Hkv;
                acc_w += cw;
            }
        }
    }
    __syncthreads();
    const int64_t b0 = misc->bnd[0];
    if (misc->bnd[1] > b0) {
        int64_t acc = my_off, acc_w = my_off_w;
        if (acc <= b0 && b0 < acc + mine) {
            for (int s = s_lo; s < s_hi; ++s) {
                const int L = lens(s);
                const int64_t nt = (L + kTile - 1) / kTile;
                const int64_t w = nt * Hkv;
                if (b0 < acc + w) {
                    misc->s0 = s;
                    misc->rem0 = b0 - acc;
                    // If the range starts inside a segment, the CTA where that
                    // segment starts (the owner of its tile 0's cost start).
                    const int64_t h0 = (b0 - acc) / nt;
                    const int64_t a = acc_w + h0 * seg_total(nt, L);
                    int64_t k = W > 0 ? a * C / W : 0;
                    while (k + 1 < C && (k + 1) * W / C <= a) ++k;
                    while (k > 0 && k * W / C > a) --k;
                    misc->first_cta = static_cast<int32_t>(k);
                    break;
                }
                acc += w;
                acc_w += seg_total(nt, L) * Hkv;
            }
        }
    }
    *odd = __syncthreads_or(bad);
    return T;
}

// The flattened (sequence, KV head, tile) space is cut into ranges of equal
// cost, not of equal tile count.  A segment of L tokens in nt tiles costs
// seg_cost + kTileCost * nt - kTokCost * L: a CTA's time grows with its
// (sequence, KV head) segments (each loads its queries, sets up and reads
// out its O) and with its tiles, and a tile's time shrinks less than its
// bytes when it is only partly filled (the ring holds a fixed number of
// tiles, so a partial tile keeps fewer bytes in flight).  The weights come
// from a least-squares fit of per-CTA times (in-kernel timestamps) to the
// tiles, pages and segments of each CTA's range, over back-to-back calls on
// five batches: a full tile costs 272, a one-token tile 399, a segment 56 --
// 200 when 16 query columns are in use (the read-out and the reference-max
// moves work on every column) -- and half as much with head pairs, whose
// tiles carry twice the bytes.
constexpr int64_t kTileCost = 400;
constexpr int kTokCost = 1;
template <int NUSED, int HP>
constexpr int64_t seg_cost() { return (NUSED > 8 ? 200 : 56) / HP; }

// Warp max of a float in one integer reduction: the bits are mapped to an
// unsigned key with the same order (a non-negative float gets its sign bit
// set, a negative one all bits flipped), reduced, and mapped back.
__device__ __forceinline__ float warp_max_redux(float v) {
    const uint32_t b = __float_as_uint(v);
    const uint32_t key = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    const uint32_t m = __reduce_max_sync(0xffffffffu, key);
    return __uint_as_float((m & 0x80000000u) ? (m & 0x7fffffffu) : ~m);
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

// HP KV heads per tile: HP = 2 pairs two adjacent KV heads at head dim 64,
// so that each token's page row is one 256-byte piece (the two heads side by
// side in the cache) instead of two 128-byte pieces 1 KiB apart.
template <int D, int NC, bool MQ, int HP>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(NC >= 1 && NC <= kNPad, "group");
    static_assert(HP == 1 || (HP == 2 && D == 64 && NC <= 8), "head pairs: head dim 64, at most 8 columns each");
    constexpr int NCH = D * HP / 64;                  // 128-byte chunks of a tile row
    // TMEM: S^T double-buffered (16 columns per head of the tile), then O^T
    // double-buffered by segment (16 columns).  P and O columns: HP == 1,
    // column g = query column g; HP == 2, columns 0-7 belong to the pair's
    // first head and 8-15 to its second, NC query columns each (the rest
    // padding); O^T rows are then (head of the pair, head-dim element).
    constexpr uint32_t kSCols = 16 * HP;
    constexpr uint32_t tS = 0, tO = 2 * kSCols;
    constexpr uint32_t kTmemCols = HP == 2 ? 128 : 64;
    constexpr int CW = HP == 2 ? 8 : kNPad;           // P columns per head of the tile
    constexpr int NCOL = HP == 2 ? 8 + NC : NC;       // columns 0 .. NCOL-1 may be in use
    constexpr int64_t kSegCost = seg_cost<HP * NC, HP>();   // a segment's cost (the columns in use, head pairs)
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
    // Hkv counts the tile's KV head groups (segments per sequence).
    const int N = p.num_seqs, Hkv = p.num_kv_heads / HP, H = p.num_heads, B = p.block_size;
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * B);
    const int Gq = H / p.num_kv_heads, lgG = __ffs(Gq) - 1;     // query heads per KV head (a power of two)
    // K and V of a tile in shared memory: each page in one TMA box as B / 8
    // blocks of 8 rows, each block [half][8 rows][64] -- so the 8-row
    // swizzle atoms of one 64-element half lie kAtomStride bytes apart
    // whatever the block size, a uniform stride for the MMA descriptors.
    constexpr uint32_t kAtomStride = 1024u * NCH;
    constexpr bool mq = MQ;                           // several query tokens per sequence
    Slot *slots = static_cast<Slot *>(p.tc_slots);
    const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&misc->full[i]), 1);
            mbar_init(smem_u32(&misc->vfull[i]), 1);
            mbar_init(smem_u32(&misc->empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&misc->s_full[i]), 1);
            mbar_init(smem_u32(&misc->p_full[i]), 4);
            mbar_init(smem_u32(&misc->o_full[i]), 1);
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
    // ---- this CTA's range of the flattened tile space ----------------------
    // With the lengths in shared memory, the range is planned before the
    // wait, while the previous grid in the stream finishes; after the wait
    // the lengths are read again and the plan is redone only if one changed.
    const bool cached = N <= kLenCache;
    const LenSrc lens{cached ? misc->lens : nullptr, p.seq_lens, cap};
    int64_t T = 0;
    int odd = 0;
    // The first tile of the range, from the plan.
    auto first_tile = [&]() -> Walk {
        Walk w{};
        w.nh = Hkv;
        w.ns = N;
        w.s = misc->s0;
        w.load(lens);
        w.h = static_cast<int>(misc->rem0 / w.nt);
        w.t = static_cast<int>(misc->rem0 % w.nt);
        return w;
    };
    // Launched as a programmatic dependent of the previous kernel in the
    // stream: what comes before the wait overlaps that kernel's tail.  Apart
    // from the lengths, which are checked after it, no global memory is read
    // before it, and none is written.
    auto wait_prev = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (threadIdx.x == 0 && slots) slots[2 * c].flag = 0;
        // The merge grid may start now; it waits for this grid's completion.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    };
    bool ahead = cached;   // planning before the wait
    if (cached) {
        const int32_t *first_read = p.lens_ahead ? p.lens_ahead : p.seq_lens;
        for (int s = threadIdx.x; s < N; s += kThreads) misc->lens[s] = ld_cg(first_read + s);
        __syncthreads();
    } else {
        wait_prev();
    }
    for (;;) {
        T = plan_range<kThreads>(lens, misc, N, Hkv, c, C, kSegCost, kTileCost, kTokCost, &odd);
        if (!ahead) break;
        ahead = false;
        wait_prev();
        // Changed values are written back only after every thread has
        // compared its own (each thread owns the same entries as above).
        int changed = 0;
        for (int s = threadIdx.x; s < N; s += kThreads) changed |= ld_cg(p.seq_lens + s) != misc->lens[s];
        if (!__syncthreads_or(changed)) break;
        for (int s = threadIdx.x; s < N; s += kThreads) misc->lens[s] = ld_cg(p.seq_lens + s);
        __syncthreads();
    }
    const int64_t beg = misc->bnd[0], end = misc->bnd[1];
    if (threadIdx.x == 0 && slots) slots[2 * c].range_beg = beg;
    const int n_tiles = static_cast<int>(end - beg);
    // Lengths outside [0, cap] are reported, and empty sequences get zeros,
    // by CTA s % C.
    if (odd || mq) {
        for (int s = c; s < N; s += C) {
            const int raw = lens.raw(s);
            if ((raw < 0 || raw > cap) && threadIdx.x == 0) set_error(p.err, PK_DEVERR_SEQ_LEN);
            const int L = lens(s);
            if (mq) {
                // A sequence has at most L query tokens (they are its newest tokens).
                const int r0 = p.cu_q_lens[s], r1 = p.cu_q_lens[s + 1];
                if (r1 < r0 || r1 - r0 > L) set_error(p.err, PK_DEVERR_SEQ_LEN);
                if (L != 0) continue;
                for (int64_t i = threadIdx.x; i < static_cast<int64_t>(max(r1 - r0, 0)) * H * D; i += kThreads)
                    store_out(p, static_cast<size_t>(r0) * H * D + i, 0.f);
                continue;
            }
            if (L != 0) continue;
            for (int i = threadIdx.x; i < H * D; i += kThreads) store_out(p, static_cast<size_t>(s) * H * D + i, 0.f);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;

    Walk w0{};
    w0.nh = Hkv;
    w0.ns = N;
    if (n_tiles > 0) w0 = first_tile();

    if (warp == 0) {
        // ================= producer =================
        Walk w = w0;
        const int MB = p.max_blocks_per_seq;
        int issued = 0;
        // The next tile's block-table entries are read one tile ahead, so
        // their latency hides behind the wait for a free stage.
        auto fetch = [&](const Walk &ww) -> int {
            const int fp = ww.t * kTile / B;
            return (lane < kTile / B && fp + lane < MB) ? p.block_tables[static_cast<size_t>(ww.s) * MB + fp + lane]
                                                        : -1;
        };
        int phys_next = n_tiles > 0 ? fetch(w) : -1;
        int seg_i0 = 0;
        bool stalled = false;
        for (int i = 0; i < n_tiles; ++i) {
            // Self-test of the bounded waits: CTA 0 stops issuing here, so
            // the barriers of this tile never complete.
            if (p.stall_tile > 0 && c == 0 && i == p.stall_tile) {
                stalled = true;
                break;
            }
            if (i == 0 || w.t == 0) seg_i0 = i;
            // The stage still holds this segment's queries from tile i - kStages.
            const bool q_resident = i - seg_i0 >= kStages;
            const int st = i % kStages;
            const int phys_raw = phys_next;
            int got = 1;
            if (lane == 0)
                got = mbar_wait(smem_u32(&misc->empty[st]), ((i / kStages) & 1) ^ 1, &misc->abort, lim);
            if (!__shfl_sync(0xffffffffu, got, 0)) {      // one decision for the whole warp
                if (lane == 0) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                }
                break;
            }
            const int tok0 = w.t * kTile;
            const int vlen = min(kTile, w.L - tok0);
            // The sequence's query rows: its newest qn tokens (one for decode).
            int qrow0 = w.s, qn = 1;
            if constexpr (MQ) {
                qrow0 = p.cu_q_lens[w.s];
                qn = p.cu_q_lens[w.s + 1] - qrow0;
            }
            constexpr uint32_t q_bytes = (MQ ? NC : kNPad) * 128u * NCH;
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
                misc->meta[st] = make_int4(w.s, w.h, w.t, w.nt);
                if constexpr (MQ) misc->qmeta[st] = make_int4(qrow0, qn, w.L - qn, 0);
                mbar_arrive_expect_tx(full, nok * B * 128u * NCH + (q_resident ? 0u : q_bytes));
                mbar_arrive_expect_tx(vfull, nok * B * 128u * NCH);
            }
            __syncwarp();
            // K (and Q) first: the scores can start while V is still landing.
            if (lane == 0 && !q_resident) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    // Chunk ch: elements 64 ch .. 64 ch + 63 of the KV head's
                    // queries (HP == 1), or all 64 of the pair's head ch (HP == 2).
                    const int qx = HP == 2 ? 0 : ch * 64;
                    const int qh = (w.h * HP + (HP == 2 ? ch : 0)) * Gq;
                    if constexpr (MQ)   // box (64, G heads, q_len tokens): column r * G + g
                        tma_load_3d(sbase + kQOff + ch * kQChunkBytes, &tm_q, full, qx, qh, qrow0);
                    else      // box (64, 16 rows) of the [N * H, D] queries
                        tma_load_2d(sbase + kQOff + ch * kQChunkBytes, &tm_q, full, qx, w.s * H + qh);
                }
            }
            if (ok) {
                // One box of K and one of V per page, at the page's place in the tile.
                const int rb = phys * (B >> 3);                  // the page's first 8-row block
                tma_load_5d(sbase + kKOff + r0 * 128 * NCH, &tm_k, full, 0, 0, 0, rb, w.h);
                tma_load_5d(sbase + kVOff + r0 * 128 * NCH, &tm_v, vfull, 0, 0, 0, rb, w.h);
            }
            ++issued;
            w.next(lens);
            if (i + 1 < n_tiles) phys_next = fetch(w);
        }
        // On abort (or a self-test stall), let this warp's copies land before
        // the CTA can exit.
        if ((misc->abort || stalled) && lane == 0) {
            for (int i = max(0, issued - kStages); i < issued; ++i) {
                mbar_wait(smem_u32(&misc->full[i % kStages]), (i / kStages) & 1, &misc->never, lim);
                mbar_wait(smem_u32(&misc->vfull[i % kStages]), (i / kStages) & 1, &misc->never, lim);
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            // Segment bookkeeping for P.V: O of a (sequence, head) segment
            // accumulates in TMEM buffer (segment index & 1) across its tiles.
            int pv_seg = -1;
            auto pv = [&](int j, bool first, int sg) {
                const int pb = j & 1;
                tc_fence_after();
                const uint32_t vbase = stage_addr + (j % kStages) * kStageBytes + kVOff;
                const uint32_t pbase = p_addr + pb * kPBytes;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    // Tokens 16kk .. 16kk+15: 8-row blocks 2kk and 2kk + 1; the
                    // two 64-element halves 1,024 bytes apart.
                    const uint64_t a = smem_desc(vbase + kk * 2 * kAtomStride, 1024, kAtomStride, kLayoutSw128);
                    const uint64_t b = smem_desc(pbase + kk * 512, 256, 128, kLayoutNone);
                    mma_bf16(tmem + tO + (sg & 1) * kNPad, a, b, kIdescPV, (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(smem_u32(&misc->o_full[pb]));
                mma_commit(smem_u32(&misc->empty[j % kStages]));
            };
            // Event loop: issue P.V of a tile as soon as its probabilities are
            // written (releasing its stage), and the scores of the next tile
            // as soon as it has arrived; neither waits for the other.
            auto qk = [&](int i) {
                const int st = i % kStages;
                tc_fence_after();
                const uint32_t sbase = stage_addr + st * kStageBytes;
                const int sb = i & 1;
#pragma unroll
                for (int kk = 0; kk < NCH * 4; ++kk) {
                    // K: the chunk (kk / 4) of each 8-row block, 1,024 bytes in
                    // for the second; atoms kAtomStride apart.  HP == 2: chunk
                    // kk / 4 is head kk / 4 of the pair, whose scores go to
                    // their own 16 columns.
                    const uint32_t off = (kk >> 2) * 1024u + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * kQChunkBytes + (kk & 3) * 32;
                    const uint64_t a = smem_desc(sbase + kKOff + off, 16, kAtomStride, kLayoutSw128);
                    const uint64_t b = smem_desc(sbase + kQOff + qoff, 16, 1024, kLayoutSw128);
                    const uint32_t dcol = tS + sb * kSCols + (HP == 2 ? (kk >> 2) * 16u : 0u);
                    const bool acc = HP == 2 ? (kk & 3) > 0 : kk > 0;
                    mma_bf16(tmem + dcol, a, b, kIdescQK, acc ? 1u : 0u);
                }
                mma_commit(smem_u32(&misc->s_full[sb]));
            };
            int nq = 0, np = 0;
            uint64_t t_idle = 0;
            uint32_t spins = 0;
            while (np < n_tiles) {
                bool prog = false;
                if (np < nq && mbar_test_wait(smem_u32(&misc->p_full[np & 1]), (np >> 1) & 1) &&
                    mbar_test_wait(smem_u32(&misc->vfull[np % kStages]), (np / kStages) & 1)) {
                    const bool first = np == 0 || misc->meta[np % kStages].z == 0;
                    const int sg = pv_seg + (first ? 1 : 0);
                    // A new segment's O buffer must have been read out (segment sg - 2).
                    if (!first || mbar_test_wait(smem_u32(&misc->o_free[sg & 1]), ((sg >> 1) & 1) ^ 1)) {
                        pv(np, first, sg);
                        pv_seg = sg;
                        ++np;
                        prog = true;
                    }
                }
                if (nq < n_tiles && nq <= np + 1 &&
                    mbar_test_wait(smem_u32(&misc->full[nq % kStages]), (nq / kStages) & 1)) {
                    qk(nq);
                    ++nq;
                    prog = true;
                }
                if (prog) {
                    spins = 0;
                } else if ((++spins & 255u) == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (spins == 256) t_idle = now;
                    else if (misc->abort || now - t_idle > lim) {
                        misc->abort = 1;
                        set_error(p.err, PK_DEVERR_TIMEOUT);
                        break;
                    }
                }
            }
            // Let every issued MMA finish before the CTA can release TMEM.
            mma_commit(smem_u32(&misc->drain));
            mbar_wait(smem_u32(&misc->drain), 0, &misc->never, lim);
        }
        __syncwarp();
    } else {
        // ================= softmax (warps 2-5): thread <-> tile row =================
        // A reference max per query head moves only when a score exceeds it
        // by more than 2^8 (then O in TMEM and the denominators are rescaled);
        // between moves p = 2^(s - m_ref) <= 2^8 and a tile costs one vote.
        // A segment's output is read out of TMEM one tile later, when its
        // last P.V is certainly done.
        constexpr float kRescaleLog2 = 8.0f;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        float m_ref[NCOL], l_run[NCOL], m_prev[NCOL], l_prev[NCOL];
#pragma unroll
        for (int j = 0; j < NCOL; ++j) m_ref[j] = l_run[j] = m_prev[j] = l_prev[j] = 0.f;
        // This thread's TMEM lane as an O^T row: the head-dim element (HP ==
        // 1), or (head of the pair, element) = (row / 64, row % 64) (HP == 2).
        const int hr = HP == 2 ? row >> 6 : 0;
        const int dd = HP == 2 ? (row & 63) : row;
        const bool row_ok = HP == 2 || row < D;
        // Query column c of this row's head, from a 16-column row of O or l.
        auto colv = [&](const float (&v)[kNPad], int cq) -> float {
            if constexpr (HP == 2) return hr ? v[CW + cq] : v[cq];
            else return v[cq];
        };
        int seg = -1, seg_t0 = 0, seg_i0 = 0;
        bool pending = false;            // a finished segment awaits its read-out
        int pend_seg = 0, pend_s = 0, pend_h = 0, pend_i = 0, pend_t0 = 0, pend_i0 = 0, pend_q0 = 0, pend_qn = 1;
        bool pend_complete = false, pend_cut_end = false;
        auto finalize = [&]() -> bool {
            // P.V of the segment's last tile (pend_i) complete.
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->o_full[pend_i & 1]), (pend_i >> 1) & 1,
                                                   &misc->never, lim)))
                return false;
            tc_fence_after();
            float ov[kNPad];
            tmem_ld16(lane_addr + tO + (pend_seg & 1) * kNPad, ov);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&misc->o_free[pend_seg & 1]));
#pragma unroll
            for (int j = 0; j < NCOL; ++j) {
                const float v = warp_sum(l_prev[j]);
                if (lane == 0) misc->lsum[quad][j] = v;
            }
            named_bar_sync(1, 128);
            float l[kNPad];
#pragma unroll
            for (int j = 0; j < kNPad; ++j)
                l[j] = j < NCOL ? misc->lsum[0][j] + misc->lsum[1][j] + misc->lsum[2][j] + misc->lsum[3][j] : 0.f;
            if (pend_complete) {
                if (row_ok) {
#pragma unroll
                    for (int cq = 0; cq < NC; ++cq) {
                        // Column cq: query token cq / G (multi-query; padded
                        // columns past the sequence's queries are not
                        // written), query head cq % G of this row's KV head.
                        if ((cq >> lgG) >= pend_qn) continue;
                        const float lv = colv(l, cq);
                        const size_t qrow = static_cast<size_t>(MQ ? pend_q0 : pend_s) + (cq >> lgG);
                        const int qh = (pend_h * HP + hr) * Gq + (cq & (Gq - 1));
                        store_out(p, (qrow * H + qh) * D + dd, lv > 0.f ? colv(ov, cq) / lv : 0.f);
                    }
                }
            } else {
                // A cut part: slot 0 if the segment is this CTA's first, 1 if not.
                const int slot_idx = pend_i0 == 0 ? 0 : 1;
                Slot *sl = slots + 2 * c + slot_idx;
                if (row_ok) {
#pragma unroll
                    for (int cq = 0; cq < NC; ++cq) sl->o[(hr * CW + cq) * 128 + row] = colv(ov, cq);
                }
                if (row == 0) {
#pragma unroll
                    for (int j = 0; j < NCOL; ++j) {
                        sl->m[j] = m_prev[j];
                        sl->l[j] = l[j];
                    }
                    sl->s = pend_s;
                    sl->h = pend_h;
                    sl->start_tile = beg + pend_i0 - pend_t0;
                    sl->total_tiles = T;
                    // Cut at its start and finished here: this CTA merges it.
                    if (slot_idx == 0) {
                        sl->flag = (pend_t0 > 0 && pend_cut_end) ? 1 : 0;
                        sl->first_cta = misc->first_cta;
                    }
                }
            }
            pending = false;
            return true;
        };
        for (int i = 0; i < n_tiles; ++i) {
            const int st = i % kStages;
            const int sb = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->s_full[sb]), (i >> 1) & 1, &misc->never,
                                                   lim))) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
            const int4 mt = misc->meta[st];   // (s, h, t, nt), written with the stage
            int4 qm = make_int4(mt.x, 1, 0, 0);
            if constexpr (MQ) qm = misc->qmeta[st];  // (first query row, query tokens, first query position)
            const bool seg_first = (i == 0) || (mt.z == 0);
            const bool seg_last = (i == n_tiles - 1) || (mt.z == mt.w - 1);
            if (seg_first) {
                ++seg;
                seg_t0 = mt.z;
                seg_i0 = i;
#pragma unroll
                for (int j = 0; j < NCOL; ++j) {
                    m_ref[j] = -INFINITY;
                    l_run[j] = 0.f;
                }
            }
            tc_fence_after();
            float sv[kNPad];
            if constexpr (HP == 2) {
                // The pair's scores: columns 0-7 of each head's 16.
                float s0[8], s1[8];
                tmem_ld<8>(lane_addr + tS + sb * kSCols, s0);
                tmem_ld<8>(lane_addr + tS + sb * kSCols + 16, s1);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    sv[j] = s0[j];
                    sv[8 + j] = s1[j];
                }
            } else {
                tmem_ld16(lane_addr + tS + sb * kSCols, sv);
            }
            const bool valid = (misc->mask[st][row >> 5] >> (row & 31)) & 1u;
            float s2[NCOL];
            bool need = false;
            const int jpos = mt.z * kTile + row;          // this row's token position
#pragma unroll
            for (int j = 0; j < NCOL; ++j) {
                if ((j % CW) >= NC) {                      // padding column of a head pair
                    s2[j] = -INFINITY;
                    continue;
                }
                // Multi-query: query column j % CW is query token (j % CW) / G,
                // which sees positions <= its own.
                const bool vg = valid && (!mq || jpos <= qm.z + ((j % CW) >> lgG));
                s2[j] = vg ? sv[j] * p.scale_log2 : -INFINITY;
                need |= s2[j] > m_ref[j] + kRescaleLog2;
            }
            if (named_bar_or(1, 128, need)) {
                // Rare: move the reference to the running max.
#pragma unroll
                for (int j = 0; j < NCOL; ++j) {
                    const float mx = warp_max_redux(s2[j]);
                    if (lane == 0) misc->red[quad][j] = mx;
                }
                named_bar_sync(1, 128);
                float a[NCOL];
#pragma unroll
                for (int j = 0; j < NCOL; ++j) {
                    const float t = fmaxf(fmaxf(misc->red[0][j], misc->red[1][j]),
                                          fmaxf(misc->red[2][j], misc->red[3][j]));
                    const float mn = fmaxf(m_ref[j], t);
                    a[j] = m_ref[j] == -INFINITY ? 0.f : fast_exp2(m_ref[j] - mn);
                    l_run[j] *= a[j];
                    m_ref[j] = mn;
                }
                if (!seg_first) {
                    // O through tile i-1, in TMEM (thread <-> head-dim row).
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->o_full[(i - 1) & 1]), ((i - 1) >> 1) & 1,
                                                           &misc->never, lim))) {
                        misc->abort = 1;
                        set_error(p.err, PK_DEVERR_TIMEOUT);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t oaddr = lane_addr + tO + (seg & 1) * kNPad;
                    float ov[16];
                    tmem_ld16(oaddr, ov);
                    float lo[8], hi[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        lo[j] = j < NCOL ? ov[j] * a[j < NCOL ? j : 0] : ov[j];
                        hi[j] = 8 + j < NCOL ? ov[8 + j] * a[8 + j < NCOL ? 8 + j : 0] : ov[8 + j];
                    }
                    tmem_st8(oaddr, lo);
                    if (NCOL > 8) tmem_st8(oaddr + 8, hi);
                }
                // red[] is rewritten only in a later rare path, after the next vote.
            }
            float pr[kNPad];
#pragma unroll
            for (int g = 0; g < kNPad; ++g) pr[g] = 0.f;
#pragma unroll
            for (int j = 0; j < NCOL; ++j) {
                if ((j % CW) >= NC) continue;              // padding column: weight 0
                if constexpr (MQ) pr[j] = s2[j] != -INFINITY ? fast_exp2(s2[j] - m_ref[j]) : 0.f;
                else pr[j] = valid ? fast_exp2(s2[j] - m_ref[j]) : 0.f;
            }
            uint32_t packed[kNPad / 2];
#pragma unroll
            for (int gp = 0; gp < kNPad / 2; ++gp) packed[gp] = pack_bf16x2(pr[2 * gp], pr[2 * gp + 1]);
            // The denominator sums the bf16 weights the MMA actually applies.
#pragma unroll
            for (int j = 0; j < NCOL; ++j)
                l_run[j] += (j & 1) ? bf16_hi(packed[j >> 1]) : bf16_lo(packed[j >> 1]);
            // P buffer sb is free once P.V of tile i-2 is done.
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->o_full[sb]), ((i >> 1) & 1) ^ 1, &misc->never,
                                                   lim))) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
            // Rows of masked tokens are zeroed once this tile's V has landed.
            if (__any_sync(0xffffffffu, !valid) &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->vfull[st]), (i / kStages) & 1, &misc->never,
                                                   lim))) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
            if (!valid) {
                // The MMA multiplies every V row by its probability; rows of
                // masked tokens may hold stale or non-finite bits, so zero them.
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(stage_ptr + st * kStageBytes + kVOff + (row >> 3) * kAtomStride +
                                                            ch * 1024 + (row & 7) * 128);
#pragma unroll
                    for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0, 0, 0, 0);
                }
            }
            uint8_t *prow = p_ptr + sb * kPBytes + (row >> 3) * 256 + (row & 7) * 16;
            *reinterpret_cast<uint4 *>(prow) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4 *>(prow + 128) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&misc->p_full[sb]));

            // The previous segment's read-out, one tile late.
            if (pending && !finalize()) {
                misc->abort = 1;
                set_error(p.err, PK_DEVERR_TIMEOUT);
                break;
            }
            if (seg_last) {
                pending = true;
                pend_seg = seg;
                pend_s = mt.x;
                pend_q0 = qm.x;
                pend_qn = qm.y;
                pend_h = mt.y;
                pend_i = i;
                pend_t0 = seg_t0;
                pend_i0 = seg_i0;
                pend_complete = seg_t0 == 0 && mt.z == mt.w - 1;
                pend_cut_end = mt.z == mt.w - 1;
#pragma unroll
                for (int j = 0; j < NCOL; ++j) {
                    m_prev[j] = m_ref[j];
                    l_prev[j] = l_run[j];
                }
                if (i == n_tiles - 1 && !finalize()) {
                    misc->abort = 1;
                    set_error(p.err, PK_DEVERR_TIMEOUT);
                    break;
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

// One CTA per decode CTA c: if c's first segment was cut at its start and
// ends in c, combine the parts of that segment from every CTA it spans.
// Thread r handles O^T row r (as the decode kernel's TMEM lanes).
template <int D, int NC, int HP>
__global__ void __launch_bounds__(128)
decode_tc_merge_kernel(const DecodeParams p, int C) {
    constexpr int CW = HP == 2 ? 8 : kNPad;
    // A decode grid launched next in the stream as this grid's programmatic
    // dependent may begin its set-up (before this grid completes it reads
    // only the sequence lengths, and reads them again afterwards).  Its CTAs
    // find room only as this decode grid's CTAs leave their SMs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the decode grid: wait for it
    // to finish and its writes to be visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const Slot *slots = static_cast<const Slot *>(p.tc_slots);
    const int c = blockIdx.x;
    const int row = threadIdx.x;
    const int hr = HP == 2 ? row >> 6 : 0;           // head of the pair (HP == 2)
    const int dd = HP == 2 ? (row & 63) : row;       // head-dim element
    const bool row_ok = HP == 2 || row < D;
    const int orow = row_ok ? row : 0;
    const Slot *mine = slots + 2 * c;
    // Everything the common case needs (this CTA's slot 0 and both slots of
    // CTA c - 1) is loaded at once, before the flag is known.
    const Slot *q0 = slots + 2 * (c > 0 ? c - 1 : c);
    const Slot *q1 = q0 + 1;
    const int flag = mine->flag;
    const int s = mine->s, h = mine->h;
    const int64_t start = mine->start_tile, T = mine->total_tiles;
    const int ca = mine->first_cta;
    const int64_t beg_prev = q0->range_beg;
    float mm[NC], ml[NC], mo[NC], am[NC], al[NC], ao[NC], bm[NC], bl[NC], bo[NC];
#pragma unroll
    for (int cq = 0; cq < NC; ++cq) {
        const int j = hr * CW + cq;
        mm[cq] = mine->m[j];
        ml[cq] = mine->l[j];
        mo[cq] = mine->o[j * 128 + orow];
        am[cq] = q0->m[j];
        al[cq] = q0->l[j];
        ao[cq] = q0->o[j * 128 + orow];
        bm[cq] = q1->m[j];
        bl[cq] = q1->l[j];
        bo[cq] = q1->o[j * 128 + orow];
    }
    if (flag != 1 || !row_ok) return;
    // First tile of CTA cc's range (the decode grid wrote it into slot 0).
    auto range_beg = [&](int cc) -> int64_t { return cc < C ? slots[2 * cc].range_beg : T; };
    float num[NC], den[NC];
    if (ca == c - 1) {
        // Two parts: CTA c - 1 (slot 0 if the segment is its first, else 1) and this CTA.
        const bool first_of_prev = beg_prev >= start;
#pragma unroll
        for (int cq = 0; cq < NC; ++cq) {
            const float pm = first_of_prev ? am[cq] : bm[cq];
            const float pl = first_of_prev ? al[cq] : bl[cq];
            const float po = first_of_prev ? ao[cq] : bo[cq];
            const float M = fmaxf(pm, mm[cq]);
            const float a0 = rescale(pm, M), a1 = rescale(mm[cq], M);
            den[cq] = a0 * pl + a1 * ml[cq];
            num[cq] = a0 * po + a1 * mo[cq];
        }
    } else {
        // Contributors are the CTAs from ca to c with a non-empty range (when
        // the grid has more CTAs than tiles, some ranges are empty and hold
        // no slot).
        float M[NC];
#pragma unroll
        for (int cq = 0; cq < NC; ++cq) M[cq] = -INFINITY;
        for (int cc = ca; cc <= c; ++cc) {
            if (range_beg(cc) == range_beg(cc + 1)) continue;
            const Slot *sl = slots + 2 * cc + (range_beg(cc) >= start ? 0 : 1);
#pragma unroll
            for (int cq = 0; cq < NC; ++cq) M[cq] = fmaxf(M[cq], sl->m[hr * CW + cq]);
        }
#pragma unroll
        for (int cq = 0; cq < NC; ++cq) num[cq] = den[cq] = 0.f;
        for (int cc = ca; cc <= c; ++cc) {
            if (range_beg(cc) == range_beg(cc + 1)) continue;
            const Slot *sl = slots + 2 * cc + (range_beg(cc) >= start ? 0 : 1);
#pragma unroll
            for (int cq = 0; cq < NC; ++cq) {
                const int j = hr * CW + cq;
                const float a = rescale(sl->m[j], M[cq]);
                den[cq] = fmaf(a, sl->l[j], den[cq]);
                num[cq] = fmaf(a, sl->o[j * 128 + row], num[cq]);
            }
        }
    }
    // Column cq: query token cq / G of the sequence, query head cq % G of
    // this row's KV head (as in the decode kernel).
    const int Gq = p.num_heads / p.num_kv_heads, lgG = __ffs(Gq) - 1;
    const int q0row = p.cu_q_lens ? p.cu_q_lens[s] : s;
    const int qn = p.cu_q_lens ? p.cu_q_lens[s + 1] - q0row : 1;
#pragma unroll
    for (int cq = 0; cq < NC; ++cq) {
        if ((cq >> lgG) >= qn) continue;
        const int qh = (h * HP + hr) * Gq + (cq & (Gq - 1));
        store_out(p, (static_cast<size_t>(q0row + (cq >> lgG)) * p.num_heads + qh) * D + dd,
                  den[cq] > 0.f ? num[cq] / den[cq] : 0.f);
    }
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

// K or V pages (L2 fetches the 128-byte pieces the box is made of: with
// 256-byte promotion the calls took 0.3 % longer) -- one box per (page,
// group of HP adjacent KV heads) holding
// its B rows as B / 8 blocks of 8 rows, each block [chunk][8 rows][64] in
// shared memory (dimensions: 64 elements; row within the block; 128-byte
// chunk of the group's row -- a 64-element half of the head, or (HP = 2,
// head dim 64) one head of the pair; 8-row block, numbered page * B / 8 +
// block; KV head group).
bool encode_page_map(CUtensorMap *m, const void *base, const DecodeParams &p, int hp) {
    auto enc = get_encoder();
    if (!enc) return false;
    const cuuint64_t D = p.head_dim, Hkv = p.num_kv_heads, B = p.block_size, HP = hp;
    const cuuint64_t P = p.num_blocks > 0 ? p.num_blocks : 1;
    cuuint64_t dims[5] = {64, 8, D * HP / 64, P * (B / 8), Hkv / HP};
    cuuint64_t strides[4] = {Hkv * D * 2, 128, 8 * Hkv * D * 2, HP * D * 2};
    cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(D * HP / 64), static_cast<cuuint32_t>(B / 8), 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap *m, const DecodeParams &p) {
    auto enc = get_encoder();
    if (!enc) return false;
    if (p.cu_q_lens) {
        // [total_q, H, D] queries; box (64 elements, G heads, q_len tokens):
        // MMA column r * G + g = query token r, head g of the group.
        const int G = p.num_heads / p.num_kv_heads;
        cuuint64_t dims3[3] = {static_cast<cuuint64_t>(p.head_dim), static_cast<cuuint64_t>(p.num_heads),
                               static_cast<cuuint64_t>(p.total_q > 0 ? p.total_q : 1)};
        cuuint64_t strides3[2] = {static_cast<cuuint64_t>(p.head_dim) * 2,
                                  static_cast<cuuint64_t>(p.head_dim) * p.num_heads * 2};
        cuuint32_t box3[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(p.q_len)};
        cuuint32_t estr3[3] = {1, 1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(p.q), dims3, strides3, box3,
                   estr3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.head_dim),
                          static_cast<cuuint64_t>(p.num_seqs) * p.num_heads};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.head_dim) * 2};
    cuuint32_t box[2] = {64, kNPad};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p.q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int NC, int HP>
cudaError_t launch_dg(const DecodeParams &p, int C, cudaStream_t stream) {
    CUtensorMap mk, mv, mq;
    if (!encode_page_map(&mk, p.k_cache, p, HP) || !encode_page_map(&mv, p.v_cache, p, HP) || !encode_q_map(&mq, p))
        return cudaErrorInvalidValue;
    {
        const cudaError_t e = p.cu_q_lens
            ? set_max_dynamic_smem(reinterpret_cast<const void *>(decode_tc_kernel<D, NC, true, HP>),
                                   static_cast<int>(kSmemBytes))
            : set_max_dynamic_smem(reinterpret_cast<const void *>(decode_tc_kernel<D, NC, false, HP>),
                                   static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = p.cu_q_lens ? cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NC, true, HP>, mk, mv, mq, p)
                                      : cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NC, false, HP>, mk, mv, mq, p);
    if (e != cudaSuccess) return e;
    if (!p.tc_slots) return cudaSuccess;   // no sequence longer than one tile: nothing is cut
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, decode_tc_merge_kernel<D, NC, HP>, p, C);
}

// Head dim 64 with at most 8 columns per KV head and an even number of KV
// heads: tiles of two adjacent KV heads (256-byte page rows).
template <int NC>
cudaError_t launch_d64(const DecodeParams &p, int C, cudaStream_t stream) {
    if constexpr (NC <= 8) {
        if (p.num_kv_heads % 2 == 0) return launch_dg<64, NC, 2>(p, C, stream);
    }
    return launch_dg<64, NC, 1>(p, C, stream);
}

cudaError_t launch_any(const DecodeParams &p, int C, cudaStream_t stream) {
    // MMA columns: the group's query heads times the query tokens per sequence.
    const int nc = (p.num_heads / p.num_kv_heads) * (p.cu_q_lens ? p.q_len : 1);
    if (p.head_dim == 64) {
        switch (nc) {
            case 1: return launch_d64<1>(p, C, stream);
            case 2: return launch_d64<2>(p, C, stream);
            case 4: return launch_d64<4>(p, C, stream);
            case 8: return launch_d64<8>(p, C, stream);
            case 16: return launch_d64<16>(p, C, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (nc) {
        case 1: return launch_dg<128, 1, 1>(p, C, stream);
        case 2: return launch_dg<128, 2, 1>(p, C, stream);
        case 4: return launch_dg<128, 4, 1>(p, C, stream);
        case 8: return launch_dg<128, 8, 1>(p, C, stream);
        case 16: return launch_dg<128, 16, 1>(p, C, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t tc_workspace_bytes() { return 2 * kMaxCtas * sizeof(Slot); }

cudaError_t launch_decode_tensor_core(const DecodeParams &p, cudaStream_t stream) {
    int C = sm_count();
    if (C <= 0) return cudaErrorNoDevice;
    if (C > static_cast<int>(kMaxCtas)) C = static_cast<int>(kMaxCtas);
    return launch_any(p, C, stream);
}

}  // namespace pk

namespace pk {

size_t tc_slot_bytes() { return sizeof(Slot); }

cudaError_t launch_multi_query_tensor_core(const DecodeParams &p, cudaStream_t stream) {
    const int G = p.num_heads / p.num_kv_heads;
    if (!p.cu_q_lens || p.q_len < 1 || (p.q_len & (p.q_len - 1)) || G * p.q_len > kNPad)
        return cudaErrorInvalidValue;
    return launch_decode_tensor_core(p, stream);
}

cudaError_t launch_decode_tensor_core_grid(const DecodeParams &p, cudaStream_t stream, int ctas) {
    if (ctas <= 0 || ctas > static_cast<int>(kMaxCtas)) return cudaErrorInvalidValue;
    return launch_any(p, ctas, stream);
}

}  // namespace pk
