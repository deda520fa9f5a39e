// Host block manager: free list, block tables, reference counts and the
// copy-on-write decisions of a decode step (C ABI in
// include/pagedkv_block_manager.h, where the rules and their sources are
// listed).
//
// Layout.  The free list is a ring over block ids (take from the front,
// return to the back, and -- only to undo a failed batch -- push back onto
// the front), reference counts are one int32 per block, and each sequence
// keeps its table as a vector of block ids.  An append costs O(1); a batch
// that fails half way is undone from a journal so that every call is all or
// nothing.
#include "pagedkv_block_manager.h"

#include <climits>
#include <cstring>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

struct pk_block_manager {
    struct Seq {
        std::vector<int32_t> table;
        int64_t length = 0;
    };

    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> ring;      // free block ids: ring[head], ring[head + 1], ... (count of them)
    int64_t head = 0;
    int64_t count = 0;
    std::vector<int32_t> ref;       // reference count per block (0 = free)
    std::unordered_map<int64_t, Seq> seqs;
    std::vector<int64_t> copies;    // queued (src, dst) pairs, flattened

    int32_t take() {
        const int32_t b = ring[head];
        head = head + 1 == num_blocks ? 0 : head + 1;
        --count;
        ref[b] = 1;
        return b;
    }
    void give_back(int32_t b) {      // to the back of the free list
        int64_t at = head + count;
        if (at >= num_blocks) at -= num_blocks;
        ring[at] = b;
        ++count;
    }
    void untake(int32_t b) {         // exact inverse of take()
        head = head == 0 ? num_blocks - 1 : head - 1;
        ring[head] = b;
        ++count;
        ref[b] = 0;
    }
    void drop(int32_t b) {
        if (--ref[b] == 0) give_back(b);
    }
};

namespace {

// What one append did, so a failed batch can be undone.
struct Undo {
    pk_block_manager::Seq *seq;
    int kind;          // 0 in place, 1 new block, 2 copy-on-write
    int32_t old_block; // kind 2: the shared block that was replaced
};

// Room for one more entry in a table, allocated before a block is taken so
// that nothing can throw between taking a block and recording it.
bool reserve_one(std::vector<int32_t> &v) {
    if (v.size() < v.capacity()) return true;
    try {
        v.reserve(v.empty() ? 8 : 2 * v.capacity());
        return true;
    } catch (...) {
        return false;
    }
}

template <typename F>
int guarded(F &&f) {
    try {
        return f();
    } catch (const std::bad_alloc &) {
        return PK_ERR_HOST_MEMORY;
    } catch (...) {
        return PK_ERR_HOST_MEMORY;
    }
}

}  // namespace

extern "C" pk_block_manager *pk_bm_create(int num_blocks, int block_size) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    try {
        auto *bm = new pk_block_manager();
        bm->num_blocks = num_blocks;
        bm->block_size = block_size;
        bm->ring.resize(num_blocks);
        for (int i = 0; i < num_blocks; ++i) bm->ring[i] = i;
        bm->count = num_blocks;
        bm->ref.assign(num_blocks, 0);
        return bm;
    } catch (...) {
        return nullptr;
    }
}

extern "C" void pk_bm_destroy(pk_block_manager *bm) { delete bm; }

extern "C" int pk_bm_add_sequence(pk_block_manager *bm, int64_t seq_id) {
    if (!bm) return PK_ERR_NULL;
    return guarded([&] {
        if (bm->seqs.count(seq_id)) return static_cast<int>(PK_ERR_SEQUENCE_EXISTS);
        bm->seqs.emplace(seq_id, pk_block_manager::Seq{});
        return static_cast<int>(PK_OK);
    });
}

extern "C" int pk_bm_append_slots(pk_block_manager *bm, const int64_t *seq_ids, int n, int64_t *slots_out) {
    if (!bm) return PK_ERR_NULL;
    if (n < 0) return PK_ERR_SHAPE;
    if (n == 0) return PK_OK;
    if (!seq_ids || !slots_out) return PK_ERR_NULL;
    return guarded([&] {
        std::vector<Undo> journal;
        journal.reserve(static_cast<size_t>(n));
        std::vector<int64_t> slots(static_cast<size_t>(n));
        const size_t copies0 = bm->copies.size();
        bm->copies.reserve(copies0 + 2 * static_cast<size_t>(n));   // no allocation once blocks move
        int status = PK_OK;
        for (int i = 0; i < n; ++i) {
            auto it = bm->seqs.find(seq_ids[i]);
            if (it == bm->seqs.end()) {
                status = PK_ERR_UNKNOWN_SEQUENCE;
                break;
            }
            pk_block_manager::Seq &sq = it->second;
            const int64_t off = sq.length % bm->block_size;
            Undo u{&sq, 0, -1};
            if (off == 0) {                                    // the token starts a new block
                if (bm->count == 0) {
                    status = PK_ERR_NO_BLOCKS;
                    break;
                }
                if (!reserve_one(sq.table)) {                  // undone below like any failure
                    status = PK_ERR_HOST_MEMORY;
                    break;
                }
                sq.table.push_back(bm->take());
                u.kind = 1;
            } else if (bm->ref[sq.table.back()] > 1) {        // shared last block: copy on write
                if (bm->count == 0) {
                    status = PK_ERR_NO_BLOCKS;
                    break;
                }
                const int32_t old = sq.table.back();
                const int32_t fresh = bm->take();
                bm->copies.push_back(old);
                bm->copies.push_back(fresh);
                --bm->ref[old];                                // still >= 1: another sequence holds it
                sq.table.back() = fresh;
                u.kind = 2;
                u.old_block = old;
            }
            ++sq.length;
            slots[static_cast<size_t>(i)] = static_cast<int64_t>(sq.table.back()) * bm->block_size + off;
            journal.push_back(u);
        }
        if (status != PK_OK) {
            // Undo in reverse order: every take() is returned to the front.
            for (size_t k = journal.size(); k-- > 0;) {
                const Undo &u = journal[k];
                --u.seq->length;
                if (u.kind == 1) {
                    const int32_t b = u.seq->table.back();
                    u.seq->table.pop_back();
                    bm->untake(b);
                } else if (u.kind == 2) {
                    const int32_t b = u.seq->table.back();
                    u.seq->table.back() = u.old_block;
                    ++bm->ref[u.old_block];
                    bm->untake(b);
                }
            }
            bm->copies.resize(copies0);
            return status;
        }
        std::memcpy(slots_out, slots.data(), sizeof(int64_t) * static_cast<size_t>(n));
        return static_cast<int>(PK_OK);
    });
}

extern "C" int pk_bm_fork(pk_block_manager *bm, int64_t parent, int64_t child, int64_t num_tokens) {
    if (!bm) return PK_ERR_NULL;
    return guarded([&] {
        auto pit = bm->seqs.find(parent);
        if (pit == bm->seqs.end()) return static_cast<int>(PK_ERR_UNKNOWN_SEQUENCE);
        if (bm->seqs.count(child)) return static_cast<int>(PK_ERR_SEQUENCE_EXISTS);
        const pk_block_manager::Seq &ps = pit->second;
        pk_block_manager::Seq cs;
        size_t nb;
        if (num_tokens == -1) {                 // the whole parent, partial last block included
            cs.length = ps.length;
            nb = ps.table.size();
        } else {
            if (num_tokens < 0 || num_tokens > ps.length || num_tokens % bm->block_size != 0)
                return static_cast<int>(PK_ERR_SHAPE);
            cs.length = num_tokens;
            nb = static_cast<size_t>(num_tokens / bm->block_size);
        }
        cs.table.assign(ps.table.begin(), ps.table.begin() + static_cast<std::ptrdiff_t>(nb));
        bm->seqs.emplace(child, std::move(cs));  // may throw: counts are touched only after it
        for (size_t j = 0; j < nb; ++j) ++bm->ref[ps.table[j]];
        return static_cast<int>(PK_OK);
    });
}

extern "C" int pk_bm_free_sequence(pk_block_manager *bm, int64_t seq_id) {
    if (!bm) return PK_ERR_NULL;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQUENCE;
    for (int32_t b : it->second.table) bm->drop(b);
    bm->seqs.erase(it);
    return PK_OK;
}

extern "C" int pk_bm_num_pending_copies(const pk_block_manager *bm) {
    if (!bm) return PK_ERR_NULL;
    return static_cast<int>(bm->copies.size() / 2);
}

extern "C" int pk_bm_take_copies(pk_block_manager *bm, int64_t *pairs_out, int max_pairs, int *num_out) {
    if (!bm || !num_out) return PK_ERR_NULL;
    const int pending = static_cast<int>(bm->copies.size() / 2);
    *num_out = pending;
    if (pending > max_pairs) return PK_ERR_SHAPE;
    if (pending > 0) {
        if (!pairs_out) return PK_ERR_NULL;
        std::memcpy(pairs_out, bm->copies.data(), sizeof(int64_t) * bm->copies.size());
    }
    bm->copies.clear();
    return PK_OK;
}

extern "C" int pk_bm_export(const pk_block_manager *bm, const int64_t *seq_ids, int n, int32_t *block_tables,
                            int max_blocks, int32_t *seq_lens) {
    if (!bm) return PK_ERR_NULL;
    if (n < 0 || max_blocks < 0) return PK_ERR_SHAPE;
    if (n == 0) return PK_OK;
    if (!seq_ids || !seq_lens || (max_blocks > 0 && !block_tables)) return PK_ERR_NULL;
    std::vector<const pk_block_manager::Seq *> found(static_cast<size_t>(n));
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQUENCE;
        if (it->second.table.size() > static_cast<size_t>(max_blocks) || it->second.length > INT32_MAX)
            return PK_ERR_SHAPE;
        found[static_cast<size_t>(i)] = &it->second;
    }
    for (int i = 0; i < n; ++i) {
        const pk_block_manager::Seq &sq = *found[static_cast<size_t>(i)];
        int32_t *row = block_tables + static_cast<size_t>(i) * static_cast<size_t>(max_blocks);
        const size_t nb = sq.table.size();
        if (nb) std::memcpy(row, sq.table.data(), sizeof(int32_t) * nb);
        for (size_t j = nb; j < static_cast<size_t>(max_blocks); ++j) row[j] = -1;
        seq_lens[i] = static_cast<int32_t>(sq.length);
    }
    return PK_OK;
}

extern "C" int pk_bm_sequence_info(const pk_block_manager *bm, int64_t seq_id, int64_t *length_out,
                                   int *num_blocks_out) {
    if (!bm) return PK_ERR_NULL;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PK_ERR_UNKNOWN_SEQUENCE;
    if (length_out) *length_out = it->second.length;
    if (num_blocks_out) *num_blocks_out = static_cast<int>(it->second.table.size());
    return PK_OK;
}

extern "C" int pk_bm_num_free_blocks(const pk_block_manager *bm) {
    if (!bm) return PK_ERR_NULL;
    return static_cast<int>(bm->count);
}

extern "C" int pk_bm_blocks_in_use(const pk_block_manager *bm) {
    if (!bm) return PK_ERR_NULL;
    return static_cast<int>(bm->num_blocks - bm->count);
}
