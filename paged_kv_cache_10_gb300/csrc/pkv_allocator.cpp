// pkv_allocator.cpp -- host block allocator (free list, reference counts,
// fork / append with copy-on-write / free).  Host memory only.
//
// "vLLM：大语言模型推理与服务库" section 4.2 ("Block Pool"): the pool is split
// into fixed-size blocks tracked by a free list; allocation takes the last
// free id in O(1) and fails when none is left; freeing pushes the id back.
// Section 4.3: a sequence receives a block only when its last block is full.
// "vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望", section
// "束搜索与并行采样的三大调度原语": fork shares the parent's physical blocks;
// append gives the writer a private copy of a shared block (copy-on-write);
// free drops reference counts and returns zero-count blocks immediately.
// "vLLM 深度解析：从 PagedAttention 到生产部署", "Prefix Caching 与
// Copy-on-Write": shared blocks have reference count > 1 and are copied only
// when modified.
//
// Automatic prefix caching ("vLLM 高性能大语言模型推理引擎深度技术评估与分布式
// 架构展望", sections "基于级联哈希的缓存结构设计" and "缓存分配、触碰与驱逐闭环"):
// a full block may be committed under its cascaded hash (parent hash, the
// block's tokens, extra hashes; the cache salt enters the first block's
// hash).  Lookup finds the longest run of leading blocks of a new prompt
// that are already in the table; touch takes a reference on them (reviving
// blocks no sequence holds any more); blocks whose count drops to zero keep
// their hash and stay cached but evictable; allocation uses never-cached
// free blocks first and then evicts the least recently released cached
// block.  A sequence releases its blocks last to first, so of the blocks
// freed together the leaf end of the chain goes first and the shared root
// (a system prompt, say) stays longest.
//
// Every public call is all-or-nothing: failures leave the state unchanged
// (OOM returns a status instead of throwing).
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <map>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
};

}  // namespace

struct pkv_alloc {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free_stack;  // never-cached free blocks; allocation pops the back
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Seq> seqs;
    int64_t fail_countdown = 0;  // >0: the fail_countdown-th allocation fails
    // prefix cache
    std::vector<uint64_t> bhash;           // hash of a committed block
    std::vector<uint8_t> hashed;           // 1: committed (in `table`)
    std::vector<int64_t> stamp;            // release stamp of an evictable block; -1 otherwise
    std::vector<int64_t> took_stamp;       // stamp of the cached block a take() evicted; -1 otherwise
    std::unordered_map<uint64_t, int32_t> table;  // hash -> block
    std::map<int64_t, int32_t> evictable;  // release stamp -> cached block with count 0
    int64_t clock = 0;

    int64_t available() const { return static_cast<int64_t>(free_stack.size() + evictable.size()); }
    bool can_take() {
        if (fail_countdown > 0) {
            if (fail_countdown == 1) {
                fail_countdown = 0;
                return false;
            }
        }
        return available() > 0;
    }
    // Only call after can_take() returned true.  Never-cached blocks first;
    // else the least recently released cached block is evicted.
    int32_t take() {
        if (fail_countdown > 0) --fail_countdown;
        int32_t id;
        if (!free_stack.empty()) {
            id = free_stack.back();
            free_stack.pop_back();
            took_stamp[id] = -1;
        } else {
            auto it = evictable.begin();
            id = it->second;
            took_stamp[id] = it->first;
            evictable.erase(it);
            stamp[id] = -1;
            table.erase(bhash[id]);
            hashed[id] = 0;
        }
        ref[id] = 1;
        return id;
    }
    // Exact inverse of take() for rollback (takes are undone last first).
    void untake(int32_t id) {
        ref[id] = 0;
        if (took_stamp[id] < 0) {
            free_stack.push_back(id);
        } else {
            hashed[id] = 1;
            table[bhash[id]] = id;
            stamp[id] = took_stamp[id];
            evictable.emplace(took_stamp[id], id);
            took_stamp[id] = -1;
        }
    }
    void release(int32_t id) {
        if (--ref[id] == 0) {
            if (hashed[id]) {
                stamp[id] = clock++;
                evictable.emplace(stamp[id], id);
            } else {
                free_stack.push_back(id);
            }
        }
    }
    // Reference on a block found by lookup; revives it if it was evictable.
    void touch(int32_t id) {
        if (ref[id] == 0) {
            evictable.erase(stamp[id]);
            stamp[id] = -1;
        }
        ref[id] += 1;
    }
};

namespace {

// Record of one append_slot, enough to undo it exactly.
struct AppendUndo {
    int64_t seq;
    int kind;  // 0: wrote in place, 1: took a fresh block, 2: copy-on-write
    int32_t src, dst;
};

pkv_status append_one(pkv_alloc* a, int64_t seq_id, int64_t* slot, int32_t* cs, int32_t* cd,
                      AppendUndo* undo) {
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    Seq& s = it->second;
    const int64_t pos = s.len;
    const int32_t off = static_cast<int32_t>(pos % a->block_size);
    int32_t src = -1, dst = -1;
    int kind = 0;
    if (off == 0) {
        if (!a->can_take()) return PKV_ERR_OOM;
        s.blocks.push_back(a->take());
        kind = 1;
    } else {
        const int32_t last = s.blocks.back();
        if (a->ref[last] > 1) {
            if (!a->can_take()) return PKV_ERR_OOM;
            dst = a->take();
            a->ref[last] -= 1;
            s.blocks.back() = dst;
            src = last;
            kind = 2;
        }
    }
    s.len = pos + 1;
    *slot = static_cast<int64_t>(s.blocks.back()) * a->block_size + off;
    if (cs) *cs = src;
    if (cd) *cd = dst;
    if (undo) *undo = AppendUndo{seq_id, kind, src, dst};
    return PKV_OK;
}

void undo_append(pkv_alloc* a, const AppendUndo& u) {
    Seq& s = a->seqs[u.seq];
    s.len -= 1;
    if (u.kind == 1) {
        a->untake(s.blocks.back());
        s.blocks.pop_back();
    } else if (u.kind == 2) {
        s.blocks.back() = u.src;
        a->ref[u.src] += 1;
        a->untake(u.dst);
    }
}

}  // namespace

extern "C" {

pkv_alloc* pkv_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pkv_alloc* a = new (std::nothrow) pkv_alloc();
    if (!a) return nullptr;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->bhash.assign(num_blocks, 0);
    a->hashed.assign(num_blocks, 0);
    a->stamp.assign(num_blocks, -1);
    a->took_stamp.assign(num_blocks, -1);
    a->free_stack.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t id = free_order[i];
            if (id < 0 || id >= num_blocks || seen[id]) {
                delete a;
                return nullptr;
            }
            seen[id] = 1;
            a->free_stack[i] = id;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[i] = i;
    }
    return a;
}

void pkv_alloc_destroy(pkv_alloc* a) { delete a; }

pkv_status pkv_alloc_seq_new(pkv_alloc* a, int64_t seq_id, int32_t num_tokens) {
    if (!a || num_tokens < 0) return PKV_ERR_INVALID;
    if (a->seqs.count(seq_id)) return PKV_ERR_INVALID;
    const int64_t need = (static_cast<int64_t>(num_tokens) + a->block_size - 1) / a->block_size;
    if (need > a->available()) return PKV_ERR_OOM;
    Seq s;
    s.blocks.reserve(need);
    for (int64_t i = 0; i < need; ++i) {
        if (!a->can_take()) {
            for (auto it = s.blocks.rbegin(); it != s.blocks.rend(); ++it) a->untake(*it);
            return PKV_ERR_OOM;
        }
        s.blocks.push_back(a->take());
    }
    s.len = num_tokens;
    a->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

pkv_status pkv_alloc_fork(pkv_alloc* a, int64_t parent_id, int64_t child_id) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(parent_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    if (a->seqs.count(child_id)) return PKV_ERR_INVALID;
    Seq child = it->second;
    for (int32_t id : child.blocks) a->ref[id] += 1;
    a->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

pkv_status pkv_alloc_append_slot(pkv_alloc* a, int64_t seq_id, int64_t* slot, int32_t* cow_src,
                                 int32_t* cow_dst) {
    if (!a || !slot) return PKV_ERR_INVALID;
    return append_one(a, seq_id, slot, cow_src, cow_dst, nullptr);
}

pkv_status pkv_alloc_seq_extend(pkv_alloc* a, int64_t seq_id, int32_t num_tokens) {
    if (!a || num_tokens < 0) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    Seq& s = it->second;
    if (num_tokens == 0) return PKV_OK;
    if (s.len % a->block_size != 0 && a->ref[s.blocks.back()] > 1) return PKV_ERR_INVALID;
    const int64_t have = static_cast<int64_t>(s.blocks.size());
    const int64_t need = (s.len + num_tokens + a->block_size - 1) / a->block_size - have;
    if (need > a->available()) return PKV_ERR_OOM;
    for (int64_t i = 0; i < need; ++i) {
        if (!a->can_take()) {
            while (static_cast<int64_t>(s.blocks.size()) > have) {
                a->untake(s.blocks.back());
                s.blocks.pop_back();
            }
            return PKV_ERR_OOM;
        }
        s.blocks.push_back(a->take());
    }
    s.len += num_tokens;
    return PKV_OK;
}

pkv_status pkv_alloc_free(pkv_alloc* a, int64_t seq_id) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    const std::vector<int32_t>& bl = it->second.blocks;
    for (auto r = bl.rbegin(); r != bl.rend(); ++r) a->release(*r);
    a->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_alloc_append_batch(pkv_alloc* a, const int64_t* seq_ids, int32_t n, int64_t* slots,
                                  int32_t* pairs, int32_t pairs_cap, int32_t* num_pairs) {
    if (!a || n < 0 || (n > 0 && (!seq_ids || !slots)) || !num_pairs) return PKV_ERR_INVALID;
    if (pairs_cap < n || (n > 0 && !pairs)) return PKV_ERR_INVALID;
    // A sequence may appear at most once per batch.
    {
        std::unordered_map<int64_t, int> seen;
        for (int32_t i = 0; i < n; ++i)
            if (seq_ids[i] >= 0 && seen[seq_ids[i]]++) return PKV_ERR_INVALID;
    }
    std::vector<AppendUndo> undo;
    undo.reserve(n);
    int32_t np = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (seq_ids[i] < 0) {
            slots[i] = -1;
            continue;
        }
        int32_t cs = -1, cd = -1;
        AppendUndo u{};
        pkv_status st = append_one(a, seq_ids[i], &slots[i], &cs, &cd, &u);
        if (st != PKV_OK) {
            for (auto r = undo.rbegin(); r != undo.rend(); ++r) undo_append(a, *r);
            return st;
        }
        undo.push_back(u);
        if (cs >= 0) {
            pairs[2 * np] = cs;
            pairs[2 * np + 1] = cd;
            ++np;
        }
    }
    *num_pairs = np;
    return PKV_OK;
}

pkv_status pkv_alloc_append_tokens(pkv_alloc* a, const int64_t* seq_ids, const int32_t* counts, int32_t n,
                                   int64_t* slots, int64_t slots_cap, int32_t* pairs, int32_t pairs_cap,
                                   int32_t* num_pairs) {
    if (!a || n < 0 || (n > 0 && (!seq_ids || !counts)) || !num_pairs) return PKV_ERR_INVALID;
    if (pairs_cap < n || (n > 0 && !pairs)) return PKV_ERR_INVALID;
    int64_t total = 0;
    {
        std::unordered_map<int64_t, int> seen;
        for (int32_t i = 0; i < n; ++i) {
            if (counts[i] < 0 || seq_ids[i] < 0 || seen[seq_ids[i]]++) return PKV_ERR_INVALID;
            total += counts[i];
        }
    }
    if (total > slots_cap || (total > 0 && !slots)) return PKV_ERR_INVALID;
    std::vector<AppendUndo> undo;
    undo.reserve(static_cast<size_t>(total));
    int32_t np = 0;
    int64_t k = 0;
    for (int32_t i = 0; i < n; ++i) {
        for (int32_t t = 0; t < counts[i]; ++t, ++k) {
            int32_t cs = -1, cd = -1;
            AppendUndo u{};
            pkv_status st = append_one(a, seq_ids[i], &slots[k], &cs, &cd, &u);
            if (st != PKV_OK) {
                for (auto r = undo.rbegin(); r != undo.rend(); ++r) undo_append(a, *r);
                return st;
            }
            undo.push_back(u);
            if (cs >= 0) {  // only a sequence's first new token can meet a shared partial block
                pairs[2 * np] = cs;
                pairs[2 * np + 1] = cd;
                ++np;
            }
        }
    }
    *num_pairs = np;
    return PKV_OK;
}

pkv_status pkv_alloc_export(const pkv_alloc* a, const int64_t* seq_ids, int32_t n, int32_t* tables,
                            int32_t max_blocks, int32_t* seq_lens) {
    if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !tables || !seq_lens)))
        return PKV_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) {
        if (seq_ids[i] < 0) continue;
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
        if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks) return PKV_ERR_INVALID;
        if (it->second.len > INT32_MAX) return PKV_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
        for (int32_t j = 0; j < max_blocks; ++j) row[j] = -1;
        seq_lens[i] = 0;
        if (seq_ids[i] < 0) continue;
        const Seq& s = a->seqs.find(seq_ids[i])->second;
        std::memcpy(row, s.blocks.data(), s.blocks.size() * sizeof(int32_t));
        seq_lens[i] = static_cast<int32_t>(s.len);
    }
    return PKV_OK;
}

pkv_status pkv_alloc_block_table(const pkv_alloc* a, int64_t seq_id, int32_t* out, int32_t cap,
                                 int32_t* n) {
    if (!a || !n || cap < 0) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    const auto& bl = it->second.blocks;
    *n = static_cast<int32_t>(bl.size());
    if (static_cast<int64_t>(bl.size()) > cap || (!out && !bl.empty())) return PKV_ERR_INVALID;
    if (!bl.empty()) std::memcpy(out, bl.data(), bl.size() * sizeof(int32_t));
    return PKV_OK;
}

pkv_status pkv_alloc_seq_len(const pkv_alloc* a, int64_t seq_id, int64_t* n) {
    if (!a || !n) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    *n = it->second.len;
    return PKV_OK;
}

int32_t pkv_alloc_refcount(const pkv_alloc* a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->ref[block];
}

int32_t pkv_alloc_num_free(const pkv_alloc* a) {
    return a ? static_cast<int32_t>(a->available()) : -1;
}

int32_t pkv_alloc_num_seqs(const pkv_alloc* a) {
    return a ? static_cast<int32_t>(a->seqs.size()) : -1;
}

pkv_status pkv_alloc_prefix_groups(const pkv_alloc* a, const int64_t* seq_ids, int32_t n, int32_t min_blocks,
                                   int32_t* seq_group, int32_t* group_blocks, int32_t* group_offsets,
                                   int32_t* group_members, int32_t* num_groups, int32_t* max_members,
                                   int32_t* max_blocks) {
    if (!a || n < 0 || min_blocks < 1 || !num_groups || !max_members || !max_blocks) return PKV_ERR_INVALID;
    if (n > 0 && (!seq_ids || !seq_group || !group_blocks || !group_offsets || !group_members)) return PKV_ERR_INVALID;
    std::vector<const Seq*> seqs(n, nullptr);
    for (int32_t i = 0; i < n; ++i) {
        if (seq_ids[i] < 0) continue;
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
        seqs[i] = &it->second;
    }
    // Bucket rows by their first block, in order of first appearance.
    std::vector<int32_t> order;
    std::unordered_map<int32_t, std::vector<int32_t>> buckets;
    for (int32_t i = 0; i < n; ++i) {
        seq_group[i] = -1;
        if (!seqs[i] || seqs[i]->len / a->block_size < min_blocks) continue;
        const int32_t first = seqs[i]->blocks[0];
        auto& b = buckets[first];
        if (b.empty()) order.push_back(first);
        b.push_back(i);
    }
    int32_t ng = 0, nm = 0, mm = 0, mb = 0;
    group_offsets[0] = 0;
    for (int32_t key : order) {
        const std::vector<int32_t>& rows = buckets[key];
        if (rows.size() < 2) continue;
        // longest common run of identical leading block ids, full blocks only
        int64_t lcp = seqs[rows[0]]->len / a->block_size;
        for (int32_t r : rows) lcp = std::min<int64_t>(lcp, seqs[r]->len / a->block_size);
        for (size_t k = 1; k < rows.size(); ++k) {
            const std::vector<int32_t>& x = seqs[rows[0]]->blocks;
            const std::vector<int32_t>& y = seqs[rows[k]]->blocks;
            int64_t j = 0;
            while (j < lcp && x[j] == y[j]) ++j;
            lcp = j;
        }
        if (lcp < min_blocks) continue;
        group_blocks[ng] = static_cast<int32_t>(lcp);
        for (int32_t r : rows) {
            seq_group[r] = ng;
            group_members[nm++] = r;
        }
        group_offsets[ng + 1] = nm;
        mm = std::max<int32_t>(mm, static_cast<int32_t>(rows.size()));
        mb = std::max<int32_t>(mb, static_cast<int32_t>(lcp));
        ++ng;
    }
    *num_groups = ng;
    *max_members = mm;
    *max_blocks = mb;
    return PKV_OK;
}

namespace {
// Moves seq_id from allocator `from` to allocator `to`: takes one block of
// `to` per block of the sequence, records (from_block, to_block) pairs,
// releases the `from` blocks.  Every block must be held by this sequence
// alone.  All or nothing.
pkv_status move_seq(pkv_alloc* from, pkv_alloc* to, int64_t seq_id, int32_t* pairs, int32_t cap, int32_t* n,
                    bool pairs_from_first) {
    if (!from || !to || !n || cap < 0 || from == to) return PKV_ERR_INVALID;
    if (from->block_size != to->block_size) return PKV_ERR_INVALID;
    auto it = from->seqs.find(seq_id);
    if (it == from->seqs.end()) return PKV_ERR_NOT_FOUND;
    if (to->seqs.count(seq_id)) return PKV_ERR_INVALID;
    const Seq& s = it->second;
    const int32_t nb = static_cast<int32_t>(s.blocks.size());
    if (nb > cap || (nb > 0 && !pairs)) return PKV_ERR_INVALID;
    for (int32_t b : s.blocks)
        if (from->ref[b] != 1) return PKV_ERR_INVALID;  // shared blocks cannot move
    if (nb > to->available()) return PKV_ERR_OOM;
    Seq moved;
    moved.len = s.len;
    for (int32_t i = 0; i < nb; ++i) {
        if (!to->can_take()) {
            for (auto r = moved.blocks.rbegin(); r != moved.blocks.rend(); ++r) to->untake(*r);
            return PKV_ERR_OOM;
        }
        moved.blocks.push_back(to->take());
    }
    for (int32_t i = 0; i < nb; ++i) {
        pairs[2 * i] = pairs_from_first ? s.blocks[i] : moved.blocks[i];
        pairs[2 * i + 1] = pairs_from_first ? moved.blocks[i] : s.blocks[i];
    }
    for (auto r = s.blocks.rbegin(); r != s.blocks.rend(); ++r) from->release(*r);
    from->seqs.erase(it);
    to->seqs.emplace(seq_id, std::move(moved));
    *n = nb;
    return PKV_OK;
}
}  // namespace

pkv_status pkv_alloc_swap_out(pkv_alloc* dev, pkv_alloc* host, int64_t seq_id, int32_t* pairs, int32_t cap,
                              int32_t* n) {
    return move_seq(dev, host, seq_id, pairs, cap, n, true);
}

pkv_status pkv_alloc_swap_in(pkv_alloc* dev, pkv_alloc* host, int64_t seq_id, int32_t* pairs, int32_t cap,
                             int32_t* n) {
    return move_seq(host, dev, seq_id, pairs, cap, n, false);
}

void pkv_alloc_fail_after(pkv_alloc* a, int64_t k) {
    if (a) a->fail_countdown = k > 0 ? k : 0;
}

// ------------------------------------------------------------ prefix cache
// FNV-1a, 64-bit (offset basis 14695981039346656037, prime 1099511628211),
// over little-endian bytes.
namespace {
struct Fnv {
    uint64_t h = 14695981039346656037ull;
    void byte(uint8_t b) {
        h ^= b;
        h *= 1099511628211ull;
    }
    void u32(uint32_t v) {
        for (int i = 0; i < 4; ++i) byte(static_cast<uint8_t>(v >> (8 * i)));
    }
    void u64(uint64_t v) {
        for (int i = 0; i < 8; ++i) byte(static_cast<uint8_t>(v >> (8 * i)));
    }
};
}  // namespace

uint64_t pkv_block_hash(uint64_t parent_hash, const int32_t* tokens, int32_t num_tokens, const uint64_t* extras,
                        int32_t num_extras) {
    Fnv f;
    f.u64(parent_hash);
    const int32_t nt = tokens && num_tokens > 0 ? num_tokens : 0;
    const int32_t ne = extras && num_extras > 0 ? num_extras : 0;
    f.u32(static_cast<uint32_t>(nt));
    for (int32_t i = 0; i < nt; ++i) f.u32(static_cast<uint32_t>(tokens[i]));
    f.u32(static_cast<uint32_t>(ne));
    for (int32_t i = 0; i < ne; ++i) f.u64(extras[i]);
    return f.h;
}

pkv_status pkv_prefix_block_hashes(const int32_t* tokens, int64_t num_tokens, int32_t block_size,
                                   const uint64_t* extras, int32_t num_extras, const uint64_t* salt,
                                   uint64_t* hashes, int64_t cap, int64_t* num_hashes) {
    if (num_tokens < 0 || block_size <= 0 || num_extras < 0 || (num_extras > 0 && !extras) || !num_hashes)
        return PKV_ERR_INVALID;
    const int64_t nb = num_tokens / block_size;
    if (nb > 0 && (!tokens || !hashes || cap < nb)) return PKV_ERR_INVALID;
    std::vector<uint64_t> ex(extras, extras + num_extras);
    uint64_t parent = 0;
    for (int64_t i = 0; i < nb; ++i) {
        if (i == 0 && salt) ex.push_back(*salt);
        hashes[i] = pkv_block_hash(parent, tokens + i * block_size, block_size, ex.data(),
                                   static_cast<int32_t>(ex.size()));
        if (i == 0 && salt) ex.pop_back();
        parent = hashes[i];
    }
    *num_hashes = nb;
    return PKV_OK;
}

int32_t pkv_alloc_lookup(const pkv_alloc* a, const uint64_t* hashes, int32_t n) {
    if (!a || n < 0 || (n > 0 && !hashes)) return -1;
    int32_t k = 0;
    while (k < n && a->table.count(hashes[k])) ++k;
    return k;
}

pkv_status pkv_alloc_seq_new_prefix(pkv_alloc* a, int64_t seq_id, const uint64_t* hashes, int32_t num_hashes,
                                    int32_t num_tokens, int32_t* hit_blocks) {
    if (!a || num_tokens < 0 || num_hashes < 0 || (num_hashes > 0 && !hashes) || !hit_blocks)
        return PKV_ERR_INVALID;
    if (a->seqs.count(seq_id)) return PKV_ERR_INVALID;
    if (static_cast<int64_t>(num_hashes) * a->block_size > num_tokens) return PKV_ERR_INVALID;  // full blocks only
    const int32_t k = pkv_alloc_lookup(a, hashes, num_hashes);
    const int64_t total = (static_cast<int64_t>(num_tokens) + a->block_size - 1) / a->block_size;
    const int64_t need = total - k;
    int64_t revived = 0;  // hits that leave the evictable set
    for (int32_t i = 0; i < k; ++i)
        if (a->ref[a->table.at(hashes[i])] == 0) ++revived;
    if (need > a->available() - revived) return PKV_ERR_OOM;
    if (a->fail_countdown > 0 && a->fail_countdown <= need) {  // the injected failure falls in this call
        a->fail_countdown = 0;
        return PKV_ERR_OOM;
    }
    Seq s;
    s.blocks.reserve(total);
    for (int32_t i = 0; i < k; ++i) {
        const int32_t id = a->table.at(hashes[i]);
        a->touch(id);
        s.blocks.push_back(id);
    }
    for (int64_t i = 0; i < need; ++i) s.blocks.push_back(a->take());
    s.len = num_tokens;
    a->seqs.emplace(seq_id, std::move(s));
    *hit_blocks = k;
    return PKV_OK;
}

pkv_status pkv_alloc_commit(pkv_alloc* a, int64_t seq_id, const uint64_t* hashes, int32_t num_hashes,
                            int32_t* committed) {
    if (!a || num_hashes < 0 || (num_hashes > 0 && !hashes)) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
    const Seq& s = it->second;
    if (static_cast<int64_t>(num_hashes) * a->block_size > s.len) return PKV_ERR_INVALID;  // full blocks only
    for (int32_t i = 0; i < num_hashes; ++i) {
        const int32_t id = s.blocks[i];
        if (a->hashed[id] && a->bhash[id] != hashes[i]) return PKV_ERR_INVALID;
    }
    int32_t c = 0;
    for (int32_t i = 0; i < num_hashes; ++i) {
        const int32_t id = s.blocks[i];
        if (a->hashed[id] || a->table.count(hashes[i])) continue;  // committed, or content held elsewhere
        a->hashed[id] = 1;
        a->bhash[id] = hashes[i];
        a->table.emplace(hashes[i], id);
        ++c;
    }
    if (committed) *committed = c;
    return PKV_OK;
}

int32_t pkv_alloc_num_cached(const pkv_alloc* a) { return a ? static_cast<int32_t>(a->evictable.size()) : -1; }

int64_t pkv_alloc_block_hash_of(const pkv_alloc* a, int32_t block, uint64_t* hash) {
    if (!a || block < 0 || block >= a->num_blocks || !hash) return -1;
    if (!a->hashed[block]) return 0;
    *hash = a->bhash[block];
    return 1;
}

void pkv_alloc_reset_prefix_cache(pkv_alloc* a) {
    if (!a) return;
    for (const auto& e : a->evictable) {
        a->stamp[e.second] = -1;
        a->free_stack.push_back(e.second);
    }
    a->evictable.clear();
    a->table.clear();
    std::fill(a->hashed.begin(), a->hashed.end(), 0);
}

}  // extern "C"
