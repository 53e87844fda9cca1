// Host-side block allocator: free stack, reference counts, fork and
// copy-on-write, block-table and slot-mapping export.
//
// Follows "PagedAttention实现" (ainanfeng.cn), section "PagedAttention管理器":
// the pool pushes ids 0..N-1 onto a free stack and allocation pops the top;
// an allocated block starts with reference count 1; cow_write duplicates a
// shared block into a fresh one, repoints the sequence's table and drops the
// old count; free_sequence drops every count and returns blocks at 0 to the
// stack. "CS349E lecture 7: 01_paged_attention.py" demo 1 fixes when a block is
// taken (only when a token starts one) and demo 3 the sharing of forked samples.
//
// Unlike the teaching listing, every failure is reported: an empty free stack
// (including during copy-on-write), an unknown sequence id, a double add.
// append() is all-or-nothing.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedattn.h"

namespace {

struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
};

}  // namespace

struct pa_allocator {
    int64_t num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;   // top = back()
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Seq> seqs;
    int64_t peak_used = 0;
    int64_t cow_copies = 0;

    int64_t used() const { return num_blocks - (int64_t)free_stack.size(); }

    int32_t take() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        if (used() > peak_used) peak_used = used();
        return b;
    }

    void drop(int32_t b) {
        if (--ref[b] == 0) free_stack.push_back(b);
    }

    // Blocks an append of n tokens takes: one copy when the partial last block
    // is shared, plus one per block boundary crossed.
    int64_t blocks_needed(const Seq &s, int64_t n) const {
        int64_t need = 0;
        const int64_t bs = block_size;
        if (n > 0 && s.len % bs != 0 && ref[s.table[s.len / bs]] > 1) need += 1;
        const int64_t end = s.len + n;
        need += (end + bs - 1) / bs - (s.len + bs - 1) / bs;
        return need;
    }

    int64_t cow_needed(const Seq &s, int64_t n) const {
        const int64_t bs = block_size;
        return (n > 0 && s.len % bs != 0 && ref[s.table[s.len / bs]] > 1) ? 1 : 0;
    }
};

// ---- checkpoint / resume ----------------------------------------------------
// Image layout (host byte order; every field a little-endian integer on the
// machines this builds for): 8-byte tag "PAALLOC1"; int64 num_blocks,
// block_size, peak_used, cow_copies; int64 free count, then the free stack
// bottom to top (int32 each); int32 reference count of every block; int64
// sequence count, then per sequence in increasing id order: int64 id, int64
// length, int64 table size, the table (int32 each).
namespace {

constexpr char kSnapTag[8] = {'P', 'A', 'A', 'L', 'L', 'O', 'C', '1'};

struct Writer {
    unsigned char *p;
    int64_t n = 0;
    template <typename T> void put(T v) {
        if (p) std::memcpy(p + n, &v, sizeof v);
        n += (int64_t)sizeof v;
    }
    void tag() {
        if (p) std::memcpy(p + n, kSnapTag, sizeof kSnapTag);
        n += (int64_t)sizeof kSnapTag;
    }
};

struct Reader {
    const unsigned char *p;
    int64_t size, n = 0;
    bool ok = true;
    template <typename T> T get() {
        T v{};
        if (!ok || size - n < (int64_t)sizeof v) {
            ok = false;
            return v;
        }
        std::memcpy(&v, p + n, sizeof v);
        n += (int64_t)sizeof v;
        return v;
    }
};

int64_t write_image(const pa_allocator *a, unsigned char *buf) {
    Writer w{buf};
    w.tag();
    w.put<int64_t>(a->num_blocks);
    w.put<int64_t>(a->block_size);
    w.put<int64_t>(a->peak_used);
    w.put<int64_t>(a->cow_copies);
    w.put<int64_t>((int64_t)a->free_stack.size());
    for (int32_t b : a->free_stack) w.put<int32_t>(b);
    for (int32_t r : a->ref) w.put<int32_t>(r);
    std::vector<int64_t> ids;
    ids.reserve(a->seqs.size());
    for (const auto &kv : a->seqs) ids.push_back(kv.first);
    std::sort(ids.begin(), ids.end());
    w.put<int64_t>((int64_t)ids.size());
    for (int64_t id : ids) {
        const Seq &s = a->seqs.find(id)->second;
        w.put<int64_t>(id);
        w.put<int64_t>(s.len);
        w.put<int64_t>((int64_t)s.table.size());
        for (int32_t b : s.table) w.put<int32_t>(b);
    }
    return w.n;
}

}  // namespace

extern "C" {

int pa_alloc_create(int64_t num_blocks, int block_size, pa_allocator **out) {
    if (!out || num_blocks < 0 || num_blocks > INT32_MAX || block_size <= 0) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    pa_allocator *a = new (std::nothrow) pa_allocator();
    if (!a) return PA_ERR_OUT_OF_BLOCKS;
    try {
        a->num_blocks = num_blocks;
        a->block_size = block_size;
        a->ref.assign((size_t)num_blocks, 0);
        a->free_stack.reserve((size_t)num_blocks);
        for (int64_t i = 0; i < num_blocks; ++i) a->free_stack.push_back((int32_t)i);
    } catch (...) {
        delete a;
        return PA_ERR_OUT_OF_BLOCKS;
    }
    *out = a;
    return PA_OK;
}

void pa_alloc_destroy(pa_allocator *a) { delete a; }

int pa_alloc_add_seq(pa_allocator *a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (a->seqs.count(seq_id)) return PA_ERR_EXISTS;
    try {
        a->seqs.emplace(seq_id, Seq{});
    } catch (...) {
        return PA_ERR_OUT_OF_BLOCKS;
    }
    return PA_OK;
}

int pa_alloc_fork(pa_allocator *a, int64_t parent, int64_t child) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (a->seqs.count(child)) return PA_ERR_EXISTS;
    try {
        Seq s = it->second;   // copy before the map may rehash
        for (int32_t b : s.table) a->ref[b] += 1;
        a->seqs.emplace(child, std::move(s));
    } catch (...) {
        return PA_ERR_OUT_OF_BLOCKS;
    }
    return PA_OK;
}

int pa_alloc_append(pa_allocator *a, int64_t seq_id, int64_t n_tokens, int32_t *slots_out,
                    int32_t *cow_pairs_out, int64_t cow_cap, int64_t *n_cow) {
    if (!a || n_tokens < 0 || (n_tokens > 0 && !slots_out) || cow_cap < 0) return PA_ERR_INVALID_ARG;
    if (n_cow) *n_cow = 0;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    Seq &s = it->second;
    const int64_t bs = a->block_size;
    if (a->blocks_needed(s, n_tokens) > (int64_t)a->free_stack.size()) return PA_ERR_OUT_OF_BLOCKS;
    if (a->cow_needed(s, n_tokens) > cow_cap || (a->cow_needed(s, n_tokens) && !cow_pairs_out))
        return PA_ERR_INVALID_ARG;
    if ((s.len + n_tokens + bs - 1) / bs > INT32_MAX) return PA_ERR_INVALID_ARG;
    try {
        s.table.reserve((size_t)((s.len + n_tokens + bs - 1) / bs));
    } catch (...) {
        return PA_ERR_OUT_OF_BLOCKS;
    }
    int64_t pairs = 0;
    for (int64_t i = 0; i < n_tokens; ++i) {
        const int64_t pos = s.len;
        const int64_t page = pos / bs;
        if (page == (int64_t)s.table.size()) {
            s.table.push_back(a->take());
        } else if (a->ref[s.table[page]] > 1) {
            const int32_t old = s.table[page];
            const int32_t fresh = a->take();
            cow_pairs_out[2 * pairs] = old;
            cow_pairs_out[2 * pairs + 1] = fresh;
            ++pairs;
            s.table[page] = fresh;
            a->ref[old] -= 1;
            a->cow_copies += 1;
        }
        slots_out[i] = (int32_t)((int64_t)s.table[page] * bs + pos % bs);
        s.len = pos + 1;
    }
    if (n_cow) *n_cow = pairs;
    return PA_OK;
}

int pa_alloc_free_seq(pa_allocator *a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    for (int32_t b : it->second.table) a->drop(b);
    a->seqs.erase(it);
    return PA_OK;
}

int pa_alloc_block_table(const pa_allocator *a, int64_t seq_id, int32_t *out, int64_t cap,
                         int64_t *n) {
    if (!a || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    const auto &t = it->second.table;
    for (int64_t i = 0; i < (int64_t)t.size() && i < cap; ++i) out[i] = t[(size_t)i];
    if (n) *n = (int64_t)t.size();
    return PA_OK;
}

int pa_alloc_seq_len(const pa_allocator *a, int64_t seq_id, int64_t *len) {
    if (!a || !len) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    *len = it->second.len;
    return PA_OK;
}

int pa_alloc_export(const pa_allocator *a, const int64_t *seq_ids, int64_t n_seqs, int32_t *tables,
                    int max_blocks_per_seq, int32_t *context_lens) {
    if (!a || n_seqs < 0 || max_blocks_per_seq < 0 || (n_seqs > 0 && (!seq_ids || !context_lens)) ||
        (n_seqs > 0 && max_blocks_per_seq > 0 && !tables))
        return PA_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n_seqs; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
        if ((int64_t)it->second.table.size() > max_blocks_per_seq) return PA_ERR_INVALID_ARG;
        if (it->second.len > INT32_MAX) return PA_ERR_INVALID_ARG;
    }
    for (int64_t i = 0; i < n_seqs; ++i) {
        const Seq &s = a->seqs.find(seq_ids[i])->second;
        int32_t *row = tables + i * (int64_t)max_blocks_per_seq;
        int64_t j = 0;
        for (; j < (int64_t)s.table.size(); ++j) row[j] = s.table[(size_t)j];
        for (; j < max_blocks_per_seq; ++j) row[j] = -1;
        context_lens[i] = (int32_t)s.len;
    }
    return PA_OK;
}

int pa_alloc_block(pa_allocator *a, int32_t *block_out) {
    if (!a || !block_out) return PA_ERR_INVALID_ARG;
    if (a->free_stack.empty()) return PA_ERR_OUT_OF_BLOCKS;
    *block_out = a->take();
    return PA_OK;
}

int pa_alloc_decref(pa_allocator *a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks || a->ref[block] <= 0) return PA_ERR_INVALID_ARG;
    a->drop(block);
    return PA_OK;
}

int pa_alloc_refcount(const pa_allocator *a, int32_t block, int32_t *count) {
    if (!a || !count || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID_ARG;
    *count = a->ref[block];
    return PA_OK;
}

int pa_alloc_get_stats(const pa_allocator *a, pa_alloc_stats *out) {
    if (!a || !out) return PA_ERR_INVALID_ARG;
    out->num_blocks = a->num_blocks;
    out->num_free = (int64_t)a->free_stack.size();
    out->num_used = a->used();
    out->peak_used = a->peak_used;
    out->num_cow_copies = a->cow_copies;
    out->num_seqs = (int64_t)a->seqs.size();
    return PA_OK;
}


int pa_alloc_snapshot(const pa_allocator *a, void *buf, int64_t cap, int64_t *size) {
    if (!a || !size || cap < 0) return PA_ERR_INVALID_ARG;
    try {
        *size = write_image(a, nullptr);
        if (!buf) return PA_OK;
        if (cap < *size) return PA_ERR_INVALID_ARG;
        write_image(a, static_cast<unsigned char *>(buf));
    } catch (...) {
        return PA_ERR_OUT_OF_BLOCKS;
    }
    return PA_OK;
}

int pa_alloc_restore(const void *buf, int64_t size, pa_allocator **out) {
    if (!out) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!buf || size < (int64_t)sizeof kSnapTag) return PA_ERR_INVALID_ARG;
    if (std::memcmp(buf, kSnapTag, sizeof kSnapTag) != 0) return PA_ERR_INVALID_ARG;
    Reader r{static_cast<const unsigned char *>(buf), size, (int64_t)sizeof kSnapTag};
    pa_allocator *a = new (std::nothrow) pa_allocator();
    if (!a) return PA_ERR_OUT_OF_BLOCKS;
    int rc = PA_ERR_INVALID_ARG;
    try {
        const int64_t nb = r.get<int64_t>(), bs = r.get<int64_t>();
        const int64_t peak = r.get<int64_t>(), copies = r.get<int64_t>(), nfree = r.get<int64_t>();
        if (!r.ok || nb < 0 || nb > INT32_MAX || bs <= 0 || bs > INT32_MAX || copies < 0 || nfree < 0 ||
            nfree > nb || (size - r.n) / 4 < nfree + nb)
            throw rc;
        a->num_blocks = nb;
        a->block_size = (int)bs;
        a->peak_used = peak;
        a->cow_copies = copies;
        a->free_stack.resize((size_t)nfree);
        for (auto &b : a->free_stack) b = r.get<int32_t>();
        a->ref.resize((size_t)nb);
        for (auto &c : a->ref) c = r.get<int32_t>();
        // the free stack is exactly the blocks nobody references, each once
        std::vector<char> seen((size_t)nb, 0);
        for (int32_t b : a->free_stack) {
            if (b < 0 || b >= nb || seen[(size_t)b] || a->ref[(size_t)b] != 0) throw rc;
            seen[(size_t)b] = 1;
        }
        int64_t zero = 0;
        for (int32_t c : a->ref) {
            if (c < 0) throw rc;
            zero += c == 0;
        }
        if (zero != nfree || peak < a->used()) throw rc;
        // sequences: increasing ids, tables as long as their lengths need, holding
        // referenced blocks; a block's count covers at least the tables holding it
        std::vector<int64_t> held((size_t)nb, 0);
        const int64_t nseq = r.get<int64_t>();
        if (!r.ok || nseq < 0 || (size - r.n) / 24 < nseq) throw rc;
        int64_t prev = 0;
        for (int64_t i = 0; i < nseq; ++i) {
            const int64_t id = r.get<int64_t>(), len = r.get<int64_t>(), nt = r.get<int64_t>();
            if (!r.ok || (i > 0 && id <= prev) || len < 0 || nt != (len + bs - 1) / bs || (size - r.n) / 4 < nt)
                throw rc;
            prev = id;
            Seq s;
            s.len = len;
            s.table.resize((size_t)nt);
            for (auto &b : s.table) {
                b = r.get<int32_t>();
                if (b < 0 || b >= nb || a->ref[(size_t)b] <= 0) throw rc;
                held[(size_t)b] += 1;
            }
            a->seqs.emplace(id, std::move(s));
        }
        for (int64_t b = 0; b < nb; ++b)
            if (held[(size_t)b] > a->ref[(size_t)b]) throw rc;
        if (!r.ok || r.n != size) throw rc;
    } catch (int) {
        delete a;
        return PA_ERR_INVALID_ARG;
    } catch (...) {
        delete a;
        return PA_ERR_OUT_OF_BLOCKS;
    }
    *out = a;
    return PA_OK;
}

int pa_prefix_groups(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                     int max_blocks_per_seq, int block_size, int max_members, int min_shared_blocks,
                     int32_t *prefix_lens, int32_t *group_members, int *num_groups) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || max_members < 2 || min_shared_blocks < 1 ||
        !num_groups || (num_seqs > 0 && (!block_tables || !context_lens || !prefix_lens || !group_members)))
        return PA_ERR_INVALID_ARG;
    *num_groups = 0;
    try {
        // candidates keyed by their first physical block, in sequence order
        std::map<int32_t, std::vector<int>> by_first;
        for (int b = 0; b < num_seqs; ++b) {
            prefix_lens[b] = 0;
            const int full = std::min(context_lens[b] / block_size, max_blocks_per_seq);
            if (full >= min_shared_blocks && block_tables[(int64_t)b * max_blocks_per_seq] >= 0)
                by_first[block_tables[(int64_t)b * max_blocks_per_seq]].push_back(b);
        }
        int ng = 0;
        for (auto &kv : by_first) {
            const std::vector<int> &mem = kv.second;
            if (mem.size() < 2) continue;
            for (size_t c0 = 0; c0 < mem.size(); c0 += (size_t)max_members) {
                const size_t c1 = std::min(mem.size(), c0 + (size_t)max_members);
                if (c1 - c0 < 2) continue;
                // leading blocks identical in every member and full in every member's context
                int shared = max_blocks_per_seq;
                for (size_t i = c0; i < c1; ++i)
                    shared = std::min(shared, context_lens[mem[i]] / block_size);
                const int32_t *lead = block_tables + (int64_t)mem[c0] * max_blocks_per_seq;
                int j = 0;
                for (; j < shared; ++j) {
                    bool same = lead[j] >= 0;
                    for (size_t i = c0 + 1; i < c1 && same; ++i)
                        same = block_tables[(int64_t)mem[i] * max_blocks_per_seq + j] == lead[j];
                    if (!same) break;
                }
                if (j < min_shared_blocks) continue;
                int32_t *row = group_members + (int64_t)ng * max_members;
                for (int i = 0; i < max_members; ++i)
                    row[i] = (size_t)i < c1 - c0 ? (int32_t)mem[c0 + (size_t)i] : -1;
                for (size_t i = c0; i < c1; ++i) prefix_lens[mem[i]] = j * block_size;
                ++ng;
            }
        }
        *num_groups = ng;
    } catch (...) {
        return PA_ERR_OUT_OF_BLOCKS;
    }
    return PA_OK;
}

}  // extern "C"
