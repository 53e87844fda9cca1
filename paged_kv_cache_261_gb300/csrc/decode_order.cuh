// Work-item order shared by the persistent tensor-core decode kernels.
//
// A work item is (sequence, partition, kv head). Items are dealt to CTAs in
// serpentine rounds (below) in order of decreasing size: first every partition with the full
// tile count (partition_size / 128 tiles: the full ones, and last partitions
// just as long in tiles), then the other last partitions by tile count -- three
// or more, two, one -- then empty contexts. prefix[] counts full-tile-count
// partitions per sequence; order[] lists the remaining sequences in that bucket
// order (stable within a bucket). Each CTA builds both in shared memory at
// kernel start (a deterministic counting sort), so no host pass or global
// scratch is needed.
#pragma once

#include "kernels.h"

namespace pa {
namespace decode_order {

constexpr int kTile = 128;   // tokens per tile

struct Item {
    int b, kvh, part, slot, t0, t1, ntiles;
    bool direct;             // write the final row, not a partial
    bool last;               // ends at the sequence's context length
};

// Per-sequence lengths cached in shared memory by build(): the clamped context
// length and the first token of this pass (after a shared prefix, else 0).
struct SeqCache {
    int *ctx;
    int *ps;
};

// seq_split (kernels.h) from the cached lengths.
__device__ __forceinline__ SeqSplit split_cached(const DecodeParams &p, const SeqCache &c, int b) {
    SeqSplit s;
    s.ctx = c.ctx[b];
    s.ps = c.ps[b];
    s.shared = (s.ps + p.partition_size - 1) / p.partition_size;
    s.priv = (s.ctx - s.ps + p.partition_size - 1) / p.partition_size;
    s.direct = s.ctx == 0 || (s.shared == 0 && s.priv <= 1);
    return s;
}

// Item idx -> its sequence, partition, kv head and token range. n4 = prefix[num_seqs].
__device__ __forceinline__ Item get_item(int idx, const int *prefix, const int *order, int n4,
                                         const DecodeParams &p, const SeqCache &c) {
    Item it;
    const int pair = idx / p.num_kv_heads;
    it.kvh = idx - pair * p.num_kv_heads;
    if (pair < n4) {
        int lo = 0, hi = p.num_seqs;              // prefix[lo] <= pair < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= pair) lo = mid; else hi = mid;
        }
        it.b = lo;
        it.part = pair - prefix[lo];
    } else {
        it.b = order[pair - n4];
        it.part = -1;                            // the sequence's last (ragged) partition
    }
    const SeqSplit sp = split_cached(p, c, it.b);
    if (it.part < 0) it.part = (sp.ctx - sp.ps) / p.partition_size;
    it.slot = sp.shared + it.part;
    it.direct = sp.direct;
    it.t0 = sp.ps + it.part * p.partition_size;
    it.t1 = min(sp.ctx, it.t0 + p.partition_size);
    it.last = it.t1 == sp.ctx;
    it.ntiles = it.t1 > it.t0 ? (it.t1 - it.t0 + kTile - 1) / kTile : 0;
    return it;
}

// Builds prefix[0 .. num_seqs] and order[] (see above), fills the length cache
// and writes counts[0] = n4, counts[1] = length of order[]. `code` is num_seqs
// bytes of scratch. Every thread of the CTA calls this; the caller synchronises
// before reading. Context lengths outside [0, context_limit] raise
// PA_DEVERR_CONTEXT (CTA 0).
__device__ __forceinline__ void build(const DecodeParams &p, int *prefix, int *order, int *counts,
                                      unsigned char *code, const SeqCache &c) {
    const int B = p.num_seqs;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // per sequence: the count of full-tile-count partitions goes to prefix[b + 1]
    // and the list bucket of its last partition to code[b]
    for (int b = tid; b < B; b += blockDim.x) {
        const int raw = p.context_lens[b];
        if ((raw < 0 || raw > p.context_limit) && blockIdx.x == 0) raise_error(p.err, PA_DEVERR_CONTEXT);
        const SeqSplit sp = seq_split(p, b);
        c.ctx[b] = sp.ctx;
        c.ps[b] = sp.ps;
        const int len = sp.ctx - sp.ps;                                      // this pass's tokens
        const int nfull = len / p.partition_size;
        const int rt = (len - nfull * p.partition_size + kTile - 1) / kTile;   // tiles of the ragged rest
        const bool rest_is_full = rt * kTile == p.partition_size;           // as many tiles as a full one
        prefix[b + 1] = nfull + (rest_is_full ? 1 : 0);
        // list bucket: 0 = empty context (or, when folding, a wholly shared one: an item
        // with no tiles), 1..3 = tiles of the rest (3 = three or more), 4 = no list entry
        // (no ragged rest, or one with the full tile count)
        const bool empty = sp.ctx == 0 || (p.fold_shared && len == 0);
        code[b] = (unsigned char)(empty ? 0 : ((rt == 0 || rest_is_full) ? 4 : min(rt, 3)));
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (B + 31) / 32;
        const int lo = lane * per, hi = min(B, lo + per);
        int s4 = 0, c0 = 0, c1 = 0, c2 = 0, c3 = 0;        // this lane's counts per bucket
        for (int i = lo; i < hi; ++i) {
            s4 += prefix[i + 1];
            const int k = code[i];
            c0 += k == 0;
            c1 += k == 1;
            c2 += k == 2;
            c3 += k == 3;
        }
        int i4 = s4, i0 = c0, i1 = c1, i2 = c2, i3 = c3;     // inclusive scans over lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n4v = __shfl_up_sync(0xffffffffu, i4, o), n0 = __shfl_up_sync(0xffffffffu, i0, o);
            const int n1 = __shfl_up_sync(0xffffffffu, i1, o), n2 = __shfl_up_sync(0xffffffffu, i2, o);
            const int n3 = __shfl_up_sync(0xffffffffu, i3, o);
            if (lane >= o) {
                i4 += n4v;
                i0 += n0;
                i1 += n1;
                i2 += n2;
                i3 += n3;
            }
        }
        const int t0 = __shfl_sync(0xffffffffu, i0, 31), t1 = __shfl_sync(0xffffffffu, i1, 31);
        const int t2 = __shfl_sync(0xffffffffu, i2, 31), t3 = __shfl_sync(0xffffffffu, i3, 31);
        // list order: bucket 3, 2, 1, then 0
        int p3 = i3 - c3, p2 = t3 + i2 - c2, p1 = t3 + t2 + i1 - c1, p0 = t3 + t2 + t1 + i0 - c0;
        int run = i4 - s4;
        for (int i = lo; i < hi; ++i) {
            run += prefix[i + 1];
            prefix[i + 1] = run;
            const int k = code[i];
            if (k == 3) order[p3++] = i;
            else if (k == 2) order[p2++] = i;
            else if (k == 1) order[p1++] = i;
            else if (k == 0) order[p0++] = i;
        }
        if (lane == 0) prefix[0] = 0;
        if (lane == 31) {
            counts[0] = i4;
            counts[1] = t0 + t1 + t2 + t3;
        }
    }
}

// ---- per-CTA item table ----------------------------------------------------------
// Items are dealt in rounds of gridDim.x, serpentine: in even rounds CTA b takes
// the round's b-th item, in odd rounds its (gridDim.x - 1 - b)-th. Down a list
// sorted by decreasing size this evens the CTAs' totals (a CTA that took a larger
// item in one round takes a smaller one in the next); round-robin left the 8B-shaped
// batch's most loaded CTA 62 tiles against a mean of 59.9. A CTA's k-th item's
// descriptor is computed once, in parallel, and kept in shared memory (16 bytes),
// so no role repeats the search and the divisions of get_item at every item.
constexpr int kTableItems = 512;       // items per CTA the table holds (8 KiB)

__device__ __forceinline__ int4 pack_item(const Item &it) {
    return make_int4(it.b | (it.kvh << 16), it.t0, it.t1 | (it.last ? int(0x80000000u) : 0),
                     it.slot | (it.direct ? int(0x80000000u) : 0));
}
__device__ __forceinline__ Item unpack_item(int4 d) {
    Item it;
    it.b = d.x & 0xFFFF;
    it.kvh = (int)((unsigned)d.x >> 16);
    it.t0 = d.y;
    it.t1 = d.z & 0x7FFFFFFF;
    it.last = d.z < 0;
    it.slot = d.w & 0x7FFFFFFF;
    it.direct = d.w < 0;
    it.part = 0;                     // not needed once the table is built
    it.ntiles = it.t1 > it.t0 ? (it.t1 - it.t0 + kTile - 1) / kTile : 0;
    return it;
}
// Index of this CTA's k-th item.
__device__ __forceinline__ int cta_item_index(int k) {
    const int g = (int)gridDim.x, b = (int)blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - b : b);
}
// Items of this CTA: one per full round, plus one in the last, partial round if
// its position there falls below the remainder. The host sizes launches so that
// this never exceeds kTableItems; the clamp only keeps every table access inside
// the table.
__device__ __forceinline__ int cta_items(int total_items) {
    const int g = (int)gridDim.x, b = (int)blockIdx.x;
    const int rounds = total_items / g, rem = total_items - rounds * g;
    const int pos = (rounds & 1) ? g - 1 - b : b;
    const int n = rounds + (pos < rem ? 1 : 0);
    return n < kTableItems ? n : kTableItems;
}
// Every thread of the CTA calls this after build() and a barrier. The table is
// written over `area` (the ordering arrays, no longer needed) once every thread
// has computed its descriptors; the caller synchronises before reading it.
template <int kPerThread>
__device__ __forceinline__ void build_item_table(const DecodeParams &p, const int *prefix, const int *order,
                                                 int n4, const SeqCache &c, int total_items, int4 *area) {
    const int n = cta_items(total_items);
    int4 d[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int k = (int)threadIdx.x + u * (int)blockDim.x;
        if (k < n) d[u] = pack_item(get_item(cta_item_index(k), prefix, order, n4, p, c));
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int k = (int)threadIdx.x + u * (int)blockDim.x;
        if (k < n) area[k] = d[u];
    }
}

// Block-table entries of one item, read once with one coalesced load per 32
// blocks: entry j (the item's j-th block) sits in register j / 32 of lane
// j % 32. Items of up to kCachedBlocks blocks (every item of a 512-token
// partition) are served from registers; entries past that are read per tile.
constexpr int kCachedBlocks = 128;

struct ItemTable {
    const int32_t *row;   // the sequence's table, from the item's first block
    int nblk;             // blocks of the item
    int e[kCachedBlocks / 32];
};

__device__ __forceinline__ ItemTable load_item_table(const DecodeParams &p, const Item &I, int lane) {
    ItemTable t;
    t.row = p.block_tables + (int64_t)I.b * p.max_blocks_per_seq + (I.t0 >> p.log2_block_size);
    t.nblk = I.t1 > I.t0 ? (I.t1 - I.t0 + p.block_size - 1) >> p.log2_block_size : 0;
#pragma unroll
    for (int k = 0; k < kCachedBlocks / 32; ++k) {
        const int j = k * 32 + lane;
        t.e[k] = j < t.nblk ? t.row[j] : -1;
    }
    return t;
}

// Entry of block `lane` of tile `tile` (nbt blocks per tile, nbt divides 32), and
// whether that block holds tokens of the item. Every lane of the warp calls this.
__device__ __forceinline__ int tile_entry(const ItemTable &t, int tile, int nbt, int lane, bool *live) {
    const int j0 = tile * nbt;                 // a multiple of nbt: the tile's blocks share j0 / 32
    const int j = j0 + lane;
    *live = lane < nbt && j < t.nblk;
    const int k = j0 >> 5;
    if (k < kCachedBlocks / 32) {
        int v = t.e[0];
#pragma unroll
        for (int i = 1; i < kCachedBlocks / 32; ++i)
            if (k == i) v = t.e[i];
        return __shfl_sync(0xffffffffu, v, j & 31);
    }
    return *live ? t.row[j] : -1;
}

}  // namespace decode_order
}  // namespace pa
