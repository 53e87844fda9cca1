// Pieces of the chunked-prefill kernel (prefill_tc.cu; also the group mode of the
// sharing-aware decode): the work items, an item's block-table entries, the
// per-CTA sort of the items by size, and small tcgen05 / arithmetic wrappers.
// Internal linkage: each translation unit that includes it gets its own copy.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace pa {
namespace prefill {
namespace {

using namespace sm100;

constexpr int kKT = 128;                       // keys per tile
constexpr int kSortBuckets = 1024;             // key-tile counts; larger ones share the last bucket
constexpr int kSortMaxEntries = 16384;         // entries the sort takes
static_assert(kSortMaxEntries <= 65536, "entries fit 16 bits");

struct PItem {
    int b, kvh, q_row0, nq, pos_first, key0, kmax, ntiles;
    int group, slot, members;      // group mode: group index, partition slot, member count
};

// Item idx -> (sequence, kv head, query tile); false when the tile is empty or
// the sequence's lengths are inconsistent (reported once, by query tile 0).
__device__ __forceinline__ bool get_pitem(int idx, const PrefillParams &p, PItem &it) {
    const int qt = idx % p.qtiles;
    const int rest = idx / p.qtiles;
    it.kvh = rest % p.num_kv_heads;
    it.b = rest / p.num_kv_heads;
    const int q_start = p.query_start_loc[it.b];
    const int q_len = p.query_start_loc[it.b + 1] - q_start;
    const int ctx = p.context_lens[it.b];
    if (q_len < 0 || q_len > p.max_query_len || ctx < q_len || ctx > p.context_limit || q_start < 0 ||
        (int64_t)q_start + q_len > p.num_query_tokens) {
        if (qt == 0 && it.kvh == 0) raise_error(p.err, PA_DEVERR_CONTEXT);
        return false;
    }
    const int qi0 = qt * p.rows_q;
    if (qi0 >= q_len) return false;
    it.q_row0 = q_start + qi0;
    it.nq = min(p.rows_q, q_len - qi0);
    it.pos_first = ctx - q_len + qi0;
    it.key0 = 0;
    it.kmax = it.pos_first + it.nq;              // keys 0 .. kmax-1 are visible to some row
    it.ntiles = (it.kmax + kKT - 1) / kKT;
    return true;
}

// Group mode: item idx -> (group, kv head, shared partition); the keys are one
// partition of the group's shared prefix, read through the first member's table.
__device__ __forceinline__ bool get_gitem(int idx, const PrefillParams &p, PItem &it) {
    it.slot = idx % p.shared_parts;
    const int rest = idx / p.shared_parts;
    it.kvh = rest % p.num_kv_heads;
    it.group = rest / p.num_kv_heads;
    const int32_t *mem = p.group_members + (int64_t)it.group * p.max_members;
    const int lead = mem[0];
    if (lead < 0 || lead >= p.num_seqs) return false;
    int n = 1;                                   // members: leading valid ids
    while (n < p.max_members && mem[n] >= 0 && mem[n] < p.num_seqs) ++n;
    it.members = n;
    int ctx = p.context_lens[lead];
    ctx = ctx < 0 ? 0 : (ctx > p.context_limit ? p.context_limit : ctx);
    int ps = p.prefix_lens[lead];
    ps = (ps < 0 ? 0 : (ps > ctx ? ctx : ps)) & ~(p.block_size - 1);   // whole blocks, as seq_split
    it.key0 = it.slot * p.partition_size;
    if (it.key0 >= ps) return false;
    it.b = lead;
    it.kmax = min(ps, it.key0 + p.partition_size);
    it.ntiles = (it.kmax - it.key0 + kKT - 1) / kKT;
    it.pos_first = it.kmax - 1;                  // no causal limit: every row sees the whole partition
    it.q_row0 = 0;
    it.nq = n;
    return true;
}

// Key tiles of query tile qt of sequence b, as get_pitem would give them; 0 for an
// empty tile or an inconsistent sequence (reported by CTA 0 when `report`).
__device__ __forceinline__ int qtile_tiles(const PrefillParams &p, int b, int qt, bool report) {
    const int q_start = p.query_start_loc[b];
    const int q_len = p.query_start_loc[b + 1] - q_start;
    const int ctx = p.context_lens[b];
    if (q_len < 0 || q_len > p.max_query_len || ctx < q_len || ctx > p.context_limit || q_start < 0 ||
        (int64_t)q_start + q_len > p.num_query_tokens) {
        if (report && qt == 0 && blockIdx.x == 0) raise_error(p.err, PA_DEVERR_CONTEXT);
        return 0;
    }
    const int qi0 = qt * p.rows_q;
    if (qi0 >= q_len) return 0;
    const int kmax = ctx - q_len + qi0 + min(p.rows_q, q_len - qi0);
    const int t = (kmax + kKT - 1) / kKT;
    return t < kSortBuckets - 1 ? t : kSortBuckets - 1;
}

// Items of this CTA, largest first across the grid. The E entries (sizes from
// size(e), 0 = no work) are sorted by size, largest first -- a counting sort,
// stable by index, so every CTA derives the same order -- each entry standing
// for `sub` consecutive items; the CTA takes every grid-th item of that list in
// serpentine rounds. my[k] = entry * sub + s for its k-th item; returns the
// count (at most max_my). Scratch: ssz, sorted (E each), cursor (kSortBuckets).
// Every thread calls this; it ends with a barrier.
template <typename SizeFn>
__device__ __forceinline__ int sort_items(int E, int sub, SizeFn size, uint16_t *ssz, uint16_t *sorted, int *cursor,
                                          int *my, int max_my) {
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < kSortBuckets; i += blockDim.x) cursor[i] = 0;
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        const int t = size(e);
        ssz[e] = (uint16_t)t;
        if (t > 0) atomicAdd(&cursor[t], 1);
    }
    __syncthreads();
    if (tid < 32) {
        // descending exclusive prefix: cursor[t] = entries with more key tiles
        int cnt[kSortBuckets / 32], tot = 0;
#pragma unroll
        for (int i = 0; i < kSortBuckets / 32; ++i) {
            cnt[i] = cursor[kSortBuckets - 1 - (lane * (kSortBuckets / 32) + i)];
            tot += cnt[i];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - tot;
#pragma unroll
        for (int i = 0; i < kSortBuckets / 32; ++i) {
            cursor[kSortBuckets - 1 - (lane * (kSortBuckets / 32) + i)] = run;
            run += cnt[i];
        }
        __syncwarp();
        // stable placement, 32 entries at a time in index order
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int t = e < E ? ssz[e] : 0;
            const unsigned m = __match_any_sync(0xffffffffu, t);
            const int leader = __ffs(m) - 1;
            int pos = 0;
            if (lane == leader && t > 0) pos = cursor[t];
            pos = __shfl_sync(0xffffffffu, pos, leader);
            if (t > 0) sorted[pos + __popc(m & ((1u << lane) - 1))] = (uint16_t)e;
            __syncwarp();
            if (lane == leader && t > 0) cursor[t] = pos + __popc(m);
            __syncwarp();
        }
    }
    __syncthreads();
    // entries placed = entries with work = the start of bucket 0
    const int total = cursor[0] * sub;
    const int g = (int)gridDim.x, b0 = (int)blockIdx.x;
    const int rounds = total / g, rem = total - rounds * g;
    int n = rounds + ((((rounds & 1) ? g - 1 - b0 : b0) < rem) ? 1 : 0);
    n = n < max_my ? n : max_my;
    for (int k = tid; k < n; k += blockDim.x) {
        const int pk = k * g + ((k & 1) ? g - 1 - b0 : b0);
        const int q = pk / sub;
        my[k] = (int)sorted[q] * sub + (pk - q * sub);
    }
    fence_proxy_async_smem();            // the scratch's next writers may be TMA copies
    __syncthreads();
    return n;
}

// Block-table entries of an item's keys, read once at item start with one
// coalesced load per 32 blocks: entry j (the item's j-th block from key0) sits in
// register j / 32 of lane j % 32. Items of up to kCachedBlocks blocks are served
// from registers; entries past that are read per tile.
constexpr int kCachedBlocks = 256;
struct KeyTable {
    const int32_t *row;
    int nblk;
    int e[kCachedBlocks / 32];
};
__device__ __forceinline__ KeyTable load_key_table(const PrefillParams &p, const PItem &I, int lane) {
    KeyTable t;
    t.row = p.block_tables + (int64_t)I.b * p.max_blocks_per_seq + (I.key0 >> p.log2_block_size);
    t.nblk = I.kmax > I.key0 ? (I.kmax - I.key0 + p.block_size - 1) >> p.log2_block_size : 0;
#pragma unroll
    for (int k = 0; k < kCachedBlocks / 32; ++k) {
        const int j = k * 32 + lane;
        t.e[k] = j < t.nblk ? t.row[j] : -1;
    }
    return t;
}
// Physical block of block `lane` of key tile `tile` (nbt blocks per tile; nbt
// divides 32), or num_blocks (TMA fills zeros) past the item's keys or for a bad
// id (reported when `report`). Every lane of the warp calls this.
__device__ __forceinline__ int tile_block(const KeyTable &t, const PrefillParams &p, int tile, int nbt, int lane,
                                          bool report) {
    const int j0 = tile * nbt, j = j0 + lane;
    const bool live = lane < nbt && j < t.nblk;
    const int k = j0 >> 5;
    int e;
    if (k < kCachedBlocks / 32) {
        int v = t.e[0];
#pragma unroll
        for (int i = 1; i < kCachedBlocks / 32; ++i)
            if (k == i) v = t.e[i];
        e = __shfl_sync(0xffffffffu, v, j & 31);
    } else {
        e = live ? t.row[j] : -1;
    }
    if (!live) return (int)p.num_blocks;
    if (e >= 0 && e < p.num_blocks) return e;
    if (report) raise_error(p.err, PA_DEVERR_BLOCK_ID);
    return (int)p.num_blocks;
}

// D (tmem) [+]= A (tmem: M rows in lanes, 16-bit K pairs per column) * B (smem desc).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::
            "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two fp32 lanes in one instruction (sm_100 and later): a * b + c and a + b.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};"
        "\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};"
        "\n\tadd.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&v);
    } else {
        const __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
}

}  // namespace
}  // namespace prefill
}  // namespace pa
