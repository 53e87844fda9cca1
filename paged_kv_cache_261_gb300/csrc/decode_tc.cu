// Decode attention on the sm_100 tensor cores (tcgen05) with TMA block gathers.
//
// Computes what "CS349E lecture 7: 01_paged_attention.py", demo 2, paper eq. 4
// defines: for each sequence and query head, scores against every cached key
// are formed block by block through the block table, one softmax is taken over
// the whole context, and V is accumulated block by block. The softmax is taken
// online (running max and sum per head, rescaled when the max grows), which
// equals the softmax over the whole context once normalised; partitions of a
// long context are merged by decode_reduce_kernel.
//
// Shape of the work. All G query heads of a kv head share one K/V read, so
// per 128-token tile the contraction is S^T[128 tok x 16] = K[128 x 128] . Q^T
// and O^T[128 d x 16] = V^T[128 x 128 tok] . P^T: two M=128, N=16 (G padded),
// K=128 tcgen05 MMAs with bf16/f16 operands in shared memory and fp32
// accumulators in tensor memory. The tensor cores take the G-fold reuse of each
// K/V element off the FP32 pipes; the kernel stays bound by HBM.
//
// CTA = one persistent worker per SM; 416 threads:
//   warp 0    TMA producer of K: per tile, reads the tile's table entries (one
//             lane per physical block, from the item's entries read once at
//             item start) and loads each block's K rows (box = 64 dims x
//             block_size tokens of one kv head, 128-byte swizzle) plus the
//             group's queries into a 3-stage ring. Blocks past the partition
//             end or with a bad id load from an out-of-range coordinate, which
//             TMA fills with zeros.
//   warp 7    TMA producer of V into the same stages (its own full barrier).
//             In a decode with append, warps 0 and 7 also store the sequence's
//             new K / V row just before they load the tile that holds it
//             (append_token).
//   warp 6    L2 prefetch: walks the same tiles up to kPrefetchTiles ahead of
//             the producer's loads and pulls their blocks into L2.
//   warp 1    S MMA issuer (one thread) and tensor-memory owner: S for tile i
//             into a double-buffered S accumulator.
//   warp 8    P.V MMA issuer (one thread): O for tile i once its probabilities
//             are in shared memory and its V has landed. Copy issue and MMA
//             issue each cost a single thread most of a tile's time when one
//             thread did both operands, so each operand has its own issuer.
//   warps 2-5, 9-12  softmax and output in two warpgroups, each taking half of
//             the query columns (thread = token for S, thread = dim for O):
//             scale, mask, tile max through shuffles + shared memory, exp2,
//             P^T to shared memory (bf16/f16, 128-byte swizzled K-major), zero
//             V rows of masked tokens (their contents may be anything; the first
//             warpgroup), and o = o * alpha + O_tile in registers. In the G = 8 and
//             joining instances an item's finish (its last O, the sum of l over
//             the warps, the output) waits until the next item's first tile has
//             been through the softmax, so no warpgroup idles at item boundaries.
// Work items = (sequence, partition, kv head), dealt to CTAs in serpentine
// rounds in order of decreasing size, from a bucketed prefix sum that each CTA
// builds in shared memory at kernel start (decode_order.cuh). The joining instance
// (kFold) serves the sharing-aware decode when one partition covers every whole
// context: each item loads its sequence's shared-prefix partial at item start and
// writes the final row, so no merge runs. Every wait is bounded (see
// sm100.cuh); on a timeout the kernel sets PA_DEVERR_WAIT, drains its copies and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "decode_order.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tma_maps.cuh"

namespace pa {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kTile = 128;                        // tokens per MMA tile (M)
constexpr int kN = 16;                            // MMA N: query heads of a group, padded
constexpr int kStages = 3;
constexpr int kChunkBytes = kTile * 128;          // 128 rows x 64 dims x 2 B
constexpr int kKVBytes = 2 * kChunkBytes;         // one tile of K (or V), both 64-dim halves
constexpr int kQBytes = 2 * kN * 128;             // 16 rows x 128 dims
constexpr int kPBytes = 2 * kN * 128;             // P^T: 16 rows x 128 tokens
constexpr int kVProdWarp = 7;                     // issues the V boxes
constexpr int kPvWarp = 8;                        // issues the P.V MMAs

// Two softmax warpgroups per CTA (warps 2-5 and 9-12), each taking half of the
// padded query columns of every tile. One warpgroup's chain per tile (the column
// maxima, the exchange, two exponentials and a store per column, the O
// accumulation) set the pace at 16 query columns; two interleave on each SM
// sub-partition: G = 16 on the 8B-shaped contexts 0.134 -> 0.112 ms; G = 8 (long
// context) 0.4040 -> 0.3998 ms; G = 4 0.0998 -> 0.0995 ms.
constexpr int kThreads = 416;
constexpr int kWg2Warp = 9;                       // first warp of the second softmax warpgroup
constexpr int kMaxSeqs = 512;                     // sequences per launch (the host splits larger batches)
constexpr uint32_t kTmemCols = 64;                // S[2] x 16 + O[2] x 16 columns
constexpr int kPrefetchTiles = 2;                 // L2 prefetch distance, in tiles, ahead of the loads

// shared-memory carve-up (from a 1024-aligned base)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffQ = kOffV + kStages * kKVBytes;
constexpr int kOffP = kOffQ + kStages * kQBytes;
constexpr int kOffRed = kOffP + 2 * kPBytes;                  // float [2][4][16]
constexpr int kOffLRed = kOffRed + 2 * 4 * kN * 4;            // float [2][4][16] (by item parity)
constexpr int kOffBar = kOffLRed + 2 * 4 * kN * 4;                // uint64 barriers
// mbarrier slots, in order; kNumBars counts them
constexpr int kBarFull = 0;                                   // [kStages] K and Q of the stage landed
constexpr int kBarEmpty = kBarFull + kStages;                 // [kStages]
constexpr int kBarSFull = kBarEmpty + kStages;                // [2]
constexpr int kBarSFree = kBarSFull + 2;                      // [2]
constexpr int kBarPFull = kBarSFree + 2;                      // [2]
constexpr int kBarOFull = kBarPFull + 2;                      // [2]
constexpr int kBarOFree = kBarOFull + 2;                      // [2]
constexpr int kBarRed = kBarOFree + 2;                        // [2 warpgroups][2]
constexpr int kBarFin = kBarRed + 4;                          // [2 warpgroups]
constexpr int kBarFullV = kBarFin + 2;                        // [kStages] V of the stage landed
constexpr int kNumBars = kBarFullV + kStages;
constexpr int kOffMisc = kOffBar + kNumBars * 8;              // tmem base, abort flag, 2 item counts
constexpr int kOffPrefix = (kOffMisc + 32 + 15) & ~15;        // int [kMaxSeqs + 1]; later the item table
constexpr int kOffOrder = kOffPrefix + (kMaxSeqs + 1) * 4;    // int [kMaxSeqs]
constexpr int kOffCtx = kOffOrder + kMaxSeqs * 4;             // int [kMaxSeqs] clamped context lengths
constexpr int kOffPs = kOffCtx + kMaxSeqs * 4;                // int [kMaxSeqs] first token of this pass
constexpr int kSmemUsed = kOffPs + kMaxSeqs * 4;
static_assert(kSmemUsed - kOffPrefix >= decode_order::kTableItems * 16, "item table fits the ordering arrays");
constexpr int kSmemBytes = kSmemUsed + 1024;                  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Bars {
    uint64_t *full, *empty;        // [kStages]
    uint64_t *s_full, *s_free;     // [2]
    uint64_t *p_full, *o_full;     // [2]
    uint64_t *o_free;              // [2]
    uint64_t *red;                 // [warpgroup][2]
    uint64_t *fin;                 // [warpgroup]
    uint64_t *full_v;              // [kStages]
};

using decode_order::Item;
using decode_order::get_item;

// Largest value over the warp in one instruction (exact, as any max).
__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The decode step's own token of the item's sequence (position ctx - 1), for the
// item's kv head, when the call carries it (decode with append). The producer warps
// read its slot and its row (K by the K producer, V by the V producer) at the start
// of the sequence's last item and write the row just before they load the item's
// last tile, so that tile's loads read it. `e` is the block-table entry of the
// token's block (the one that tile loads). The slot must be that of position
// ctx - 1 (a different one sets PA_DEVERR_SLOT and is not written; -1 writes nothing).
constexpr int kAppVecs = kD * 2 / 16;          // one kv head's row: 16 vectors of 16 bytes

__device__ __forceinline__ uint4 append_row(const DecodeParams &p, const Item &I, bool is_v, int lane) {
    const uint4 *src = reinterpret_cast<const uint4 *>(is_v ? p.app_v : p.app_k) +
                       ((int64_t)I.b * p.num_kv_heads + I.kvh) * kAppVecs;
    return lane < kAppVecs ? src[lane] : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void append_token(const DecodeParams &p, const Item &I, int slot, int e, uint4 row,
                                             bool is_v, int lane) {
    const int pos = I.t1 - 1;
    const int64_t expect = (int64_t)e * p.block_size + (pos & (p.block_size - 1));
    if (e < 0 || e >= p.num_blocks || (int64_t)slot != expect) {
        if (!is_v && lane == 0) raise_error(p.err, PA_DEVERR_SLOT);
        return;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(const_cast<void *>(is_v ? p.value_cache : p.key_cache)) +
                 ((int64_t)slot * p.num_kv_heads + I.kvh) * kAppVecs;
    if (lane < kAppVecs) dst[lane] = row;
    asm volatile("fence.proxy.async.global;" ::: "memory");   // the tile's TMA loads read it
}

template <typename T> __device__ __forceinline__ uint16_t to_bits(float x);
template <> __device__ __forceinline__ uint16_t to_bits<__nv_bfloat16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <> __device__ __forceinline__ uint16_t to_bits<__half>(float x) {
    return __half_as_ushort(__float2half_rn(x));
}
template <typename T> __device__ __forceinline__ float from_bits(uint16_t b);
template <> __device__ __forceinline__ float from_bits<__nv_bfloat16>(uint16_t b) {
    return __uint_as_float((uint32_t)b << 16);
}
template <> __device__ __forceinline__ float from_bits<__half>(uint16_t b) {
    return __half2float(__ushort_as_half(b));
}

template <typename T, int GT, bool kFold>
__global__ __launch_bounds__(kThreads, 1) void decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                const __grid_constant__ CUtensorMap tm_v,
                                                                const __grid_constant__ CUtensorMap tm_q,
                                                                const DecodeParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sK = smem + kOffK;
    unsigned char *sV = smem + kOffV;
    unsigned char *sQ = smem + kOffQ;
    unsigned char *sP = smem + kOffP;
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    float *lred = reinterpret_cast<float *>(smem + kOffLRed);
    uint64_t *bar_base = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    volatile uint32_t *loads_issued = reinterpret_cast<volatile uint32_t *>(smem + kOffMisc + 16);
    int *prefix = reinterpret_cast<int *>(smem + kOffPrefix);

    Bars bars;
    bars.full = bar_base + kBarFull;
    bars.empty = bar_base + kBarEmpty;
    bars.s_full = bar_base + kBarSFull;
    bars.s_free = bar_base + kBarSFree;
    bars.p_full = bar_base + kBarPFull;
    bars.o_full = bar_base + kBarOFull;
    bars.o_free = bar_base + kBarOFree;
    bars.red = bar_base + kBarRed;
    bars.fin = bar_base + kBarFin;
    bars.full_v = bar_base + kBarFullV;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.full_v[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        constexpr uint32_t kSoftWarps = 8;                     // two warpgroups
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], kSoftWarps);
            mbar_init(&bars.p_full[i], kSoftWarps);
            mbar_init(&bars.o_full[i], 1);
            mbar_init(&bars.o_free[i], kSoftWarps);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&bars.red[i], 4);   // one arrival per warp of a warpgroup
        mbar_init(&bars.fin[0], 4);
        mbar_init(&bars.fin[1], 4);
        *abort_flag = 0;
        *loads_issued = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // Programmatic dependent launch: the merge kernel may launch now (it waits for
    // this grid to finish). The set-up above and the item order below, which reads
    // only the call's lengths, overlap the preceding kernel (the previous call's
    // merge, which writes only output rows); everything after the wait may touch
    // what that kernel reads or writes.
    asm volatile("griddepcontrol.launch_dependents;");

    // Item order (see decode_order.cuh); the byte codes use the P buffer, which is
    // unused until the first tile.
    int *order = reinterpret_cast<int *>(smem + kOffOrder);
    int *counts = reinterpret_cast<int *>(smem + kOffMisc + 8);   // [0] = n4, [1] = list length
    const decode_order::SeqCache cache{reinterpret_cast<int *>(smem + kOffCtx), reinterpret_cast<int *>(smem + kOffPs)};
    decode_order::build(p, prefix, order, counts, sP, cache);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n4 = counts[0];
    const int total_items = (counts[0] + counts[1]) * p.num_kv_heads;
    // this CTA's item descriptors, computed once and kept over the ordering arrays
    int4 *items = reinterpret_cast<int4 *>(smem + kOffPrefix);
    decode_order::build_item_table<(decode_order::kTableItems + kThreads - 1) / kThreads>(p, prefix, order, n4, cache, total_items, items);
    const int nmy = decode_order::cta_items(total_items);
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0 || warp == kVProdWarp) {
        // ------------------------------------------------------------ producers
        const bool is_v = warp == kVProdWarp;
        uint64_t *fullb = is_v ? bars.full_v : bars.full;
        const CUtensorMap *tm = is_v ? &tm_v : &tm_k;
        unsigned char *dst0 = is_v ? sV : sK;
        const int nbt = kTile / p.block_size;       // physical blocks per tile
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const decode_order::ItemTable tb = decode_order::load_item_table(p, I, lane);
            // decode with append: the slot of the sequence's new token, read here and
            // used at the item's last tile (an empty context takes only -1)
            int app_slot = -1;
            uint4 app_row = make_uint4(0, 0, 0, 0);
            if (p.app_slots != nullptr && I.last) {
                app_slot = p.app_slots[I.b];
                if (I.ntiles > 0) app_row = append_row(p, I, is_v, lane);
            }
            if (app_slot != -1 && I.ntiles == 0 && I.t1 == 0 && !is_v && lane == 0) raise_error(p.err, PA_DEVERR_SLOT);
            const int qrow = I.b * p.num_heads + I.kvh * G;
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int stage = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                bool live;
                const int e = decode_order::tile_entry(tb, tile, nbt, lane, &live);
                if (app_slot != -1 && tile == I.ntiles - 1) {
                    // lane of the token's block among this tile's blocks
                    const int jl = (((I.t1 - 1) >> p.log2_block_size) - (I.t0 >> p.log2_block_size)) - tile * nbt;
                    append_token(p, I, app_slot, __shfl_sync(0xffffffffu, e, jl), app_row, is_v, lane);
                    __syncwarp();
                }
                int phys = (int)p.num_blocks;           // out of range: TMA fills zeros
                if (live) {
                    if (e >= 0 && e < p.num_blocks) phys = e;
                    else if (!is_v) raise_error(p.err, PA_DEVERR_BLOCK_ID);
                }
                int w = 1;
                if (lane == 0) w = mbar_wait(&bars.empty[stage], ph ^ 1) ? 1 : 0;
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w || *abort_flag) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&fullb[stage], is_v ? kKVBytes : kKVBytes + kQBytes);
                __syncwarp();
                if (lane < nbt) {
                    unsigned char *d = dst0 + stage * kKVBytes + lane * p.block_size * 128;
                    tma_load_4d(d, tm, &fullb[stage], 0, I.kvh, 0, phys);
                    tma_load_4d(d + kChunkBytes, tm, &fullb[stage], 64, I.kvh, 0, phys);
                }
                if (lane == 0 && !is_v) {
                    unsigned char *dq = sQ + stage * kQBytes;
                    tma_load_2d(dq, &tm_q, &fullb[stage], 0, qrow);
                    tma_load_2d(dq + kN * 128, &tm_q, &fullb[stage], 64, qrow);
                    *loads_issued = it + 1;             // tiles whose loads are issued
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
        if (lane == 0) {
            const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
            for (uint32_t j = first; j < it; ++j) mbar_wait(&fullb[j % kStages], (j / kStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t idesc_s = instr_desc_f16(kTile, kN, kBf16, false, false);
            const uint32_t idesc_o = instr_desc_f16(kD, kN, kBf16, true, false);
            const uint32_t sK0 = smem_addr(sK), sV0 = smem_addr(sV), sQ0 = smem_addr(sQ), sP0 = smem_addr(sP);
            uint32_t it = 0;
            bool ok = true;
            for (int k = 0; k < nmy && ok; ++k) {
                const Item I = decode_order::unpack_item(items[k]);
                for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                    const int stage = it % kStages, buf = it & 1;
                    if (*abort_flag || !mbar_wait(&bars.full[stage], (it / kStages) & 1) ||
                        !mbar_wait(&bars.s_free[buf], ((it >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kbase = sK0 + stage * kKVBytes;
                    const uint32_t qbase = sQ0 + stage * kQBytes;
                    const uint32_t dcol = tmem + buf * kN;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                        const uint32_t qoff = (kk >> 2) * (kN * 128) + (kk & 3) * 32;
                        const uint64_t a = smem_desc(kbase + off, 16, 1024);
                        const uint64_t b = smem_desc(qbase + qoff, 16, 1024);
                        mma_f16(dcol, a, b, idesc_s, kk > 0);
                    }
                    mma_commit(&bars.s_full[buf]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, PA_DEVERR_WAIT);
            }
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t idesc_o = instr_desc_f16(kD, kN, kBf16, true, false);
            const uint32_t sV0 = smem_addr(sV), sP0 = smem_addr(sP);
            uint32_t it = 0;
            bool ok = true;
            auto issue_pv = [&](uint32_t j) -> bool {
                const int buf = j & 1, stage = j % kStages;
                const uint32_t bph = (j >> 1) & 1;
                if (!mbar_wait(&bars.p_full[buf], bph)) return false;
                if (!mbar_wait(&bars.o_free[buf], bph ^ 1)) return false;
                if (!mbar_wait(&bars.full_v[stage], (j / kStages) & 1)) return false;
                tc_fence_after();
                const uint32_t vbase = sV0 + stage * kKVBytes;
                const uint32_t pbase = sP0 + buf * kPBytes;
                const uint32_t dcol = tmem + 2 * kN + buf * kN;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t a = smem_desc(vbase + kk * 2048, kChunkBytes, 1024);
                    const uint64_t b = smem_desc(pbase + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
                    mma_f16(dcol, a, b, idesc_o, kk > 0);
                }
                mma_commit(&bars.o_full[buf]);
                mma_commit(&bars.empty[stage]);
                return true;
            };
            for (int k = 0; k < nmy && ok; ++k) {
                const Item I = decode_order::unpack_item(items[k]);
                for (int tile = 0; tile < I.ntiles; ++tile, ++it)
                    if (*abort_flag || !issue_pv(it)) {
                        ok = false;
                        break;
                    }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, PA_DEVERR_WAIT);
            }
        }
        __syncwarp();
    } else if (warp == 6) {
        // ------------------------------------------------------------ L2 prefetch
        // Walks the same tiles as the producer, at most kPrefetchTiles ahead of its
        // loads, pulling each tile's blocks into L2 so that the ring's loads find
        // them there. Prefetches are hints: if this warp falls behind or gives up,
        // only speed changes.
        const int nbt = kTile / p.block_size;
        uint32_t n = 0;
        bool go = true;
        for (int k = 0; k < nmy && go; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const decode_order::ItemTable tb = decode_order::load_item_table(p, I, lane);
            for (int tile = 0; tile < I.ntiles; ++tile, ++n) {
                bool live;
                int e = decode_order::tile_entry(tb, tile, nbt, lane, &live);
                if (!live) e = -1;
                if (n >= *loads_issued + kPrefetchTiles) {
                    const unsigned long long t0 = globaltimer_ns();
                    while (n >= *loads_issued + kPrefetchTiles) {
                        if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                            go = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (!go) break;
                }
                if (e >= 0 && e < p.num_blocks) {
                    tma_prefetch_4d(&tm_k, 0, I.kvh, 0, e);
                    tma_prefetch_4d(&tm_k, 64, I.kvh, 0, e);
                    tma_prefetch_4d(&tm_v, 0, I.kvh, 0, e);
                    tma_prefetch_4d(&tm_v, 64, I.kvh, 0, e);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax / output
        // Warpgroup wg handles query columns [c0, c0 + kC) of every tile.
        constexpr int kC = GT / 2;
        const int wg = warp >= kWg2Warp ? 1 : 0;
        const int c0 = wg * kC;
        const int q4 = warp & 3;                       // tensor-memory lane quadrant
        const int row = q4 * 32 + lane;                // token (S) or dim (O) of this thread
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        uint64_t *red_bar = bars.red + 2 * wg;
        uint64_t *fin_bar = bars.fin + wg;
        T *out = reinterpret_cast<T *>(p.out);
        uint32_t it = 0, nfin = 0;              // tile counter; uses of the finalize barrier
        bool ok = true;
        float m_run[kC], l_part[kC], o_acc[kC], alpha_prev[kC];
        // An item's finish (its last tile's O, the sum of l over the warps, the output)
        // is deferred until the next item's first tile has been through the softmax, so
        // the warpgroup does not wait for the last P.V at every item boundary: this is
        // the item waiting for it. Measured per instance: long context (G = 8) 0.3955 ->
        // 0.3933 ms, the sharing-aware batch's joining pass (G = 4) 0.0699 -> 0.0690 ms,
        // but the 8B-shaped batch (G = 4) 0.0931 -> 0.0943 ms; the other instances
        // finish each item at its end.
        constexpr bool kDefer = kFold || GT == 8;
        bool pend = false;
        uint32_t pend_it = 0;                     // the tile whose O completes it
        int64_t pend_head0 = 0;
        int pend_slot = 0;
        bool pend_direct = false, pend_fold = false;
        float pm[kC], pl[kC], po[kC], pa[kC], pfm[kC], pfl[kC], pfo[kC];
        // this warpgroup's columns of a tile's accumulator at tensor-memory column `col`
        // (8 columns loaded; the first kC are this warpgroup's)
        auto load_cols = [&](uint32_t col, float *v) { tmem_ld8(tmem + lane_off + col + c0, v); };
        // acc = acc * alpha + O of tile j
        auto accumulate = [&](uint32_t j, float *acc, const float *alpha) -> bool {
            const int buf = j & 1;
            if (!warp_wait(&bars.o_full[buf], (j >> 1) & 1)) return false;
            tc_fence_after();
            float o[8];
            load_cols(2 * kN + buf * kN, o);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.o_free[buf]);
#pragma unroll
            for (int u = 0; u < kC; ++u) acc[u] = fmaf(acc[u], alpha[u], o[u]);
            return true;
        };
        // An item's output: the sum of the token lanes' partial l per head (lred is
        // double-buffered by finish parity: one barrier per item), then the final row,
        // the join with the shared pass's partial, or this partition's partial.
        auto finish = [&](int64_t head0, int slot, bool direct, bool fold, const float *m, const float *lp,
                          const float *acc, const float *fm, const float *fl, const float *fo) -> bool {
            float *lr = lred + (nfin & 1) * 4 * kN;
#pragma unroll
            for (int u = 0; u < kC; ++u) {
                const float ls = warp_sum(lp[u]);
                if (lane == 0) lr[q4 * kN + c0 + u] = ls;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(fin_bar);
            if (!warp_wait(fin_bar, nfin++ & 1)) return false;
            float l_tot[kC];
#pragma unroll
            for (int u = 0; u < kC; ++u) {
                const int g = c0 + u;
                l_tot[u] = lr[g] + lr[kN + g] + lr[2 * kN + g] + lr[3 * kN + g];
            }
            if (kFold && fold) {
                // the shared pass's partial of these heads (slot 0, written before this
                // kernel) joined with this item's: one softmax over the whole context
#pragma unroll
                for (int u = 0; u < kC; ++u) {
                    if (c0 + u < G) {
                        const float M = fmaxf(m[u], fm[u]);
                        const float f = m[u] == -INFINITY ? 0.f : fast_exp2(m[u] - M);
                        const float fs = fm[u] == -INFINITY ? 0.f : fast_exp2(fm[u] - M);
                        const float num = fmaf(fo[u], fs, acc[u] * f), den = fmaf(fl[u], fs, l_tot[u] * f);
                        out[(head0 + c0 + u) * kD + row] = Elem<T>::from_f(num / den);
                    }
                }
            } else if (direct) {
#pragma unroll
                for (int u = 0; u < kC; ++u)
                    if (c0 + u < G) out[(head0 + c0 + u) * kD + row] = Elem<T>::from_f(acc[u] / l_tot[u]);
            } else {
                const int P = p.max_partitions;
#pragma unroll
                for (int u = 0; u < kC; ++u) {
                    if (c0 + u < G) {
                        const int64_t r = (head0 + c0 + u) * P + slot;
                        p.ws_o[r * kD + row] = acc[u];
                        if (row == 0) {
                            p.ws_ml[2 * r] = m[u];
                            p.ws_ml[2 * r + 1] = l_tot[u];
                        }
                    }
                }
            }
            return true;
        };
        auto finish_pending = [&]() -> bool {
            if constexpr (!kDefer) return true;
            if (!pend) return true;
            pend = false;
            return accumulate(pend_it, po, pa) &&
                   finish(pend_head0, pend_slot, pend_direct, pend_fold, pm, pl, po, pfm, pfl, pfo);
        };
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const int64_t head0 = (int64_t)I.b * p.num_heads + (int64_t)I.kvh * G;
            // joining the shared pass's partial (kFold: one slot, since one partition
            // covers the whole context): loaded now so the loads overlap the tiles
            const bool fold = kFold && I.slot > 0;
            float f_m[kC], f_l[kC], f_o[kC];
            if constexpr (kFold) {
                if (fold) {
#pragma unroll
                    for (int u = 0; u < kC; ++u) {
                        const int64_t r0 = (head0 + (c0 + u < G ? c0 + u : 0)) * p.max_partitions;
                        f_m[u] = p.ws_ml[2 * r0];
                        f_l[u] = p.ws_ml[2 * r0 + 1];
                        f_o[u] = p.ws_o[r0 * kD + row];
                    }
                }
            }
            if (I.ntiles == 0 && !fold) {
#pragma unroll
                for (int u = 0; u < kC; ++u)
                    if (c0 + u < G) out[(head0 + c0 + u) * kD + row] = Elem<T>::from_f(0.f);
                continue;
            }
#pragma unroll
            for (int u = 0; u < kC; ++u) {
                m_run[u] = -INFINITY;
                l_part[u] = 0.f;
                o_acc[u] = 0.f;
                alpha_prev[u] = 0.f;
            }
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int buf = it & 1, stage = it % kStages;
                if (__any_sync(0xffffffffu, *abort_flag != 0) || !warp_wait(&bars.s_full[buf], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[8];
                load_cols(buf * kN, s);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.s_free[buf]);

                const int tok = I.t0 + tile * kTile + row;
                const bool valid = tok < I.t1;
                float* rd = red + (it & 1) * 4 * kN;
#pragma unroll
                for (int u = 0; u < kC; ++u) {
                    const int g = c0 + u;
                    s[u] = valid ? s[u] * p.scale_log2 : -INFINITY;
                    const float mx = warp_max(s[u]);
                    if (lane == 0) rd[q4 * kN + g] = mx;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&red_bar[it & 1]);
                if (!warp_wait(&red_bar[it & 1], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                float alpha[kC];
                unsigned char *pb = sP + buf * kPBytes + (row >> 6) * (kN * 128);
                const int colb = (row & 63) * 2;
#pragma unroll
                for (int u = 0; u < kC; ++u) {
                    const int g = c0 + u;
                    const float tmax = fmaxf(fmaxf(rd[g], rd[kN + g]), fmaxf(rd[2 * kN + g], rd[3 * kN + g]));
                    const float m_new = fmaxf(m_run[u], tmax);
                    alpha[u] = fast_exp2(m_run[u] - m_new);
                    m_run[u] = m_new;
                    const uint16_t bits = to_bits<T>(valid ? fast_exp2(s[u] - m_new) : 0.f);
                    l_part[u] = fmaf(l_part[u], alpha[u], from_bits<T>(bits));
                    // P^T element (row n = g, column k = token) in a 128-byte swizzled K-major tile
                    unsigned char *dst = pb + g * 128 + ((((colb >> 4) ^ (g & 7)) << 4) | (colb & 15));
                    *reinterpret_cast<uint16_t *>(dst) = bits;
                }
                // masked token: its V row may hold anything (NaN included) and P = 0,
                // so zero the row once the stage's copies have landed (first warpgroup)
                if (wg == 0) {
                    if (__any_sync(0xffffffffu, !valid) && !warp_wait(&bars.full_v[stage], (it / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    if (!valid) {
                        uint4 *v0 = reinterpret_cast<uint4 *>(sV + stage * kKVBytes + row * 128);
                        uint4 *v1 = reinterpret_cast<uint4 *>(sV + stage * kKVBytes + kChunkBytes + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {       // rotated by row: no bank conflicts
                            v0[c ^ (row & 7)] = make_uint4(0, 0, 0, 0);
                            v1[c ^ (row & 7)] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full[buf]);
                // the previous tile's O: this item's, or the last tile of the item before
                if (tile > 0 ? !accumulate(it - 1, o_acc, alpha_prev) : !finish_pending()) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int u = 0; u < kC; ++u) alpha_prev[u] = alpha[u];
            }
            if (!ok) break;
            if (I.ntiles == 0) {
                // a join with no tiles of its own (kFold): nothing to defer
                if (!finish_pending() || !finish(head0, I.slot, I.direct, fold, m_run, l_part, o_acc, f_m, f_l, f_o)) {
                    ok = false;
                    break;
                }
                continue;
            }
            if constexpr (!kDefer) {
                if (!accumulate(it - 1, o_acc, alpha_prev) ||
                    !finish(head0, I.slot, I.direct, fold, m_run, l_part, o_acc, f_m, f_l, f_o)) {
                    ok = false;
                    break;
                }
                continue;
            }
            pend = true;
            pend_it = it - 1;
            pend_head0 = head0;
            pend_slot = I.slot;
            pend_direct = I.direct;
            pend_fold = fold;
#pragma unroll
            for (int u = 0; u < kC; ++u) {
                pm[u] = m_run[u];
                pl[u] = l_part[u];
                po[u] = o_acc[u];
                pa[u] = alpha_prev[u];
                if constexpr (kFold) {
                    pfm[u] = f_m[u];
                    pfl[u] = f_l[u];
                    pfo[u] = f_o[u];
                }
            }
        }
        if (ok && !finish_pending()) ok = false;
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side -----------------------------------------------------------------

bool make_cache_map(CUtensorMap *m, const void *base, const DecodeParams &p, CUtensorMapDataType dt) {
    return make_kv_cache_map(m, base, p.num_blocks, p.block_size, p.num_kv_heads, dt);
}

bool make_q_map(CUtensorMap *m, const DecodeParams &p, CUtensorMapDataType dt) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.num_seqs * p.num_heads};
    cuuint64_t strides[1] = {kD * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kN};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(p.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int GT, bool kFold>
int launch_tc_t(const DecodeParams &p, CUtensorMapDataType dt, cudaStream_t stream) {
    auto kern = decode_tc_kernel<T, GT, kFold>;
    static bool attr_set[kMaxDevices] = {};
    static int num_sms[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
            return -1;
        if (cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        attr_set[dev] = true;
    }
    CUtensorMap mk, mv, mq;
    if (!make_cache_map(&mk, p.key_cache, p, dt) || !make_cache_map(&mv, p.value_cache, p, dt) ||
        !make_q_map(&mq, p, dt))
        return -1;
    const int64_t max_items = (int64_t)p.num_seqs * p.num_kv_heads * p.max_partitions;
    const int grid = (int)(max_items < num_sms[dev] ? max_items : num_sms[dev]);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, stream, mk, mv, mq, p);
}

// The joining instance (fold_shared) exists for groups of up to 8 heads; the host sets
// fold_shared only there.
template <typename T>
int launch_tc_g(const DecodeParams &p, CUtensorMapDataType dt, cudaStream_t stream) {
    if (p.fold_shared) {
        if (p.group <= 4) return launch_tc_t<T, 4, true>(p, dt, stream);
        if (p.group <= 8) return launch_tc_t<T, 8, true>(p, dt, stream);
        return -2;
    }
    if (p.group <= 4) return launch_tc_t<T, 4, false>(p, dt, stream);
    if (p.group <= 8) return launch_tc_t<T, 8, false>(p, dt, stream);
    return launch_tc_t<T, 16, false>(p, dt, stream);
}

}  // namespace

bool decode_tc_supported(const DecodeParams &p, int dtype) {
    return (dtype == PA_DTYPE_BF16 || dtype == PA_DTYPE_F16) && p.head_dim == kD && p.group >= 1 &&
           p.group <= kN && p.block_size >= 8 && p.block_size <= kTile && p.partition_size % kTile == 0 &&
           p.num_blocks < INT32_MAX && (int64_t)p.num_seqs * p.num_heads < INT32_MAX;
}

// Batches above kMaxSeqs sequences run as independent launches of up to kMaxSeqs
// sequences (the sequences share nothing but the cache).
int launch_decode_tc(const DecodeParams &p, int dtype, cudaStream_t stream) {
    if (!decode_tc_supported(p, dtype)) return -2;
    // sequences per launch: at most kMaxSeqs, and few enough that no CTA gets more
    // than the item table holds (items <= num_seqs * kv heads * partitions)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    const int64_t per_seq = (int64_t)p.num_kv_heads * p.max_partitions;
    const int64_t by_items = (int64_t)decode_order::kTableItems * sms / (per_seq > 0 ? per_seq : 1);
    const int chunk = (int)(by_items < 1 ? 1 : (by_items < kMaxSeqs ? by_items : kMaxSeqs));
    for (int b0 = 0; b0 < p.num_seqs; b0 += chunk) {
        DecodeParams c = p;
        const int64_t rows = (int64_t)b0 * p.num_heads;
        c.num_seqs = min(chunk, p.num_seqs - b0);
        c.q = static_cast<const char *>(p.q) + rows * kD * 2;
        c.out = static_cast<char *>(p.out) + rows * kD * 2;
        c.block_tables = p.block_tables + (int64_t)b0 * p.max_blocks_per_seq;
        c.context_lens = p.context_lens + b0;
        if (p.prefix_lens) c.prefix_lens = p.prefix_lens + b0;
        if (p.app_slots) {
            c.app_slots = p.app_slots + b0;
            c.app_k = static_cast<const char *>(p.app_k) + (int64_t)b0 * p.num_kv_heads * kD * 2;
            c.app_v = static_cast<const char *>(p.app_v) + (int64_t)b0 * p.num_kv_heads * kD * 2;
        }
        if (p.ws_ml) {
            c.ws_ml = p.ws_ml + rows * p.max_partitions * 2;
            c.ws_o = p.ws_o + rows * p.max_partitions * kD;
        }
        const int rc = dtype == PA_DTYPE_BF16
                           ? launch_tc_g<__nv_bfloat16>(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, stream)
                           : launch_tc_g<__half>(c, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, stream);
        if (rc != 0) return rc;
    }
    return 0;
}

}  // namespace pa
