// Chunked-prefill attention over the paged cache on the sm_100 tensor cores.
//
// The paged step of "CS349E lecture 7: 01_paged_attention.py" (demo 1, demo 2)
// writes a chunk's K/V into its blocks and then lets every position of the
// chunk attend; "04 - Paged Attention 实现进度" B.2/D.2 packs the chunks of a
// batch with cu_seqlens_q (query_start_loc). Query row i of sequence b sits at
// position ctx_b - q_len_b + i and attends to positions 0..pos (causal), each
// query head h reading kv head h / G. For every (row, head) the result is one
// softmax over its visible keys, taken online here: a running max and sum per
// row, with the accumulated output rescaled when the max grows.
//
// Work item = (sequence, kv head, tile of query tokens). The item's 128 MMA
// rows are (query token, head of the group) pairs: QT = 128 / Gp tokens x Gp
// heads, Gp = G rounded up to a power of two. Per tile of 128 keys:
//   S[128 rows x 128 keys] = Q . K^T    (tcgen05 kind::f16, M=128 N=128 K=128,
//                                        Q from tensor memory, K from shared memory)
//   O[128 rows x 128 dims] += P . V     (P from tensor memory, V MN-major)
// Tensor memory (512 columns): S double-buffered (256), O (128), the item's query
// rows Q (64, 16-bit pairs per lane) and P (64, 16-bit pairs per lane). With both
// operands of the S MMA in shared memory, it and the TMA writes of each tile's K
// and V moved about 160 KB of shared memory per tile; with Q in tensor memory the S
// MMA reads only K. P is written by the softmax threads (each thread's row is its
// lane), where the P.V MMA takes its A operand, so P makes no shared-memory round
// trip; it is single-buffered: tile j's softmax writes it once P(j-1).V has run.
// Thread = row for the softmax, so the max and the sum are thread-local; O is
// rescaled (tcgen05.ld / st of the row) only when a row's max grows by more than
// 2^8, otherwise the stale reference max is kept (the final O / l is the same).
// The row sum adds the fp32 weights; the P.V MMA sees them rounded to 16 bits (a
// relative difference of at most 2^-9 per weight, of either sign). The exponent
// arguments and the sums use the paired fp32 instructions (two lanes each).
//
// Roles (256 threads, one persistent CTA per SM):
//   warp 0     TMA: per key tile the K boxes of each physical block into a
//              2-stage K ring.
//   warp 6     TMA: the V boxes of every key tile into a 2-stage V ring with its
//              own barriers (K freed after its S MMA, V after its P.V MMA). Each
//              producer reads an item's block ids once, coalesced, at item start;
//              blocks past the last visible key load from an out-of-range
//              coordinate (zeros). With one producer warp for both operands the
//              producer was busy 95 % of the time and the MMA waited on K.
//   warp 7     TMA: each item's query rows (3-D map over [tokens, heads, dims];
//              group mode: one 2-D box per member) into shared memory, as soon
//              as the previous item's rows have moved to tensor memory.
//   warp 1     one thread issues the MMAs and owns tensor memory.
//   warps 2-5  softmax (scale, causal mask, exp2, P to tensor memory, V rows of
//              keys past the last visible one zeroed), the copy of the next
//              item's query rows from shared to tensor memory once this item's
//              last S has been read (its S MMAs then run during this epilogue),
//              and the epilogue O / l.
// Items differ in size by up to the context length (key tiles = causal extent
// / 128), and a persistent CTA ends with its last item: dealt in index order the
// most loaded CTA of the chunked-prefill batch had 13 % more key tiles than the
// mean. So each CTA first sorts the (sequence, query tile) entries by key-tile
// count, largest first (a counting sort, stable by index, so every CTA derives
// the same order), and takes every grid-th item of that list in serpentine
// rounds; an entry's kv heads stay adjacent. Batches too large for the sort's
// scratch (which lives in the K/V rings before the first load) keep index order.
// Every wait is bounded; on a timeout the kernel sets PA_DEVERR_WAIT and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "prefill_common.cuh"
#include "sm100.cuh"
#include "tma_maps.cuh"

namespace pa {
namespace {

using namespace sm100;
using namespace prefill;

constexpr int kD = 128;
constexpr int kRows = 128;                     // MMA rows per item
constexpr int kKStages = 2;                    // K ring
constexpr int kVStages = 2;                    // V ring
constexpr int kChunk = 128 * 128;              // 128 rows x 128 bytes (one 64-element half)
constexpr int kKVBytes = 2 * kChunk;           // one K (or V) tile
constexpr int kQBytes = 2 * kChunk;
constexpr int kThreads = 256;                  // + warp 6: V producer, warp 7: Q producer
constexpr int kVProdWarp = 6;
constexpr int kQProdWarp = 7;
constexpr uint32_t kTmemCols = 512;            // S[2] x 128 + O x 128 + Q x 64 + P x 64
constexpr uint32_t kColO = 2 * kKT;
constexpr uint32_t kColQ = 3 * kKT;            // the item's query rows: 16-bit pairs per lane (row)
constexpr uint32_t kColP = 3 * kKT + 64;       // P: 64 columns, 16-bit pairs per lane (row)
constexpr float kRescaleLog2 = 8.f;            // keep the reference max until a row's max grows by 2^8

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kKVBytes;
constexpr int kOffQ = kOffV + kVStages * kKVBytes;
constexpr int kOffBar = kOffQ + kQBytes;
constexpr int kNumBars = 22;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kMaxMyItems = 1024;              // a CTA's items after the sort
constexpr int kOffMy = kOffMisc + 16;          // int [kMaxMyItems]: this CTA's items, in order
constexpr int kSmemUsed = kOffMy + kMaxMyItems * 4;
// sort scratch, in the K/V rings (unused until the first load)
constexpr int kOffSortSize = kOffK;                                  // uint16 [kSortMaxEntries]
constexpr int kOffSorted = kOffSortSize + 2 * kSortMaxEntries;       // uint16 [kSortMaxEntries]
constexpr int kOffCursor = kOffSorted + 2 * kSortMaxEntries;         // int [kSortBuckets]
static_assert(kOffCursor + 4 * kSortBuckets <= kOffQ, "sort scratch fits the rings");
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// 32 lanes x 64 consecutive 32-bit columns, issued without waiting.
__device__ __forceinline__ void tmem_ld64_nowait(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}
// Wait for the tensor-memory loads issued so far; the registers' uses follow the wait.
template <int N> __device__ __forceinline__ void tmem_wait_ld_pinned(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

template <typename T, bool kGroup>
__global__ __launch_bounds__(kThreads, 1) void prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                 const __grid_constant__ CUtensorMap tm_v,
                                                                 const __grid_constant__ CUtensorMap tm_q,
                                                                 const PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sK = smem + kOffK;
    unsigned char *sV = smem + kOffV;
    unsigned char *sQ = smem + kOffQ;
    uint64_t *bb = reinterpret_cast<uint64_t *>(smem + kOffBar);
    // K and V stages have separate barriers: a K stage is free again as soon as its
    // S MMA is done, a V stage only after its P.V MMA.
    uint64_t *k_full = bb, *k_empty = bb + 3, *v_full = bb + 6, *v_empty = bb + 8;
    uint64_t *s_full = bb + 10, *s_free = bb + 12, *p_full = bb + 14, *o_done = bb + 16;
    uint64_t *q_full = bb + 18, *q_empty = bb + 19, *o_free = bb + 20, *q_tm = bb + 21;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group, Gp = p.group_pad;
    const int total_items = kGroup ? p.num_groups * p.num_kv_heads * p.shared_parts
                                   : p.num_seqs * p.num_kv_heads * p.qtiles;

    if (tid == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 4);           // the softmax warps, the rows copied to tensor memory
        mbar_init(q_tm, 4);              // the same arrivals: Q is in tensor memory
        mbar_init(o_free, 4);
        *abort_flag = 0;
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
    // a decode launched after this kernel (the sharing-aware decode's per-sequence
    // pass) may set itself up now; it waits for this grid before reading its partials
    asm volatile("griddepcontrol.launch_dependents;");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the items of this CTA: a sorted list, or every grid-th index
    int *my_items = reinterpret_cast<int *>(smem + kOffMy);
    bool use_list = false;
    int nloop = total_items > (int)blockIdx.x ? (total_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    if constexpr (!kGroup) {
        if (p.sorted_items) {
            use_list = true;
            const int E = p.num_seqs * p.qtiles, Hk = p.num_kv_heads, qtiles = p.qtiles;
            nloop = sort_items(
                E, Hk, [&](int e) { return qtile_tiles(p, e / qtiles, e % qtiles, true); },
                reinterpret_cast<uint16_t *>(smem + kOffSortSize), reinterpret_cast<uint16_t *>(smem + kOffSorted),
                reinterpret_cast<int *>(smem + kOffCursor), my_items, kMaxMyItems);
            // (entry, kv head) -> item index
            for (int k = tid; k < nloop; k += kThreads) {
                const int e = my_items[k] / Hk, kvh = my_items[k] - (my_items[k] / Hk) * Hk;
                const int b = e / qtiles, qt = e - b * qtiles;
                my_items[k] = (b * Hk + kvh) * qtiles + qt;
            }
            __syncthreads();
        }
    }
    // Group mode is launched as a programmatic dependent: the set-up above, which
    // reads only the call's lengths, overlaps the preceding kernel; everything below
    // may touch what it reads or writes.
    if constexpr (kGroup) asm volatile("griddepcontrol.wait;" ::: "memory");
    auto item_at = [&](int k) { return use_list ? my_items[k] : (int)blockIdx.x + k * (int)gridDim.x; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer: K
        // Per key tile its K boxes, into a 2-stage ring. The item's block ids are read
        // once at item start.
        const int nbt = kKT / p.block_size;
        uint32_t it = 0;                                // K tiles issued
        bool ok = true;
        for (int k = 0; k < nloop && ok; ++k) {
            const int idx = item_at(k);
            PItem I;
            if (!(kGroup ? get_gitem(idx, p, I) : get_pitem(idx, p, I))) continue;
            const KeyTable tb = load_key_table(p, I, lane);
            for (int j = 0; j < I.ntiles; ++j, ++it) {
                const int stage = it % kKStages;
                const uint32_t ph = (it / kKStages) & 1;
                const int phys = tile_block(tb, p, j, nbt, lane, true);
                int w = 1;
                if (lane == 0) w = mbar_wait(&k_empty[stage], ph ^ 1) ? 1 : 0;
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w || *abort_flag) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&k_full[stage], kKVBytes);
                __syncwarp();
                if (lane < nbt) {
                    unsigned char *dk = sK + stage * kKVBytes + lane * p.block_size * 128;
                    tma_load_4d(dk, &tm_k, &k_full[stage], 0, I.kvh, 0, phys);
                    tma_load_4d(dk + kChunk, &tm_k, &k_full[stage], 64, I.kvh, 0, phys);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
        if (lane == 0)   // drain copies in flight
            for (uint32_t j = it > (uint32_t)kKStages ? it - kKStages : 0; j < it; ++j)
                mbar_wait(&k_full[j % kKStages], (j / kKStages) & 1);
    } else if (warp == kQProdWarp) {
        // ------------------------------------------------------------ TMA producer: Q
        // Each item's query rows as soon as the previous item's rows have gone to tensor
        // memory, so the load overlaps the item before.
        if (lane == 0) {
            uint32_t n = 0;                             // items issued
            bool ok = true;
            for (int k = 0; k < nloop && ok; ++k) {
                const int idx = item_at(k);
                PItem I;
                if (!(kGroup ? get_gitem(idx, p, I) : get_pitem(idx, p, I))) continue;
                if (*abort_flag || !mbar_wait(q_empty, (n & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(q_full, kQBytes);
                if constexpr (kGroup) {
                    // one box of Gp head rows per member slot; empty slots read zeros
                    const int32_t *mem = p.group_members + (int64_t)I.group * p.max_members;
                    for (int m = 0; m < p.rows_q; ++m) {
                        const int row = m < I.members ? mem[m] * p.num_heads + I.kvh * G : p.num_seqs * p.num_heads;
                        tma_load_2d(sQ + m * Gp * 128, &tm_q, q_full, 0, row);
                        tma_load_2d(sQ + kChunk + m * Gp * 128, &tm_q, q_full, 64, row);
                    }
                } else {
                    tma_load_3d(sQ, &tm_q, q_full, 0, I.kvh * G, I.q_row0);
                    tma_load_3d(sQ + kChunk, &tm_q, q_full, 64, I.kvh * G, I.q_row0);
                }
                ++n;
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, PA_DEVERR_WAIT);
            }
            if (n > 0) mbar_wait(q_full, (n - 1) & 1);   // drain the copy in flight
        }
        __syncwarp();
    } else if (warp == kVProdWarp) {
        // ------------------------------------------------------------ TMA producer: V
        const int nbt = kKT / p.block_size;
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < nloop && ok; ++k) {
            const int idx = item_at(k);
            PItem I;
            if (!(kGroup ? get_gitem(idx, p, I) : get_pitem(idx, p, I))) continue;
            const KeyTable tb = load_key_table(p, I, lane);
            for (int j = 0; j < I.ntiles; ++j, ++it) {
                const int stage = it & 1;
                const int phys = tile_block(tb, p, j, nbt, lane, false);
                int w = 1;
                if (lane == 0) w = mbar_wait(&v_empty[stage], ((it >> 1) & 1) ^ 1) ? 1 : 0;
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w || *abort_flag) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&v_full[stage], kKVBytes);
                __syncwarp();
                if (lane < nbt) {
                    unsigned char *dv = sV + stage * kKVBytes + lane * p.block_size * 128;
                    tma_load_4d(dv, &tm_v, &v_full[stage], 0, I.kvh, 0, phys);
                    tma_load_4d(dv + kChunk, &tm_v, &v_full[stage], 64, I.kvh, 0, phys);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
        if (lane == 0)
            for (uint32_t j = it > 2u ? it - 2 : 0; j < it; ++j) mbar_wait(&v_full[j & 1], (j >> 1) & 1);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t idesc_s = instr_desc_f16(kRows, kKT, kBf16, false, false);
            const uint32_t idesc_o = instr_desc_f16(kRows, kD, kBf16, false, true);
            const uint32_t sK0 = smem_addr(sK), sV0 = smem_addr(sV);
            uint32_t it = 0, n = 0;
            bool ok = true;
            // O += P(j) V(j); `first` starts the item's accumulator
            auto issue_pv = [&](uint32_t j, bool first) -> bool {
                if (first && n > 1 && !mbar_wait(o_free, (n - 2) & 1)) return false;
                if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1)) return false;
                if (!mbar_wait(&v_full[j & 1], (j >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t vb = sV0 + (j & 1) * kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kKT / 16; ++kk) {
                    const uint64_t b = smem_desc(vb + kk * 2048, kChunk, 1024);
                    mma_f16_tmem_a(tmem + kColO, tmem + kColP + kk * 8, b, idesc_o,
                                   (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(&o_done[j & 1]);
                mma_commit(&v_empty[j & 1]);
                return true;
            };
            for (int k = 0; k < nloop && ok; ++k) {
                const int idx = item_at(k);
                PItem I;
                if (!(kGroup ? get_gitem(idx, p, I) : get_pitem(idx, p, I))) continue;
                if (!mbar_wait(q_tm, n & 1)) {
                    ok = false;
                    break;
                }
                ++n;
                for (int j = 0; j < I.ntiles; ++j, ++it) {
                    const int stage = it & 1;                 // S buffer
                    const int kst = it % kKStages;            // K stage
                    if (*abort_flag || !mbar_wait(&k_full[kst], (it / kKStages) & 1) ||
                        !mbar_wait(&s_free[stage], ((it >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kb = sK0 + kst * kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {       // A = Q from tensor memory, B = K
                        const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
                        mma_f16_tmem_a(tmem + stage * kKT, tmem + kColQ + kk * 8, smem_desc(kb + off, 16, 1024),
                                       idesc_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&s_full[stage]);
                    mma_commit(&k_empty[kst]);
                    if (j > 0 && !issue_pv(it - 1, j == 1)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                if (!issue_pv(it - 1, I.ntiles == 1)) {
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
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------------------ softmax / epilogue
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                 // MMA row of this thread (and key row for V zeroing)
        const int gshift = 31 - __clz(Gp);
        const int qi = r >> gshift, g = r & (Gp - 1);
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        T *out = reinterpret_cast<T *>(p.out);
        uint32_t it = 0, n = 0;
        bool ok = true;
        // Item n's query rows, from the TMA tile in shared memory (128-byte rows, 16-byte
        // chunks rotated by row) to Q in tensor memory, where the S MMAs take their A
        // operand; then the shared tile is free for the next item's rows.
        auto copy_q = [&](uint32_t nq_idx) -> bool {
            if (!warp_wait(q_full, nq_idx & 1)) return false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 *row = reinterpret_cast<const uint4 *>(sQ + h * kChunk + r * 128);
                uint32_t qv[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = row[c ^ (r & 7)];
                    qv[4 * c] = x.x;
                    qv[4 * c + 1] = x.y;
                    qv[4 * c + 2] = x.z;
                    qv[4 * c + 3] = x.w;
                }
                tmem_st32(tmem + lane_off + kColQ + h * 32, qv);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(q_empty);
                mbar_arrive(q_tm);
            }
            return true;
        };
        auto valid_item = [&](int kk) {
            PItem J;
            return kGroup ? get_gitem(item_at(kk), p, J) : get_pitem(item_at(kk), p, J);
        };
        for (int k = 0; k < nloop && ok; ++k) {
            const int idx = item_at(k);
            PItem I;
            if (!(kGroup ? get_gitem(idx, p, I) : get_pitem(idx, p, I))) continue;
            if (n == 0 && !copy_q(0)) {
                ok = false;
                break;
            }
            const bool row_valid = qi < I.nq && g < G;
            // causal position (prefill), or the last shared key (group mode: no causal limit)
            const int pos = !row_valid ? -1 : (kGroup ? I.kmax - 1 : I.pos_first + qi);
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < I.ntiles; ++j, ++it) {
                const int buf = it & 1;
                if (__any_sync(0xffffffffu, *abort_flag != 0) || !warp_wait(&s_full[buf], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[kKT];
                tmem_ld64_nowait(tmem + lane_off + buf * kKT, sr);          // both halves in flight,
                tmem_ld64_nowait(tmem + lane_off + buf * kKT + 64, sr + 64);  // then one wait
                tmem_wait_ld_pinned<kKT>(sr);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[buf]);

                // Raw scores; the scale (> 0) is folded into the exponent below. Only tiles
                // reaching past the item's first position need the causal mask.
                const int k0 = I.key0 + j * kKT;
                if (k0 + kKT - 1 > I.pos_first) {
#pragma unroll
                    for (int c = 0; c < kKT; ++c)
                        if (k0 + c > pos) sr[c] = __float_as_uint(-INFINITY);
                }
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(sr[e]);
#pragma unroll
                for (int c = 8; c < kKT; c += 8) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], __uint_as_float(sr[c + e]));
                }
                const float m_raw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                          fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const float m_tile = m_raw * p.scale_log2;
                const bool grow = m_tile > m_ref + kRescaleLog2;
                const float alpha = grow ? fast_exp2(m_ref - m_tile) : 1.f;
                if (grow) m_ref = m_tile;
                l *= alpha;
                if (__any_sync(0xffffffffu, grow && j > 0)) {
                    // O holds tiles up to j-1: rescale it once their MMA has finished
                    const uint32_t pj = it - 1;
                    if (!warp_wait(&o_done[pj & 1], (pj >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_off + kColO + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_off + kColO + c * 32, o);
                    }
                    tmem_wait_st();
                }
                const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;    // rows with no visible key: p = 0
                float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(neg_m, neg_m);
                // the weights in registers first (keys as 16-bit pairs), so they are computed
                // while the previous tile's P.V runs; P is stored once that MMA has read it
                uint32_t pw[64];
#pragma unroll
                for (int q = 0; q < 64; ++q) {
                    const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1])),
                                           sc2, nm2);
                    const float2 pv = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                    pw[q] = pack2<T>(pv.x, pv.y);
                    ls2[q & 1] = fadd2(ls2[q & 1], pv);
                }
                // P was last read by the MMA of tile it-1
                if (it >= 1 && !warp_wait(&o_done[(it - 1) & 1], ((it - 1) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st32(tmem + lane_off + kColP, pw);
                tmem_st32(tmem + lane_off + kColP + 32, pw + 32);
                tmem_wait_st();
                l += (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
                // key row r past every row's last visible key: its slot may hold anything
                const bool zero_v = k0 + r >= I.kmax;
                if (__any_sync(0xffffffffu, zero_v) && !warp_wait(&v_full[buf], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (zero_v) {
                    uint4 *v0 = reinterpret_cast<uint4 *>(sV + buf * kKVBytes + r * 128);
                    uint4 *v1 = reinterpret_cast<uint4 *>(sV + buf * kKVBytes + kChunk + r * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {           // rotated by row: no bank conflicts
                        v0[c ^ (r & 7)] = make_uint4(0, 0, 0, 0);
                        v1[c ^ (r & 7)] = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[buf]);
            }
            if (!ok) break;
            // The next item's query rows, now that every S MMA of this one has run: its S
            // MMAs then proceed during this epilogue.
            {
                int k2 = k + 1;
                while (k2 < nloop && !valid_item(k2)) ++k2;
                if (k2 < nloop && !copy_q(n + 1)) {
                    ok = false;
                    break;
                }
            }
            // ---- epilogue: O / l of this item's rows
            const uint32_t last = it - 1;
            if (!warp_wait(&o_done[last & 1], (last >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if constexpr (kGroup) {
                // split-K partial of this member row: unnormalised O, reference max, sum
                const int64_t wrow = row_valid ? ((int64_t)p.group_members[(int64_t)I.group * p.max_members + qi] *
                                                      p.num_heads + I.kvh * G + g) * p.max_partitions + I.slot
                                               : 0;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[64];
                    tmem_ld64(tmem + lane_off + kColO + c * 64, o);
                    if (row_valid) {
                        float4 *dst = reinterpret_cast<float4 *>(p.ws_o + wrow * kD + c * 64);
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            dst[u] = make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]),
                                                 __uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3]));
                    }
                }
                if (row_valid) *reinterpret_cast<float2 *>(p.ws_ml + 2 * wrow) = make_float2(m_ref, l);
            } else {
            const float inv = row_valid ? 1.f / l : 0.f;
            T *orow = out + ((int64_t)(I.q_row0 + qi) * p.num_heads + I.kvh * G + g) * kD;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t o[64];
                tmem_ld64(tmem + lane_off + kColO + c * 64, o);
                if (row_valid) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        uint4 pk;
                        pk.x = pack2<T>(__uint_as_float(o[u * 8 + 0]) * inv, __uint_as_float(o[u * 8 + 1]) * inv);
                        pk.y = pack2<T>(__uint_as_float(o[u * 8 + 2]) * inv, __uint_as_float(o[u * 8 + 3]) * inv);
                        pk.z = pack2<T>(__uint_as_float(o[u * 8 + 4]) * inv, __uint_as_float(o[u * 8 + 5]) * inv);
                        pk.w = pack2<T>(__uint_as_float(o[u * 8 + 6]) * inv, __uint_as_float(o[u * 8 + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + c * 64 + u * 8) = pk;
                    }
                }
            }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            ++n;
        }
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

template <typename T, bool kGroup>
int launch_prefill_t(const PrefillParams &p, CUtensorMapDataType dt, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<T, kGroup>;
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
    if (!make_kv_cache_map(&mk, p.key_cache, p.num_blocks, p.block_size, p.num_kv_heads, dt) ||
        !make_kv_cache_map(&mv, p.value_cache, p.num_blocks, p.block_size, p.num_kv_heads, dt))
        return -1;
    auto enc = tensor_map_encoder();
    if (!enc) return -1;
    CUresult rc;
    if (kGroup) {
        // decode queries as [sequences * heads, dims]; one box = 64 dims x Gp head rows
        cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.num_seqs * p.num_heads};
        cuuint64_t strides[1] = {kD * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)p.group_pad};
        cuuint32_t estr[2] = {1, 1};
        rc = enc(&mq, dt, 2, const_cast<void *>(p.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // queries as [tokens, heads, dims]; one box = 64 dims x Gp heads x QT tokens (128 rows)
        cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.num_heads, (cuuint64_t)p.num_query_tokens};
        cuuint64_t strides[2] = {kD * 2, (cuuint64_t)p.num_heads * kD * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)p.group_pad, (cuuint32_t)p.rows_q};
        cuuint32_t estr[3] = {1, 1, 1};
        rc = enc(&mq, dt, 3, const_cast<void *>(p.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (rc != CUDA_SUCCESS) return -1;
    const int64_t items = kGroup ? (int64_t)p.num_groups * p.num_kv_heads * p.shared_parts
                                 : (int64_t)p.num_seqs * p.num_kv_heads * p.qtiles;
    if (items == 0) return 0;
    const int grid = (int)(items < num_sms[dev] ? items : num_sms[dev]);
    PrefillParams q = p;
    const int64_t entries = (int64_t)p.num_seqs * p.qtiles;
    q.sorted_items = !kGroup && entries <= kSortMaxEntries && (items + grid - 1) / grid <= kMaxMyItems;
    // As the sharing-aware decode's shared pass it is launched as a programmatic
    // dependent (its set-up overlaps the 256-token scatter before it: 0.0711 -> 0.0695
    // ms a call); as a prefill, plainly: its CTAs, resident early, slowed the
    // chunk's 8192-token scatter by more than the sort they overlap.
    if (kGroup) return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, stream, mk, mv, mq, q);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(mk, mv, mq, q);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

bool prefill_tc_supported(const PrefillParams &p, int dtype) {
    return (dtype == PA_DTYPE_BF16 || dtype == PA_DTYPE_F16) && p.head_dim == kD && p.group >= 1 &&
           p.group <= 16 && p.block_size >= 8 && p.block_size <= kKT && p.num_blocks < INT32_MAX &&
           p.num_query_tokens < INT32_MAX && (int64_t)p.num_seqs * p.num_kv_heads * p.qtiles < INT32_MAX;
}

int launch_prefill_tc(const PrefillParams &p, int dtype, cudaStream_t stream) {
    if (!prefill_tc_supported(p, dtype)) return -2;
    if (dtype == PA_DTYPE_BF16)
        return launch_prefill_t<__nv_bfloat16, false>(p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, stream);
    return launch_prefill_t<__half, false>(p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, stream);
}

int launch_shared_prefix_tc(const PrefillParams &p, int dtype, cudaStream_t stream) {
    if (!prefill_tc_supported(p, dtype) || p.max_members < 1 || p.max_members * p.group_pad > kRows) return -2;
    if (dtype == PA_DTYPE_BF16)
        return launch_prefill_t<__nv_bfloat16, true>(p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, stream);
    return launch_prefill_t<__half, true>(p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, stream);
}

}  // namespace pa
