// Decode attention over an 8-bit (OCP FP8 E4M3) paged cache on the sm_100
// tensor cores, with the cache codes fed to the MMAs as they are stored.
//
// What is computed is the decode attention of "CS349E lecture 7:
// 01_paged_attention.py", demo 2, paper eq. 4 (block-wise scores through the
// block table, one softmax over the whole context, block-wise V accumulation)
// over the dequantised cache: element = decoded(code) * k_scale for K and
// decoded(code) * v_scale for V. The 8-bit cache itself is not on the pages;
// it halves the bytes each decode step reads, and the step is bound by them.
//
// The tensor cores multiply E4M3 operands natively (tcgen05 kind::f8f6f4, 32
// codes of the reduction per instruction), so the K and V boxes TMA lands in
// shared memory are MMA operands as they are: no expansion pass. The other
// operand of each product has to be E4M3 as well, and is carried as the sum of
// two codes per element:
//   S^T[128 tok x N] = K . [Qhi ; Qlo]^T    Q * 2^e = Qhi + Qlo, per head
//   O^T[128 d x N]   = V^T . [Phi ; Plo]^T  P * 256 = Phi + Plo, per token and head
// with head g's hi term in column g and its lo term in column GT + g (GT = the
// group size rounded up to 4, 8 or 16; N = max(16, 2 GT)). 2^e puts the largest
// magnitude of the query row in [128, 256): then a bf16 query is exactly
// Qhi + Qlo (8 significant bits = 4 + 4) at every element within 2^-9 of the
// row's largest, and an f16 query keeps 8 of its 11 bits. P in (0, 1] is
// scaled by 256 and split alike (about a bf16's precision); the row sums add
// the split values, so numerator and denominator use the same weights. k_scale
// and 2^-e fold into each head's score scale, v_scale into the output.
//
// A context that ends inside a block leaves the rest of that block's rows in
// the last tile. Their scores are masked; their V rows are overwritten with
// zeros before the P.V product, since a stale code may be NaN and 0 x NaN is
// NaN.
//
// CTA = a persistent worker, two per SM (one for groups above 8, whose softmax
// needs more registers): each tile's chain of S product, softmax barriers and
// P.V product is latency-bound, and a second independent chain on the SM hides
// much of it. 320 threads:
//   warp 0     TMA producer of the K boxes (128 codes x block_size tokens of one
//              kv head per physical block, 128-byte rows, 128-byte swizzle) into
//              a 2-stage ring.
//   warp 7     TMA producer of the V boxes into a 3-stage ring (a V stage is held
//              until the P.V product, after the softmax).
//   warp 8     query split: per item, the group's query rows -> hi/lo code rows
//              and per-head score scales, into a 2-slot ring.
//   warp 9     L2 prefetch of the next tile's blocks, ahead of the K loads (groups
//              up to 4; with larger groups the softmax, not the loads, sets the pace,
//              and the extra L2 traffic only costs).
//   warp 1     S MMA issuer (one thread) and tensor-memory owner.
//   warp 6     P.V MMA issuer (one thread).
//   warps 2-5  softmax and output (thread = token for S, = dim for O).
// Item order: decode_order.cuh. Every wait is bounded; on a timeout the kernel
// sets PA_DEVERR_WAIT, drains its copies and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "decode_order.cuh"
#include "fp8_encode.cuh"
#include "kernels.h"
#include "kernels_fp8.h"
#include "sm100.cuh"
#include "tma_maps.cuh"

namespace pa {
namespace {

using namespace sm100;
using decode_order::Item;

constexpr int kD = 128;
constexpr int kTile = 128;                        // tokens per MMA tile (M of the S product)
constexpr int kMaxG = 16;                         // query heads per kv head
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr int kQSlots = 2;
constexpr int kTileBytes = kTile * kD;            // 128 rows x 128 codes
constexpr int kOpBytes = 32 * 128;                // one hi/lo operand: up to 32 rows x 128 codes
constexpr int kThreads = 320;
constexpr int kPvWarp = 6, kVProdWarp = 7, kQWarp = 8, kPrefetchWarp = 9;
constexpr int kPrefetchTiles = 1;                 // L2 prefetch distance, in tiles, ahead of the K loads
constexpr int kMaxSeqs = 512;                     // sequences per launch (the host splits larger batches)
constexpr uint32_t kTmemCols = 128;               // S[2] and O[2], N columns each

// Resident CTAs per SM: two (96 registers a thread) where the softmax fits them.
__host__ __device__ constexpr int ctas_per_sm(int gt) { return gt <= 8 ? 2 : 1; }
// MMA N: hi and lo rows of GT heads, at least 16.
__host__ __device__ constexpr int n_cols(int gt) { return 2 * gt < 16 ? 16 : 2 * gt; }

// shared-memory carve-up (from a 1024-aligned base)
constexpr int kOffK = 0;                                      // [kKStages] K code tiles
constexpr int kOffV = kOffK + kKStages * kTileBytes;          // [kVStages] V code tiles
constexpr int kOffQ = kOffV + kVStages * kTileBytes;          // [kQSlots] query hi/lo rows
constexpr int kOffP = kOffQ + kQSlots * kOpBytes;             // [2] P hi/lo rows
constexpr int kOffQScale = kOffP + 2 * kOpBytes;              // float [kQSlots][kMaxG] score scales
constexpr int kOffRed = kOffQScale + kQSlots * kMaxG * 4;     // float [2][4][kMaxG] tile maxima
constexpr int kOffLRed = kOffRed + 2 * 4 * kMaxG * 4;         // float [2][4][kMaxG] row sums (by item parity)
constexpr int kOffBar = kOffLRed + 2 * 4 * kMaxG * 4;
// mbarrier slots, in order; kNumBars counts them
constexpr int kBarKFull = 0;                                  // [kKStages]
constexpr int kBarKEmpty = kBarKFull + kKStages;              // [kKStages]
constexpr int kBarVFull = kBarKEmpty + kKStages;              // [kVStages]
constexpr int kBarVEmpty = kBarVFull + kVStages;              // [kVStages]
constexpr int kBarQFull = kBarVEmpty + kVStages;              // [kQSlots]
constexpr int kBarQEmpty = kBarQFull + kQSlots;               // [kQSlots]
constexpr int kBarSFull = kBarQEmpty + kQSlots;               // [2]
constexpr int kBarSFree = kBarSFull + 2;                      // [2]
constexpr int kBarPFull = kBarSFree + 2;                      // [2]
constexpr int kBarOFull = kBarPFull + 2;                      // [2]
constexpr int kBarOFree = kBarOFull + 2;                      // [2]
constexpr int kBarRed = kBarOFree + 2;                        // [2]
constexpr int kBarFin = kBarRed + 2;                          // [1]
constexpr int kNumBars = kBarFin + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;              // tmem base, abort flag, 2 item counts, loads issued
constexpr int kOffPrefix = (kOffMisc + 32 + 15) & ~15;        // int [kMaxSeqs + 1]; later the item table
constexpr int kOffOrder = kOffPrefix + (kMaxSeqs + 1) * 4;    // int [kMaxSeqs]
constexpr int kOffCtx = kOffOrder + kMaxSeqs * 4;             // int [kMaxSeqs] clamped context lengths
constexpr int kOffPs = kOffCtx + kMaxSeqs * 4;                // int [kMaxSeqs] first token of this pass
constexpr int kSmemUsed = kOffPs + kMaxSeqs * 4;
static_assert(kSmemUsed - kOffPrefix >= decode_order::kTableItems * 16, "item table fits the ordering arrays");
constexpr int kSmemBytes = kSmemUsed + 1024;                  // + alignment slack
static_assert(kSmemBytes <= 115712, "shared memory budget: two CTAs per SM");
static_assert(kOffV % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kOpBytes % 1024 == 0,
              "128-byte-swizzled tiles need 1024-byte alignment");
static_assert(2 * kOpBytes >= kMaxSeqs, "the P rows serve as the ordering scratch");

struct Bars {
    uint64_t *k_full, *k_empty;    // [kKStages]
    uint64_t *v_full, *v_empty;    // [kVStages]
    uint64_t *q_full, *q_empty;    // [kQSlots]
    uint64_t *s_full, *s_free;     // [2]
    uint64_t *p_full, *o_full;     // [2]
    uint64_t *o_free, *red;        // [2]
    uint64_t *fin;                 // [1]
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- E4M3 pairs ---------------------------------------------------------------
// Two floats -> two codes, nearest with ties to even, saturating at +-448:
// `a` in the low byte, `b` in the high byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
    return h;
}
// The two codes of the low 16 bits -> their values (low byte -> .x); exact.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t c) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
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

// Byte offset of element (row n, column c) in a 128-byte-swizzled K-major tile of
// 8-bit elements: 128-byte rows, 16-byte chunks permuted within 8-row groups.
__device__ __forceinline__ int sw128_byte(int n, int c) { return n * 128 + ((((c >> 4) ^ n) & 7) << 4) + (c & 15); }

// ---- tcgen05 (kind::f8f6f4) ------------------------------------------------------
// Instruction descriptor: A and B E4M3, fp32 accumulation; a_mn: A is MN-major.
__host__ __device__ constexpr uint32_t instr_desc_e4m3(int M, int N, bool a_mn) {
    return (1u << 4)                                 // D format: f32
           | (0u << 7) | (0u << 10)                  // A, B format: E4M3
           | ((a_mn ? 1u : 0u) << 15)                // A major
           | ((uint32_t)(N >> 3) << 17)              // N / 8
           | ((uint32_t)(M >> 4) << 24);             // M / 16
}
// D (tmem) [+]= A (smem desc) * B (smem desc), 32 codes of the reduction; one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, "
        "p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x NC consecutive fp32 columns (NC = 8, 16 or 32), load and wait.
template <int NC> __device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float *v);
template <> __device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <> __device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, float *v) { tmem_ld16(taddr, v); }
template <> __device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, float *v) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Four 16-bit values (one 8-byte load) -> floats.
template <typename T> __device__ __forceinline__ void unpack4(uint2 u, float *x);
template <> __device__ __forceinline__ void unpack4<__nv_bfloat16>(uint2 u, float *x) {
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
template <> __device__ __forceinline__ void unpack4<__half>(uint2 u, float *x) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    x[0] = a.x;
    x[1] = a.y;
    x[2] = b.x;
    x[3] = b.y;
}

// Decode with append (kApp): the step's own token of the item's sequence (position
// ctx - 1), for the item's kv head. At the start of the sequence's last item, before
// any of its tiles is loaded, the producer warps read its slot, encode their row (K
// with k_scale by the K producer, V with v_scale by the V producer: lanes 0-7 each
// 16 elements, the scatter's encoding) and store the codes, so the item's TMA loads
// read them. (Storing just before the last tile's loads instead, with a check on
// every tile, measured slower: long context 0.2368 against 0.2346 ms a step.) `e`
// is the block-table entry of the token's block. The slot must be that of position
// ctx - 1 (a different one sets PA_DEVERR_SLOT and is not written; -1 writes
// nothing).
template <typename T>
__device__ __forceinline__ uint4 append_codes(const DecodeParams &p, const Item &I, bool is_v, float scale,
                                              int lane) {
    if (lane >= kD / 16) return make_uint4(0, 0, 0, 0);
    const T *src = static_cast<const T *>(is_v ? p.app_v : p.app_k) +
                   ((int64_t)I.b * p.num_kv_heads + I.kvh) * kD + lane * 16;
    float x[16];
    fp8::load16(src, x);
    return fp8::encode16(x, scale);
}

__device__ __forceinline__ void append_store(const DecodeParams &p, const Item &I, int slot, int e, uint4 codes,
                                             bool is_v, int lane) {
    const int pos = I.t1 - 1;
    const int64_t expect = (int64_t)e * p.block_size + (pos & (p.block_size - 1));
    if (e < 0 || e >= p.num_blocks || (int64_t)slot != expect) {
        if (!is_v && lane == 0) raise_error(p.err, PA_DEVERR_SLOT);
        return;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(
                     const_cast<void *>(is_v ? p.value_cache : p.key_cache)) +
                     ((int64_t)slot * p.num_kv_heads + I.kvh) * kD);
    if (lane < kD / 16) dst[lane] = codes;
    asm volatile("fence.proxy.async.global;" ::: "memory");   // the tile's TMA loads read them
}

template <typename T, int GT, bool kApp>
__global__ __launch_bounds__(kThreads, ctas_per_sm(GT)) void decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                 const __grid_constant__ CUtensorMap tm_v,
                                                                 const DecodeParams p, const float v_scale,
                                                                 const float k_scale) {
    constexpr int NT = n_cols(GT);
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sK = smem + kOffK;
    unsigned char *sV = smem + kOffV;
    unsigned char *sQ = smem + kOffQ;
    unsigned char *sP = smem + kOffP;
    float *qscale = reinterpret_cast<float *>(smem + kOffQScale);
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    float *lred = reinterpret_cast<float *>(smem + kOffLRed);
    uint64_t *bar_base = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    volatile uint32_t *loads_issued = reinterpret_cast<volatile uint32_t *>(smem + kOffMisc + 16);
    int *prefix = reinterpret_cast<int *>(smem + kOffPrefix);

    Bars bars;
    bars.k_full = bar_base + kBarKFull;
    bars.k_empty = bar_base + kBarKEmpty;
    bars.v_full = bar_base + kBarVFull;
    bars.v_empty = bar_base + kBarVEmpty;
    bars.q_full = bar_base + kBarQFull;
    bars.q_empty = bar_base + kBarQEmpty;
    bars.s_full = bar_base + kBarSFull;
    bars.s_free = bar_base + kBarSFree;
    bars.p_full = bar_base + kBarPFull;
    bars.o_full = bar_base + kBarOFull;
    bars.o_free = bar_base + kBarOFree;
    bars.red = bar_base + kBarRed;
    bars.fin = bar_base + kBarFin;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group;

    if (tid == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);      // the S MMAs' commit
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_empty[s], 1);      // the P.V MMAs' commit
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(&bars.q_full[s], 1);
            mbar_init(&bars.q_empty[s], 1 + 4);  // the item's last S commit + the softmax warps (scales read)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], 4);
            mbar_init(&bars.p_full[i], 4);
            mbar_init(&bars.o_full[i], 1);
            mbar_init(&bars.o_free[i], 4);
            mbar_init(&bars.red[i], 4);          // one arrival per softmax warp
        }
        mbar_init(bars.fin, 4);
        *abort_flag = 0;
        *loads_issued = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // Programmatic dependent launch: the set-up above and the item order below,
    // which reads only the call's lengths, overlap the preceding kernel (the previous
    // call's merge, or the 8-bit scatter, which writes cache rows); everything after
    // the wait may touch what that kernel reads or writes.
    asm volatile("griddepcontrol.launch_dependents;");

    int *order = reinterpret_cast<int *>(smem + kOffOrder);
    int *counts = reinterpret_cast<int *>(smem + kOffMisc + 8);   // [0] = n4, [1] = list length
    const decode_order::SeqCache cache{reinterpret_cast<int *>(smem + kOffCtx), reinterpret_cast<int *>(smem + kOffPs)};
    decode_order::build(p, prefix, order, counts, sP, cache);            // P rows as scratch until the first tile
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n4 = counts[0];
    const int total_items = (counts[0] + counts[1]) * p.num_kv_heads;
    // this CTA's item descriptors, computed once and kept over the ordering arrays
    int4 *items = reinterpret_cast<int4 *>(smem + kOffPrefix);
    decode_order::build_item_table<(decode_order::kTableItems + kThreads - 1) / kThreads>(p, prefix, order, n4, cache,
                                                                                         total_items, items);
    const int nmy = decode_order::cta_items(total_items);
    // P rows past 2 GT stay zero (their columns are never read, but the MMA
    // multiplies them)
    for (int i = tid; i < 2 * kOpBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(sP)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0 || warp == kVProdWarp) {
        // ------------------------------------------------------------ producers
        const bool is_v = warp == kVProdWarp;
        const int nstages = is_v ? kVStages : kKStages;
        uint64_t *fullb = is_v ? bars.v_full : bars.k_full;
        uint64_t *emptyb = is_v ? bars.v_empty : bars.k_empty;
        unsigned char *ring = is_v ? sV : sK;
        const CUtensorMap *tm = is_v ? &tm_v : &tm_k;
        const int nbt = kTile / p.block_size;       // physical blocks per tile
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const decode_order::ItemTable tb = decode_order::load_item_table(p, I, lane);
            // decode with append: the new token's slot and codes, used at the item's
            // last tile (an empty context takes only -1)
            if constexpr (kApp) {
                if (I.last) {
                    const int app_slot = p.app_slots[I.b];
                    if (app_slot != -1 && I.ntiles > 0) {
                        const uint4 app_codes = append_codes<T>(p, I, is_v, is_v ? v_scale : k_scale, lane);
                        // the token's block among the item's blocks, from the table in registers
                        const int jb = ((I.t1 - 1) >> p.log2_block_size) - (I.t0 >> p.log2_block_size);
                        bool lv;
                        const int e = decode_order::tile_entry(tb, jb / nbt, nbt, lane, &lv);
                        append_store(p, I, app_slot, __shfl_sync(0xffffffffu, e, jb % nbt), app_codes, is_v, lane);
                        __syncwarp();
                    }
                    if (app_slot != -1 && I.ntiles == 0 && I.t1 == 0 && !is_v && lane == 0)
                        raise_error(p.err, PA_DEVERR_SLOT);
                }
            }
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int stage = it % nstages;
                const uint32_t ph = (it / nstages) & 1;
                bool live;
                const int e = decode_order::tile_entry(tb, tile, nbt, lane, &live);
                int phys = (int)p.num_blocks;           // out of range: TMA fills zeros
                if (live) {
                    if (e >= 0 && e < p.num_blocks) phys = e;
                    else if (!is_v) raise_error(p.err, PA_DEVERR_BLOCK_ID);
                }
                int w = 1;
                if (lane == 0) w = mbar_wait(&emptyb[stage], ph ^ 1) ? 1 : 0;
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w || *abort_flag) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&fullb[stage], kTileBytes);
                __syncwarp();
                if (lane < nbt)
                    tma_load_4d(ring + stage * kTileBytes + lane * p.block_size * 128, tm, &fullb[stage], 0, I.kvh, 0,
                                phys);
                if (lane == 0 && !is_v) *loads_issued = it + 1;
            }
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
        // drain: every issued stage's copies must have landed before the CTA exits
        if (lane == 0) {
            const uint32_t first = it > (uint32_t)nstages ? it - nstages : 0;
            for (uint32_t j = first; j < it; ++j) mbar_wait(&fullb[j % nstages], (j / nstages) & 1);
        }
    } else if (warp == kQWarp) {
        // ------------------------------------------------------------ query split
        // Lane l holds dims 4l .. 4l+3 of every row of the group. Rows past the
        // group (and past 2 GT) are written as zeros, with a zero score scale.
        const T *q = reinterpret_cast<const T *>(p.q);
        uint32_t qi = 0;
        bool ok = true;
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            if (I.ntiles == 0) continue;
            const int slot = qi % kQSlots;
            if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                !warp_wait(&bars.q_empty[slot], ((qi / kQSlots) & 1) ^ 1)) {
                ok = false;
                break;
            }
            const T *qrow = q + ((int64_t)I.b * p.num_heads + (int64_t)I.kvh * G) * kD + 4 * lane;
            uint2 raw[GT];                               // all loads in flight before the first use
#pragma unroll
            for (int g = 0; g < GT; ++g)
                raw[g] = g < G ? __ldg(reinterpret_cast<const uint2 *>(qrow + g * kD)) : make_uint2(0, 0);
            unsigned char *dst = sQ + slot * kOpBytes;
#pragma unroll
            for (int g = 0; g < GT; ++g) {
                float x[4];
                unpack4<T>(raw[g], x);
                const float amax = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
                // amax = 1.f * 2^(E - 127): scale by 2^(134 - E), so amax lands in [128, 256)
                const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF);
                int e2 = E == 0 ? 126 : 134 - E;
                e2 = e2 < -126 ? -126 : (e2 > 126 ? 126 : e2);
                const float up = __uint_as_float((uint32_t)(e2 + 127) << 23);     // 2^e2
                const float down = __uint_as_float((uint32_t)(127 - e2) << 23);   // 2^-e2
                float y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = x[i] * up;
                const uint32_t h01 = e4m3x2(y[0], y[1]), h23 = e4m3x2(y[2], y[3]);
                const float2 f01 = e4m3x2_value(h01), f23 = e4m3x2_value(h23);
                const uint32_t l01 = e4m3x2(y[0] - f01.x, y[1] - f01.y), l23 = e4m3x2(y[2] - f23.x, y[3] - f23.y);
                *reinterpret_cast<uint32_t *>(dst + sw128_byte(g, 4 * lane)) = h01 | (h23 << 16);
                *reinterpret_cast<uint32_t *>(dst + sw128_byte(GT + g, 4 * lane)) = l01 | (l23 << 16);
                if (lane == 0) qscale[slot * kMaxG + g] = g < G ? p.scale_log2 * down : 0.f;
            }
#pragma unroll
            for (int n = 2 * GT; n < NT; ++n) *reinterpret_cast<uint32_t *>(dst + sw128_byte(n, 4 * lane)) = 0u;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.q_full[slot]);
            ++qi;
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = instr_desc_e4m3(kTile, NT, false);
            const uint32_t sK0 = smem_addr(sK), sQ0 = smem_addr(sQ);
            uint32_t it = 0, qi = 0;
            bool ok = true;
            for (int k = 0; k < nmy && ok; ++k) {
                const Item I = decode_order::unpack_item(items[k]);
                if (I.ntiles == 0) continue;
                const int slot = qi % kQSlots;
                if (*abort_flag || !mbar_wait(&bars.q_full[slot], (qi / kQSlots) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t qbase = sQ0 + slot * kOpBytes;
                for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                    const int stage = it % kKStages, buf = it & 1;
                    if (*abort_flag || !mbar_wait(&bars.k_full[stage], (it / kKStages) & 1) ||
                        !mbar_wait(&bars.s_free[buf], ((it >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kbase = sK0 + stage * kTileBytes;
                    const uint32_t dcol = tmem + buf * NT;
#pragma unroll
                    for (int kk = 0; kk < kD / 32; ++kk) {
                        const uint64_t a = smem_desc(kbase + kk * 32, 16, 1024);
                        const uint64_t b = smem_desc(qbase + kk * 32, 16, 1024);
                        mma_e4m3(dcol, a, b, idesc_s, kk > 0);
                    }
                    mma_commit(&bars.s_full[buf]);
                    mma_commit(&bars.k_empty[stage]);
                }
                if (!ok) break;
                mma_commit(&bars.q_empty[slot]);
                ++qi;
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, PA_DEVERR_WAIT);
            }
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ P.V MMA issuer
        if (lane == 0) {
            const uint32_t idesc_o = instr_desc_e4m3(kD, NT, true);
            const uint32_t sV0 = smem_addr(sV), sP0 = smem_addr(sP);
            uint32_t it = 0;
            bool ok = true;
            for (int k = 0; k < nmy && ok; ++k) {
                const Item I = decode_order::unpack_item(items[k]);
                for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                    const int buf = it & 1, stage = it % kVStages;
                    const uint32_t bph = (it >> 1) & 1;
                    if (*abort_flag || !mbar_wait(&bars.p_full[buf], bph) || !mbar_wait(&bars.o_free[buf], bph ^ 1) ||
                        !mbar_wait(&bars.v_full[stage], (it / kVStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t vbase = sV0 + stage * kTileBytes;
                    const uint32_t pbase = sP0 + buf * kOpBytes;
                    const uint32_t dcol = tmem + 2 * NT + buf * NT;
                    // A = V^T: 128 dims (one 128-byte swizzle atom) x 32 tokens per
                    // instruction, MN-major, 8-token groups 1024 bytes apart
#pragma unroll
                    for (int kk = 0; kk < kTile / 32; ++kk) {
                        const uint64_t a = smem_desc(vbase + kk * 4096, kTileBytes, 1024);
                        const uint64_t b = smem_desc(pbase + kk * 32, 16, 1024);
                        mma_e4m3(dcol, a, b, idesc_o, kk > 0);
                    }
                    mma_commit(&bars.o_full[buf]);
                    mma_commit(&bars.v_empty[stage]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, PA_DEVERR_WAIT);
            }
        }
        __syncwarp();
    } else if (warp == kPrefetchWarp) {
        // ------------------------------------------------------------ L2 prefetch
        // Walks the same tiles as the K producer, at most kPrefetchTiles ahead of
        // its loads, pulling each tile's K and V blocks into L2. Prefetches are
        // hints: if this warp falls behind or gives up, only speed changes.
        const int nbt = kTile / p.block_size;
        uint32_t n = 0;
        bool go = GT <= 4;
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
                    tma_prefetch_4d(&tm_v, 0, I.kvh, 0, e);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax / output
        const int q4 = warp & 3;                       // tensor-memory lane quadrant
        const int row = q4 * 32 + lane;                // token (S) or dim (O) of this thread
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        T *out = reinterpret_cast<T *>(p.out);
        uint32_t it = 0, nfin = 0, qi = 0;
        bool ok = true;
        float m_run[GT], l_part[GT], o_acc[GT], alpha_prev[GT], qs[GT];
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const int64_t head0 = (int64_t)I.b * p.num_heads + (int64_t)I.kvh * G;
            if (I.ntiles == 0) {
#pragma unroll
                for (int g = 0; g < GT; ++g)
                    if (g < G) out[(head0 + g) * kD + row] = Elem<T>::from_f(0.f);
                continue;
            }
            // the item's per-head score scales
            const int slot = qi % kQSlots;
            if (__any_sync(0xffffffffu, *abort_flag != 0) || !warp_wait(&bars.q_full[slot], (qi / kQSlots) & 1)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int g = 0; g < GT; ++g) qs[g] = qscale[slot * kMaxG + g];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.q_empty[slot]);
            ++qi;
#pragma unroll
            for (int g = 0; g < GT; ++g) {
                m_run[g] = -INFINITY;
                l_part[g] = 0.f;
                o_acc[g] = 0.f;
                alpha_prev[g] = 0.f;
            }
            auto accumulate = [&](uint32_t j) -> bool {
                const int buf = j & 1;
                if (!warp_wait(&bars.o_full[buf], (j >> 1) & 1)) return false;
                tc_fence_after();
                float o[2 * GT];
                tmem_ld_cols<2 * GT>(tmem + lane_off + 2 * NT + buf * NT, o);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.o_free[buf]);
#pragma unroll
                for (int g = 0; g < GT; ++g) o_acc[g] = fmaf(o_acc[g], alpha_prev[g], o[g] + o[GT + g]);
                return true;
            };
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int buf = it & 1;
                if (__any_sync(0xffffffffu, *abort_flag != 0) || !warp_wait(&bars.s_full[buf], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[2 * GT];
                tmem_ld_cols<2 * GT>(tmem + lane_off + buf * NT, s);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.s_free[buf]);

                const int valid_rows = I.t1 - (I.t0 + tile * kTile);
                const bool valid = row < valid_rows;
                float *rd = red + (it & 1) * 4 * kMaxG;
                float sv[GT];
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    sv[g] = valid ? (s[g] + s[GT + g]) * qs[g] : -INFINITY;
                    const float mx = warp_max(sv[g]);
                    if (lane == 0) rd[q4 * kMaxG + g] = mx;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.red[it & 1]);
                if (!warp_wait(&bars.red[it & 1], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                if (valid_rows < kTile) {
                    // last tile of a context ending mid-tile: zero the V rows past it
                    const int vs = it % kVStages;
                    if (!warp_wait(&bars.v_full[vs], (it / kVStages) & 1)) {
                        ok = false;
                        break;
                    }
                    if (!valid) {
                        uint4 *vrow = reinterpret_cast<uint4 *>(sV + vs * kTileBytes + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) vrow[c ^ (row & 7)] = make_uint4(0, 0, 0, 0);
                    }
                }
                float alpha[GT];
                unsigned char *pb = sP + buf * kOpBytes;
#pragma unroll
                const float2 neg1 = make_float2(-1.f, -1.f);
                for (int g = 0; g < GT; g += 2) {
                    float mn[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = g + e;
                        const float tmax = fmaxf(fmaxf(rd[h], rd[kMaxG + h]), fmaxf(rd[2 * kMaxG + h], rd[3 * kMaxG + h]));
                        const float m_new = fmaxf(m_run[h], tmax);
                        alpha[h] = fast_exp2(m_run[h] - m_new);
                        m_run[h] = m_new;
                        mn[e] = m_new;
                    }
                    // the pair of heads in paired fp32 instructions where the registers
                    // allow (groups up to 4; at 8 the pairs spilled: 0.281 vs 0.234 ms)
                    float2 x, hf, lf;
                    uint32_t hi, lo;
                    if constexpr (GT <= 4) {
                        const float2 dl = ffma2(make_float2(mn[0], mn[1]), neg1, make_float2(sv[g], sv[g + 1]));
                        x = ffma2(make_float2(fast_exp2(dl.x), fast_exp2(dl.y)), make_float2(256.f, 256.f),
                                  make_float2(0.f, 0.f));
                        if (!valid) x = make_float2(0.f, 0.f);
                        hi = e4m3x2(x.x, x.y);
                        hf = e4m3x2_value(hi);
                        const float2 res = ffma2(hf, neg1, x);
                        lo = e4m3x2(res.x, res.y);
                        lf = e4m3x2_value(lo);
                        const float2 l2 = ffma2(make_float2(l_part[g], l_part[g + 1]),
                                                make_float2(alpha[g], alpha[g + 1]), fadd2(hf, lf));
                        l_part[g] = l2.x;
                        l_part[g + 1] = l2.y;
                    } else {
                        x.x = valid ? fast_exp2(sv[g] - mn[0]) * 256.f : 0.f;
                        x.y = valid ? fast_exp2(sv[g + 1] - mn[1]) * 256.f : 0.f;
                        hi = e4m3x2(x.x, x.y);
                        hf = e4m3x2_value(hi);
                        lo = e4m3x2(x.x - hf.x, x.y - hf.y);
                        lf = e4m3x2_value(lo);
                        l_part[g] = fmaf(l_part[g], alpha[g], hf.x + lf.x);
                        l_part[g + 1] = fmaf(l_part[g + 1], alpha[g + 1], hf.y + lf.y);
                    }
                    pb[sw128_byte(g, row)] = (unsigned char)hi;
                    pb[sw128_byte(g + 1, row)] = (unsigned char)(hi >> 8);
                    pb[sw128_byte(GT + g, row)] = (unsigned char)lo;
                    pb[sw128_byte(GT + g + 1, row)] = (unsigned char)(lo >> 8);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full[buf]);
                if (tile > 0 && !accumulate(it - 1)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int g = 0; g < GT; ++g) alpha_prev[g] = alpha[g];
            }
            if (!ok) break;
            if (!accumulate(it - 1)) {
                ok = false;
                break;
            }
            // ---- finalize the item: sum of the token lanes' partial l per head
            // (lred is double-buffered by item parity: one barrier per item)
            float *lr = lred + (nfin & 1) * 4 * kMaxG;
#pragma unroll
            for (int g = 0; g < GT; ++g) {
                const float ls = warp_sum(l_part[g]);
                if (lane == 0) lr[q4 * kMaxG + g] = ls;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.fin);
            if (!warp_wait(bars.fin, nfin++ & 1)) {
                ok = false;
                break;
            }
            float l_tot[GT];
#pragma unroll
            for (int g = 0; g < GT; ++g) l_tot[g] = lr[g] + lr[kMaxG + g] + lr[2 * kMaxG + g] + lr[3 * kMaxG + g];
            // o_acc and l_tot both carry the factor 256 of the split P
            if (I.direct) {
#pragma unroll
                for (int g = 0; g < GT; ++g)
                    if (g < G) out[(head0 + g) * kD + row] = Elem<T>::from_f(o_acc[g] * v_scale / l_tot[g]);
            } else {
                const int P = p.max_partitions;
                const float vs256 = v_scale * (1.f / 256.f);
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    if (g < G) {
                        const int64_t r = (head0 + g) * P + I.slot;
                        p.ws_o[r * kD + row] = o_acc[g] * vs256;
                        if (row == 0) {
                            p.ws_ml[2 * r] = m_run[g];
                            p.ws_ml[2 * r + 1] = l_tot[g] * (1.f / 256.f);
                        }
                    }
                }
            }
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

// ---- host side -----------------------------------------------------------------

// 4-D map over a [num_blocks, block_size, num_kv_heads, 128] 8-bit cache, listed
// innermost first as (dim, kv head, token in block, block). One box = 128 codes x
// 1 kv head x block_size tokens: block_size rows of 128 bytes in shared memory,
// 128-byte swizzled. Coordinates past num_blocks read as zeros.
bool make_cache_map_u8(CUtensorMap *m, const void *base, const DecodeParams &p) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t D = kD;
    cuuint64_t dims[4] = {D, (cuuint64_t)p.num_kv_heads, (cuuint64_t)p.block_size, (cuuint64_t)p.num_blocks};
    cuuint64_t strides[3] = {D, (cuuint64_t)p.num_kv_heads * D, (cuuint64_t)p.block_size * p.num_kv_heads * D};
    cuuint32_t box[4] = {(cuuint32_t)kD, 1, (cuuint32_t)p.block_size, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int GT, bool kApp>
int launch_t(const DecodeParams &p, float v_scale, float k_scale, cudaStream_t stream) {
    auto kern = decode_fp8_kernel<T, GT, kApp>;
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
    CUtensorMap mk, mv;
    if (!make_cache_map_u8(&mk, p.key_cache, p) || !make_cache_map_u8(&mv, p.value_cache, p)) return -1;
    const int64_t max_items = (int64_t)p.num_seqs * p.num_kv_heads * p.max_partitions;
    const int64_t slots = (int64_t)ctas_per_sm(GT) * num_sms[dev];
    const int grid = (int)(max_items < slots ? max_items : slots);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, stream, mk, mv, p, v_scale, k_scale);
}

template <typename T, bool kApp>
int launch_g(const DecodeParams &p, float v_scale, float k_scale, cudaStream_t stream) {
    if (p.group <= 4) return launch_t<T, 4, kApp>(p, v_scale, k_scale, stream);
    if (p.group <= 8) return launch_t<T, 8, kApp>(p, v_scale, k_scale, stream);
    return launch_t<T, 16, kApp>(p, v_scale, k_scale, stream);
}

template <typename T>
int launch_a(const DecodeParams &p, float v_scale, float k_scale, cudaStream_t stream) {
    return p.app_slots ? launch_g<T, true>(p, v_scale, k_scale, stream) : launch_g<T, false>(p, v_scale, k_scale, stream);
}

}  // namespace

bool decode_fp8_supported(const DecodeParams &p, int dtype) {
    return (dtype == PA_DTYPE_BF16 || dtype == PA_DTYPE_F16) && p.head_dim == kD && p.group >= 1 &&
           p.group <= kMaxG && p.block_size >= 8 && p.block_size <= kTile && p.partition_size % kTile == 0 &&
           p.num_blocks < INT32_MAX && (int64_t)p.num_seqs * p.num_heads < INT32_MAX;
}

// Batches above kMaxSeqs sequences run as independent launches of up to kMaxSeqs.
int launch_decode_fp8(const DecodeParams &p, float v_scale, float k_scale, int dtype, cudaStream_t stream) {
    if (!decode_fp8_supported(p, dtype)) return -2;
    // sequences per launch: at most kMaxSeqs, and few enough that no CTA gets more
    // than the item table holds (items <= num_seqs * kv heads * partitions)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    const int64_t per_seq = (int64_t)p.num_kv_heads * p.max_partitions;
    const int cps = p.group <= 8 ? ctas_per_sm(8) : ctas_per_sm(16);
    const int64_t by_items = (int64_t)decode_order::kTableItems * cps * sms / (per_seq > 0 ? per_seq : 1);
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
        if (p.ws_ml) {
            c.ws_ml = p.ws_ml + rows * p.max_partitions * 2;
            c.ws_o = p.ws_o + rows * p.max_partitions * kD;
        }
        if (p.app_slots) {
            c.app_slots = p.app_slots + b0;
            c.app_k = static_cast<const char *>(p.app_k) + (int64_t)b0 * p.num_kv_heads * kD * 2;
            c.app_v = static_cast<const char *>(p.app_v) + (int64_t)b0 * p.num_kv_heads * kD * 2;
        }
        const int rc = dtype == PA_DTYPE_BF16 ? launch_a<__nv_bfloat16>(c, v_scale, k_scale, stream)
                                              : launch_a<__half>(c, v_scale, k_scale, stream);
        if (rc != 0) return rc;
    }
    return 0;
}

}  // namespace pa
