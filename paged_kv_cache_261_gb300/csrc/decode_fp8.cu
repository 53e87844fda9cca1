// Decode attention over an 8-bit (OCP FP8 E4M3) paged cache on the sm_100
// tensor cores.
//
// What is computed is the decode attention of "CS349E lecture 7:
// 01_paged_attention.py", demo 2, paper eq. 4 (block-wise scores through the
// block table, one softmax over the whole context, block-wise V accumulation)
// over the dequantised cache: element = decoded(code) * k_scale for K and
// decoded(code) * v_scale for V. The 8-bit cache itself is not on the pages;
// it halves the bytes each decode step reads, and the step is bound by them.
//
// Every E4M3 value is exact in bf16 and in f16, so the kernel expands codes to
// the query's 16-bit type without rounding and runs the same two MMAs per
// 128-token tile as the 16-bit kernel: S^T[128 tok x 16] = K . Q^T and
// O^T[128 d x 16] = V^T . P^T (tcgen05 kind::f16, M=128, N=16, K=128). The
// expanded K tile goes to tensor memory (thread = token = lane, the A operand
// of the S MMA is read from there; two buffers), the expanded V tile to shared
// memory (two buffers). k_scale is folded into the score scale and v_scale into
// the output.
//
// CTA = one persistent worker per SM; 512 threads (384 for groups above 8):
//   warp 0     TMA producer of the K boxes (128 codes x block_size tokens of one
//              kv head per physical block, 128-byte rows, 128-byte swizzle)
//              and the group's 16 query rows, into a 4-stage ring.
//   last warp  TMA producer of the V boxes into the same stages.
//   warp 1     S MMA issuer (one thread) and tensor-memory owner.
//   warp 6     P.V MMA issuer (one thread). S and P.V each have their own
//              issuing thread: a single issuer spent most of each tile issuing.
//   warps 7-14 converters (thread = token row): warps 7-10 expand each tile's
//              K codes into tensor memory, warps 11-14 its V codes into a
//              128-byte-swizzled shared-memory tile. V rows of tokens past the
//              partition end are written as zeros (their slots may hold
//              anything). With more than 8 query heads per kv head the softmax
//              needs more registers, and warps 7-10 alone expand tile i+1's K,
//              then tile i's V.
//   warps 2-5  softmax and output, as in the 16-bit kernel.
// Item order: decode_order.cuh. Every wait is bounded; on a timeout the kernel
// sets PA_DEVERR_WAIT, drains its copies and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "decode_order.cuh"
#include "kernels.h"
#include "kernels_fp8.h"
#include "sm100.cuh"
#include "tma_maps.cuh"

namespace pa {
namespace {

using namespace sm100;
using decode_order::get_item;
using decode_order::Item;

constexpr int kD = 128;
constexpr int kTile = 128;                        // tokens per MMA tile (M)
constexpr int kN = 16;                            // MMA N: query heads of a group, padded
constexpr int kStages = 4;                        // 8-bit ring
constexpr int kTile8Bytes = kTile * kD;           // 128 rows x 128 codes
constexpr int kQBytes = 2 * kN * 128;             // 16 rows x 128 dims (16-bit)
constexpr int kStageBytes = 2 * kTile8Bytes + kQBytes;
constexpr int kChunkBytes = kTile * 128;          // 128 rows x 64 dims x 2 B
constexpr int kKVBytes = 2 * kChunkBytes;         // one 16-bit tile, both 64-dim halves
constexpr int kPBytes = 2 * kN * 128;             // P^T: 16 rows x 128 tokens
constexpr int kConvWarp0 = 7;                     // first converter warp
// Converter warps: 8 (one warpgroup for K, one for V) where the softmax warps'
// registers allow it (up to 8 query heads per kv head), else 4 doing both.
__host__ __device__ constexpr int conv_warps(int gt) { return gt <= 8 ? 8 : 4; }
__host__ __device__ constexpr int threads_for(int gt) { return (kConvWarp0 + conv_warps(gt) + 1) * 32; }
constexpr int kPvWarp = 6;                        // issues the P.V MMAs
constexpr int kMaxSeqs = 512;                     // sequences per launch (the host splits larger batches)
constexpr uint32_t kTmemCols = 256;               // S[2] x 16 + O[2] x 16 + K[2] x 64 columns
constexpr uint32_t kColK = 64;                    // first column of the expanded K tiles
constexpr uint32_t kKCols = kD / 2;               // one K tile: 128 dims of 16 bits per lane

// shared-memory carve-up (from a 1024-aligned base)
constexpr int kOff8 = 0;                                      // [kStages] x {K codes, V codes, Q}
constexpr int kOffVb = kOff8 + kStages * kStageBytes;         // two 16-bit V tiles
constexpr int kOffP = kOffVb + 2 * kKVBytes;
constexpr int kOffRed = kOffP + 2 * kPBytes;                  // float [2][4][16]
constexpr int kOffLRed = kOffRed + 2 * 4 * kN * 4;            // float [2][4][16] (by item parity)
constexpr int kOffBar = kOffLRed + 2 * 4 * kN * 4;
// mbarrier slots, in order; kNumBars counts them
constexpr int kBarFull = 0;                                   // [kStages]
constexpr int kBarEmpty = kBarFull + kStages;                 // [kStages]
constexpr int kBarSFull = kBarEmpty + kStages;                // [2]
constexpr int kBarSFree = kBarSFull + 2;                      // [2]
constexpr int kBarPFull = kBarSFree + 2;                      // [2]
constexpr int kBarOFull = kBarPFull + 2;                      // [2]
constexpr int kBarOFree = kBarOFull + 2;                      // [2]
constexpr int kBarRed = kBarOFree + 2;                        // [2]
constexpr int kBarFin = kBarRed + 2;                          // [1]
constexpr int kBarKbFull = kBarFin + 1;                       // [2]
constexpr int kBarKbFree = kBarKbFull + 2;                    // [2]
constexpr int kBarVbFull = kBarKbFree + 2;                    // [2]
constexpr int kBarVbFree = kBarVbFull + 2;                    // [2]
constexpr int kBarFullV = kBarVbFree + 2;                     // [kStages]
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
static_assert(kStageBytes % 1024 == 0 && kOffVb % 1024 == 0 && kOffP % 1024 == 0,
              "128-byte-swizzled tiles need 1024-byte alignment");

struct Bars {
    uint64_t *full, *empty;        // [kStages] 8-bit ring
    uint64_t *s_full, *s_free;     // [2]
    uint64_t *p_full, *o_full;     // [2]
    uint64_t *o_free, *red;        // [2]
    uint64_t *fin;                 // [1]
    uint64_t *kb_full, *kb_free;   // [2] expanded K tiles (tensor memory)
    uint64_t *vb_full, *vb_free;   // [2] expanded V tiles
    uint64_t *full_v;              // [kStages] the stage's V boxes landed (full: its K boxes and Q)
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

// ---- E4M3 -> 16-bit expansion (exact) ------------------------------------------
// Four codes in a 32-bit word (code k in byte k) -> two words of 16-bit values,
// code 0/1 in the low/high half of the first word, code 2/3 in the second.
template <typename T> struct Expand;

// f16: the hardware conversion of a code pair (exact: E4M3 is a subset of f16).
template <> struct Expand<__half> {
    static __device__ __forceinline__ void x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
        const uint16_t a = (uint16_t)(w & 0xFFFFu), b = (uint16_t)(w >> 16);
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(a));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(b));
    }
};

// bf16: move the code's exponent and mantissa bits under bf16's (exponent field
// e of the code lands in the low 4 bits of bf16's 8-bit field, the 3 mantissa
// bits on top of bf16's 7), keep the sign, then multiply by 2^120 = 2^(127 - 7)
// to re-bias the exponent. The same factor maps the code's subnormals
// (m/8 * 2^-6) from bf16's subnormals (m/8 * 2^-126), and the product is exact.
template <> struct Expand<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t pair(uint32_t x) {      // codes at bits 8..15 and 24..31
        const uint32_t r = ((x >> 4) & 0x07F007F0u) | (x & 0x80008000u);
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&r);
        const uint32_t k = 0x7B807B80u;                                 // bf16 2^120 in both halves
        const __nv_bfloat162 f = __hmul2(v, *reinterpret_cast<const __nv_bfloat162 *>(&k));
        return *reinterpret_cast<const uint32_t *>(&f);
    }
    static __device__ __forceinline__ void x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
        lo = pair(__byte_perm(w, 0u, 0x1404));    // bytes {0, code0, 0, code1}
        hi = pair(__byte_perm(w, 0u, 0x3424));    // bytes {0, code2, 0, code3}
    }
};

// One token row: 128 codes (8 chunks of 16, 128-byte swizzled) -> 128 16-bit
// values in two 64-dim halves (8 chunks of 8 each, 128-byte swizzled), or zeros.
template <typename T>
__device__ __forceinline__ void expand_row(const unsigned char *src8, unsigned char *dst16, int r, bool zero) {
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
        if (!zero) {
            const uint4 in = *reinterpret_cast<const uint4 *>(src8 + r * 128 + ((c ^ sw) << 4));
            Expand<T>::x4(in.x, o0.x, o0.y);
            Expand<T>::x4(in.y, o0.z, o0.w);
            Expand<T>::x4(in.z, o1.x, o1.y);
            Expand<T>::x4(in.w, o1.z, o1.w);
        }
        const int j = 2 * (c & 3);                                  // 16-bit chunk within the half
        unsigned char *row = dst16 + (c >> 2) * kChunkBytes + r * 128;
        *reinterpret_cast<uint4 *>(row + ((j ^ sw) << 4)) = o0;
        *reinterpret_cast<uint4 *>(row + (((j + 1) ^ sw) << 4)) = o1;
    }
}

// One token row's 128 codes (128-byte swizzled in shared memory) -> 64 words of
// 16-bit pairs, word j = dims (2j, 2j + 1): the row's lane of a K tile in tensor
// memory.
template <typename T>
__device__ __forceinline__ void expand_row_regs(const unsigned char *src8, int r, uint32_t *w) {
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 in = *reinterpret_cast<const uint4 *>(src8 + r * 128 + ((c ^ sw) << 4));
        Expand<T>::x4(in.x, w[8 * c + 0], w[8 * c + 1]);
        Expand<T>::x4(in.y, w[8 * c + 2], w[8 * c + 3]);
        Expand<T>::x4(in.z, w[8 * c + 4], w[8 * c + 5]);
        Expand<T>::x4(in.w, w[8 * c + 6], w[8 * c + 7]);
    }
}

// D (tmem) [+]= A (tmem: M rows in lanes, 16-bit K pairs per column) * B (smem desc).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::
            "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Expand tile rows of K into tensor-memory buffer `buf` (thread = lane = token)
// and signal the MMA issuer.
template <typename T>
__device__ __forceinline__ void expand_k_tmem(const unsigned char *src8, uint32_t tmem, uint32_t lane_off, int r,
                                              int buf, uint64_t *full_bar, int lane) {
    uint32_t w[64];
    expand_row_regs<T>(src8, r, w);
    const uint32_t col = tmem + lane_off + kColK + buf * kKCols;
    tmem_st32(col, w);
    tmem_st32(col + 32, w + 32);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(full_bar);
}

template <typename T, int GT>
__global__ __launch_bounds__(threads_for(GT), 1) void decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                 const __grid_constant__ CUtensorMap tm_v,
                                                                 const __grid_constant__ CUtensorMap tm_q,
                                                                 const DecodeParams p, const float v_scale) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *s8 = smem + kOff8;
    unsigned char *sVb = smem + kOffVb;
    unsigned char *sP = smem + kOffP;
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    float *lred = reinterpret_cast<float *>(smem + kOffLRed);
    uint64_t *bar_base = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
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
    bars.kb_full = bar_base + kBarKbFull;
    bars.kb_free = bar_base + kBarKbFree;
    bars.vb_full = bar_base + kBarVbFull;
    bars.vb_free = bar_base + kBarVbFree;
    bars.full_v = bar_base + kBarFullV;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group;
    constexpr int kVProdWarp = kConvWarp0 + conv_warps(GT);   // last warp: V producer

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.full_v[s], 1);
            mbar_init(&bars.empty[s], conv_warps(GT) + 1);   // converter warps + the S MMA's commit (it reads Q)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_free[i], 4);
            mbar_init(&bars.p_full[i], 4);
            mbar_init(&bars.o_full[i], 1);
            mbar_init(&bars.o_free[i], 4);
            mbar_init(&bars.red[i], 4);          // one arrival per softmax warp
            mbar_init(&bars.vb_full[i], 4);
            mbar_init(&bars.vb_free[i], 1);
            mbar_init(&bars.kb_full[i], 4);
            mbar_init(&bars.kb_free[i], 1);
        }
        mbar_init(bars.fin, 4);
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
    // Programmatic dependent launch: only barrier set-up and the tensor-memory
    // allocation above overlap the preceding kernel.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int *order = reinterpret_cast<int *>(smem + kOffOrder);
    int *counts = reinterpret_cast<int *>(smem + kOffMisc + 8);   // [0] = n4, [1] = list length
    const decode_order::SeqCache cache{reinterpret_cast<int *>(smem + kOffCtx), reinterpret_cast<int *>(smem + kOffPs)};
    decode_order::build(p, prefix, order, counts, sP, cache);            // P buffer as scratch until the first tile
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n4 = counts[0];
    const int total_items = (counts[0] + counts[1]) * p.num_kv_heads;
    // this CTA's item descriptors, computed once and kept over the ordering arrays
    int4 *items = reinterpret_cast<int4 *>(smem + kOffPrefix);
    decode_order::build_item_table<(decode_order::kTableItems + threads_for(GT) - 1) / threads_for(GT)>(p, prefix, order, n4, cache, total_items, items);
    const int nmy = decode_order::cta_items(total_items);
    __syncthreads();

    if (warp == 0 || warp == kVProdWarp) {
        // ------------------------------------------------------------ producers
        // warp 0: the tile's K boxes and the group's query rows (on `full`);
        // the V producer: the tile's V boxes (on `full_v`). One issuing warp
        // per operand halves the copy-issue time each tile waits for.
        const bool is_v = warp == kVProdWarp;
        uint64_t *fullb = is_v ? bars.full_v : bars.full;
        const int nbt = kTile / p.block_size;       // physical blocks per tile
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const decode_order::ItemTable tb = decode_order::load_item_table(p, I, lane);
            const int qrow = I.b * p.num_heads + I.kvh * G;
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int stage = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                bool live;
                const int e = decode_order::tile_entry(tb, tile, nbt, lane, &live);
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
                if (lane == 0) mbar_arrive_expect_tx(&fullb[stage], is_v ? kTile8Bytes : kTile8Bytes + kQBytes);
                __syncwarp();
                unsigned char *st = s8 + stage * kStageBytes;
                if (lane < nbt)
                    tma_load_4d(st + (is_v ? kTile8Bytes : 0) + lane * p.block_size * 128, is_v ? &tm_v : &tm_k,
                                &fullb[stage], 0, I.kvh, 0, phys);
                if (lane == 0 && !is_v) {
                    unsigned char *dq = st + 2 * kTile8Bytes;
                    tma_load_2d(dq, &tm_q, &fullb[stage], 0, qrow);
                    tma_load_2d(dq + kN * 128, &tm_q, &fullb[stage], 64, qrow);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
        // drain: every issued stage's copies must have landed before the CTA exits
        if (lane == 0) {
            const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
            for (uint32_t j = first; j < it; ++j) mbar_wait(&fullb[j % kStages], (j / kStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S MMA issuer
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t idesc_s = instr_desc_f16(kTile, kN, kBf16, false, false);
            const uint32_t s80 = smem_addr(s8);
            uint32_t it = 0;
            bool ok = true;
            for (int k = 0; k < nmy && ok; ++k) {
                const Item I = decode_order::unpack_item(items[k]);
                for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                    const int stage = it % kStages, buf = it & 1;
                    if (*abort_flag || !mbar_wait(&bars.full[stage], (it / kStages) & 1) ||
                        !mbar_wait(&bars.kb_full[buf], (it >> 1) & 1) ||
                        !mbar_wait(&bars.s_free[buf], ((it >> 1) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qbase = s80 + stage * kStageBytes + 2 * kTile8Bytes;
                    const uint32_t dcol = tmem + buf * kN;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t qoff = (kk >> 2) * (kN * 128) + (kk & 3) * 32;
                        const uint64_t b = smem_desc(qbase + qoff, 16, 1024);
                        mma_f16_tmem_a(dcol, tmem + kColK + buf * kKCols + kk * 8, b, idesc_s, kk > 0);
                    }
                    mma_commit(&bars.s_full[buf]);
                    mma_commit(&bars.kb_free[buf]);
                    mma_commit(&bars.empty[stage]);
                }
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
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            const uint32_t idesc_o = instr_desc_f16(kD, kN, kBf16, true, false);
            const uint32_t sVb0 = smem_addr(sVb), sP0 = smem_addr(sP);
            uint32_t it = 0;
            bool ok = true;
            for (int k = 0; k < nmy && ok; ++k) {
                const Item I = decode_order::unpack_item(items[k]);
                for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                    const int buf = it & 1;
                    const uint32_t bph = (it >> 1) & 1;
                    if (*abort_flag || !mbar_wait(&bars.p_full[buf], bph) || !mbar_wait(&bars.vb_full[buf], bph) ||
                        !mbar_wait(&bars.o_free[buf], bph ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t vbase = sVb0 + buf * kKVBytes;
                    const uint32_t pbase = sP0 + buf * kPBytes;
                    const uint32_t dcol = tmem + 2 * kN + buf * kN;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t a = smem_desc(vbase + kk * 2048, kChunkBytes, 1024);
                        const uint64_t b = smem_desc(pbase + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
                        mma_f16(dcol, a, b, idesc_o, kk > 0);
                    }
                    mma_commit(&bars.o_full[buf]);
                    mma_commit(&bars.vb_free[buf]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, PA_DEVERR_WAIT);
            }
        }
        __syncwarp();
    } else if (warp >= kConvWarp0 && conv_warps(GT) == 8) {   // (the V producer is handled above)
        // ------------------------------------------------------------ converters (K | V)
        const bool is_k = warp < kConvWarp0 + 4;
        const int r = (warp & 3) * 32 + lane;            // token row = tensor-memory lane of this thread
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int stage = it % kStages, buf = it & 1;
                uint64_t *free_bar = is_k ? &bars.kb_free[buf] : &bars.vb_free[buf];
                if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                    !warp_wait(is_k ? &bars.full[stage] : &bars.full_v[stage], (it / kStages) & 1) ||
                    !warp_wait(free_bar, ((it >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const unsigned char *src = s8 + stage * kStageBytes;
                if (is_k) {
                    tc_fence_after();
                    expand_k_tmem<T>(src, tmem, lane_off, r, buf, &bars.kb_full[buf], lane);
                } else {
                    const int valid_rows = I.t1 - (I.t0 + tile * kTile);
                    expand_row<T>(src + kTile8Bytes, sVb + buf * kKVBytes, r, r >= valid_rows);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.vb_full[buf]);
                }
                if (lane == 0) mbar_arrive(&bars.empty[stage]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
    } else if (warp >= kConvWarp0) {
        // ------------------------------------------------------------ converters (K then V)
        // Tile j's K is expanded before tile j-1's V, so the S MMA of the next
        // tile never waits behind a V expansion.
        const int r = (warp & 3) * 32 + lane;            // token row = tensor-memory lane of this thread
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        bool have_prev = false;
        uint32_t prev_it = 0;
        int prev_valid_rows = 0;                        // rows of the previous tile inside its partition
        auto expand_v = [&](uint32_t j, int valid_rows) -> bool {
            const int buf = j & 1, stage = j % kStages;
            if (!warp_wait(&bars.full_v[stage], (j / kStages) & 1) ||
                !warp_wait(&bars.vb_free[buf], ((j >> 1) & 1) ^ 1))
                return false;
            expand_row<T>(s8 + stage * kStageBytes + kTile8Bytes, sVb + buf * kKVBytes, r, r >= valid_rows);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars.vb_full[buf]);
                mbar_arrive(&bars.empty[stage]);
            }
            return true;
        };
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int stage = it % kStages, buf = it & 1;
                if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                    !warp_wait(&bars.full[stage], (it / kStages) & 1) ||
                    !warp_wait(&bars.kb_free[buf], ((it >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                expand_k_tmem<T>(s8 + stage * kStageBytes, tmem, lane_off, r, buf, &bars.kb_full[buf], lane);
                if (have_prev && !expand_v(prev_it, prev_valid_rows)) {
                    ok = false;
                    break;
                }
                have_prev = true;
                prev_it = it;
                prev_valid_rows = I.t1 - (I.t0 + tile * kTile);
            }
        }
        if (ok && have_prev && !expand_v(prev_it, prev_valid_rows)) ok = false;
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, PA_DEVERR_WAIT);
        }
    } else {
        // ------------------------------------------------------------ softmax / output
        const int q4 = warp & 3;                       // tensor-memory lane quadrant
        const int row = q4 * 32 + lane;                // token (S) or dim (O) of this thread
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        T *out = reinterpret_cast<T *>(p.out);
        uint32_t it = 0, nfin = 0;
        bool ok = true;
        float m_run[GT], l_part[GT], o_acc[GT], alpha_prev[GT];
        for (int k = 0; k < nmy && ok; ++k) {
            const Item I = decode_order::unpack_item(items[k]);
            const int64_t head0 = (int64_t)I.b * p.num_heads + (int64_t)I.kvh * G;
            if (I.ntiles == 0) {
#pragma unroll
                for (int g = 0; g < GT; ++g)
                    if (g < G) out[(head0 + g) * kD + row] = Elem<T>::from_f(0.f);
                continue;
            }
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
                float o[16];
                tmem_ld16(tmem + lane_off + 2 * kN + buf * kN, o);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.o_free[buf]);
#pragma unroll
                for (int g = 0; g < GT; ++g) o_acc[g] = fmaf(o_acc[g], alpha_prev[g], o[g]);
                return true;
            };
            for (int tile = 0; tile < I.ntiles; ++tile, ++it) {
                const int buf = it & 1;
                if (__any_sync(0xffffffffu, *abort_flag != 0) || !warp_wait(&bars.s_full[buf], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float s[16];
                tmem_ld16(tmem + lane_off + buf * kN, s);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.s_free[buf]);

                const int tok = I.t0 + tile * kTile + row;
                const bool valid = tok < I.t1;
                float *rd = red + (it & 1) * 4 * kN;
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    s[g] = valid ? s[g] * p.scale_log2 : -INFINITY;
                    const float mx = warp_max(s[g]);
                    if (lane == 0) rd[q4 * kN + g] = mx;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.red[it & 1]);
                if (!warp_wait(&bars.red[it & 1], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                float alpha[GT];
                unsigned char *pb = sP + buf * kPBytes + (row >> 6) * (kN * 128);
                const int colb = (row & 63) * 2;
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    const float tmax = fmaxf(fmaxf(rd[g], rd[kN + g]), fmaxf(rd[2 * kN + g], rd[3 * kN + g]));
                    const float m_new = fmaxf(m_run[g], tmax);
                    alpha[g] = fast_exp2(m_run[g] - m_new);
                    m_run[g] = m_new;
                    const uint16_t bits = to_bits<T>(valid ? fast_exp2(s[g] - m_new) : 0.f);
                    l_part[g] = fmaf(l_part[g], alpha[g], from_bits<T>(bits));
                    unsigned char *dst = pb + g * 128 + ((((colb >> 4) ^ (g & 7)) << 4) | (colb & 15));
                    *reinterpret_cast<uint16_t *>(dst) = bits;
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
            float *lr = lred + (nfin & 1) * 4 * kN;
#pragma unroll
            for (int g = 0; g < GT; ++g) {
                const float ls = warp_sum(l_part[g]);
                if (lane == 0) lr[q4 * kN + g] = ls;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.fin);
            if (!warp_wait(bars.fin, nfin++ & 1)) {
                ok = false;
                break;
            }
            float l_tot[GT];
#pragma unroll
            for (int g = 0; g < GT; ++g) l_tot[g] = lr[g] + lr[kN + g] + lr[2 * kN + g] + lr[3 * kN + g];
            if (I.direct) {
#pragma unroll
                for (int g = 0; g < GT; ++g)
                    if (g < G) out[(head0 + g) * kD + row] = Elem<T>::from_f(o_acc[g] * v_scale / l_tot[g]);
            } else {
                const int P = p.max_partitions;
#pragma unroll
                for (int g = 0; g < GT; ++g) {
                    if (g < G) {
                        const int64_t r = (head0 + g) * P + I.slot;
                        p.ws_o[r * kD + row] = o_acc[g] * v_scale;
                        if (row == 0) {
                            p.ws_ml[2 * r] = m_run[g];
                            p.ws_ml[2 * r + 1] = l_tot[g];
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

template <typename T, int GT>
int launch_t(const DecodeParams &p, float v_scale, CUtensorMapDataType dt, cudaStream_t stream) {
    auto kern = decode_fp8_kernel<T, GT>;
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
    if (!make_cache_map_u8(&mk, p.key_cache, p) || !make_cache_map_u8(&mv, p.value_cache, p) ||
        !make_q_map(&mq, p, dt))
        return -1;
    const int64_t max_items = (int64_t)p.num_seqs * p.num_kv_heads * p.max_partitions;
    const int grid = (int)(max_items < num_sms[dev] ? max_items : num_sms[dev]);
    return launch_pdl(kern, dim3(grid), dim3(threads_for(GT)), kSmemBytes, stream, mk, mv, mq, p, v_scale);
}

template <typename T>
int launch_g(const DecodeParams &p, float v_scale, CUtensorMapDataType dt, cudaStream_t stream) {
    if (p.group <= 4) return launch_t<T, 4>(p, v_scale, dt, stream);
    if (p.group <= 8) return launch_t<T, 8>(p, v_scale, dt, stream);
    return launch_t<T, 16>(p, v_scale, dt, stream);
}

}  // namespace

bool decode_fp8_supported(const DecodeParams &p, int dtype) {
    return (dtype == PA_DTYPE_BF16 || dtype == PA_DTYPE_F16) && p.head_dim == kD && p.group >= 1 &&
           p.group <= kN && p.block_size >= 8 && p.block_size <= kTile && p.partition_size % kTile == 0 &&
           p.num_blocks < INT32_MAX && (int64_t)p.num_seqs * p.num_heads < INT32_MAX;
}

// Batches above kMaxSeqs sequences run as independent launches of up to kMaxSeqs.
int launch_decode_fp8(const DecodeParams &p, float v_scale, int dtype, cudaStream_t stream) {
    if (!decode_fp8_supported(p, dtype)) return -2;
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
        if (p.ws_ml) {
            c.ws_ml = p.ws_ml + rows * p.max_partitions * 2;
            c.ws_o = p.ws_o + rows * p.max_partitions * kD;
        }
        const int rc = dtype == PA_DTYPE_BF16
                           ? launch_g<__nv_bfloat16>(c, v_scale, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, stream)
                           : launch_g<__half>(c, v_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, stream);
        if (rc != 0) return rc;
    }
    return 0;
}

}  // namespace pa
