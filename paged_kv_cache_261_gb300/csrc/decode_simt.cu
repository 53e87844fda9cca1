// Decode attention, SIMT variant (fp32/fp16/bf16 caches; head_dim 64 or 128).
//
// Computes, for each sequence b and query head h (kv head h / G), the
// single-query attention of "CS349E lecture 7: 01_paged_attention.py", demo 2,
// paper eq. 4: scores against every cached key are formed block by block
// through the block table, one softmax is taken over the whole context, and V
// is accumulated block by block. The one softmax is computed online: a running
// max and sum per head, rescaled whenever the max grows, give exactly the
// softmax over the whole context once normalised.
//
// Work unit: one CTA per (partition of partition_size tokens, kv head,
// sequence); all G query heads of the kv head share each K/V tile read. Tiles
// of 32 tokens are gathered row by row through the block table with 16-byte
// cp.async into a double-buffered shared-memory ring (rows XOR-swizzled at
// 16-byte granularity so a warp reading 32 different rows is conflict-free).
// Scores: lane = token, each warp owns whole query heads, so the tile max is a
// warp shuffle reduction and no block barrier is needed for it. PV: each thread
// owns two adjacent output columns of a subset of the heads.
//
// A sequence with one partition gets its final row here; otherwise the
// partition writes its max (log2 units), sum and unnormalised output to the
// workspace and decode_reduce merges them.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kTile = 32;

template <typename T, int D, int GT>
struct SimtCfg {
    static constexpr int kVN = Vec16<T>::N;                 // elements per 16-byte chunk
    static constexpr int kChunks = D / kVN;                 // chunks per row
    static constexpr int kRowBytes = D * (int)sizeof(T);
    static constexpr int kHeadsPerWarp = (GT + 3) / 4;
    static constexpr int kPairs = D / 2;
    static constexpr int kHeadSlices = kThreads / kPairs;   // 2 (D=128) or 4 (D=64)
    static constexpr int kHeadsPerThread = (GT + kHeadSlices - 1) / kHeadSlices;
    // shared memory carve-up (bytes)
    static constexpr int kQBytes = GT * D * 4;
    static constexpr int kStageBytes = 2 * kTile * kRowBytes;   // K and V
    static constexpr int kPBytes = kTile * GT * 4;
    static constexpr int kSmem = kQBytes + 2 * kStageBytes + kPBytes + 4 * GT * 4;
    static_assert(kChunks >= 8, "swizzle needs at least 8 chunks per row");
};

template <typename T, int D, int GT>
__global__ __launch_bounds__(kThreads) void decode_simt_kernel(const DecodeParams p) {
    using C = SimtCfg<T, D, GT>;
    extern __shared__ __align__(16) unsigned char smem[];
    float *q_s = reinterpret_cast<float *>(smem);                                   // [GT][D]
    unsigned char *stage_base = smem + C::kQBytes;                                  // 2 stages
    float *p_s = reinterpret_cast<float *>(smem + C::kQBytes + 2 * C::kStageBytes); // [kTile][GT]
    float *alpha_s = p_s + kTile * GT;                                              // [GT]
    float *m_s = alpha_s + GT;
    float *l_s = m_s + GT;

    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.group;
    // programmatic dependent launch: the merge kernel may launch now, and nothing
    // below is read before the preceding kernel in the stream has finished
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.context_limit) {
        if (tid == 0 && part == 0 && kvh == 0) raise_error(p.err, PA_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : p.context_limit;
    }
    const int nparts = ctx == 0 ? 1 : (ctx + p.partition_size - 1) / p.partition_size;
    if (part >= nparts) return;

    T *out = reinterpret_cast<T *>(p.out);
    const int64_t head0 = (int64_t)b * p.num_heads + (int64_t)kvh * G;
    if (ctx == 0) {
        for (int i = tid; i < G * D; i += kThreads) out[head0 * D + i] = Elem<T>::from_f(0.f);
        return;
    }
    const int t0 = part * p.partition_size;
    const int t1 = min(ctx, t0 + p.partition_size);

    // queries of the group, pre-multiplied by scale*log2(e)
    const T *q = reinterpret_cast<const T *>(p.q);
    for (int i = tid; i < GT * D; i += kThreads) {
        const int g = i / D;
        q_s[i] = g < G ? Elem<T>::to_f(q[head0 * D + i]) * p.scale_log2 : 0.f;
    }

    const T *kc = reinterpret_cast<const T *>(p.key_cache);
    const T *vc = reinterpret_cast<const T *>(p.value_cache);
    const int32_t *table = p.block_tables + (int64_t)b * p.max_blocks_per_seq;
    const int bs_mask = p.block_size - 1;

    auto issue_tile = [&](int tile_start, int stage) {
        unsigned char *ks = stage_base + stage * C::kStageBytes;
        unsigned char *vs = ks + kTile * C::kRowBytes;
        for (int idx = tid; idx < kTile * C::kChunks; idx += kThreads) {
            const int r = idx / C::kChunks, c = idx % C::kChunks;
            const int t = tile_start + r;
            const T *ksrc = kc, *vsrc = vc;
            int bytes = 0;
            if (t < t1) {
                const int32_t phys = table[t >> p.log2_block_size];
                if (phys >= 0 && phys < p.num_blocks) {
                    const int64_t row = ((int64_t)phys * p.block_size + (t & bs_mask)) * p.num_kv_heads + kvh;
                    ksrc = kc + row * D + c * C::kVN;
                    vsrc = vc + row * D + c * C::kVN;
                    bytes = 16;
                } else if (c == 0) {
                    raise_error(p.err, PA_DEVERR_BLOCK_ID);
                }
            }
            const int off = r * C::kRowBytes + ((c ^ (r & 7)) * 16);
            cp_async16(ks + off, ksrc, bytes);
            cp_async16(vs + off, vsrc, bytes);
        }
    };

    // per-warp running max (log2 units) of the heads the warp owns
    float m_run[C::kHeadsPerWarp], l_lane[C::kHeadsPerWarp];
#pragma unroll
    for (int hh = 0; hh < C::kHeadsPerWarp; ++hh) {
        m_run[hh] = -INFINITY;
        l_lane[hh] = 0.f;
    }
    // PV accumulators: column pair `pair`, heads slice + kHeadSlices*k
    const int pair = tid % C::kPairs, slice = tid / C::kPairs;
    float o[C::kHeadsPerThread][2];
#pragma unroll
    for (int k = 0; k < C::kHeadsPerThread; ++k) o[k][0] = o[k][1] = 0.f;

    const int ntiles = (t1 - t0 + kTile - 1) / kTile;
    issue_tile(t0, 0);
    cp_async_commit();
    for (int it = 0; it < ntiles; ++it) {
        const int stage = it & 1;
        if (it + 1 < ntiles) issue_tile(t0 + (it + 1) * kTile, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const unsigned char *ks = stage_base + stage * C::kStageBytes;
        const unsigned char *vs = ks + kTile * C::kRowBytes;
        const int tile_start = t0 + it * kTile;
        const int nvalid = min(kTile, t1 - tile_start);

        // ---- scores: lane = token, warp owns heads warp, warp+4, ...
        {
            const int r = lane;
            float acc[C::kHeadsPerWarp];
#pragma unroll
            for (int hh = 0; hh < C::kHeadsPerWarp; ++hh) acc[hh] = 0.f;
#pragma unroll 4
            for (int c = 0; c < C::kChunks; ++c) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(ks + r * C::kRowBytes + ((c ^ (r & 7)) * 16));
                float kf[C::kVN];
                Vec16<T>::unpack(raw, kf);
#pragma unroll
                for (int hh = 0; hh < C::kHeadsPerWarp; ++hh) {
                    const int g = warp + 4 * hh;
                    if (g < GT) {
                        const float4 *qv = reinterpret_cast<const float4 *>(q_s + g * D + c * C::kVN);
#pragma unroll
                        for (int e4 = 0; e4 < C::kVN / 4; ++e4) {
                            const float4 qq = qv[e4];
                            acc[hh] = fmaf(qq.x, kf[4 * e4 + 0], acc[hh]);
                            acc[hh] = fmaf(qq.y, kf[4 * e4 + 1], acc[hh]);
                            acc[hh] = fmaf(qq.z, kf[4 * e4 + 2], acc[hh]);
                            acc[hh] = fmaf(qq.w, kf[4 * e4 + 3], acc[hh]);
                        }
                    }
                }
            }
            // ---- online softmax over the tile (warp-local per head)
#pragma unroll
            for (int hh = 0; hh < C::kHeadsPerWarp; ++hh) {
                const int g = warp + 4 * hh;
                if (g < GT) {
                    const float s = r < nvalid ? acc[hh] : -INFINITY;
                    float mx = s;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    const float m_new = fmaxf(m_run[hh], mx);
                    const float alpha = fast_exp2(m_run[hh] - m_new);
                    const float pr = r < nvalid ? fast_exp2(s - m_new) : 0.f;
                    l_lane[hh] = l_lane[hh] * alpha + pr;
                    m_run[hh] = m_new;
                    p_s[r * GT + g] = pr;
                    if (lane == 0) alpha_s[g] = alpha;
                }
            }
        }
        __syncthreads();

        // ---- PV: o[g][d] = o[g][d]*alpha[g] + sum_r p[r][g] * V[r][d]
#pragma unroll
        for (int k = 0; k < C::kHeadsPerThread; ++k) {
            const int g = slice + C::kHeadSlices * k;
            if (g < GT) {
                const float a = alpha_s[g];
                o[k][0] *= a;
                o[k][1] *= a;
            }
        }
        {
            const int byte_in_row = pair * 2 * (int)sizeof(T);
            const int c = byte_in_row / 16, within = byte_in_row % 16;
            for (int r = 0; r < nvalid; ++r) {
                const unsigned char *vp = vs + r * C::kRowBytes + ((c ^ (r & 7)) * 16) + within;
                float v0, v1;
                if constexpr (sizeof(T) == 4) {
                    const float2 f = *reinterpret_cast<const float2 *>(vp);
                    v0 = f.x; v1 = f.y;
                } else {
                    const T *e = reinterpret_cast<const T *>(vp);
                    v0 = Elem<T>::to_f(e[0]);
                    v1 = Elem<T>::to_f(e[1]);
                }
#pragma unroll
                for (int k = 0; k < C::kHeadsPerThread; ++k) {
                    const int g = slice + C::kHeadSlices * k;
                    if (g < GT) {
                        const float pr = p_s[r * GT + g];
                        o[k][0] = fmaf(pr, v0, o[k][0]);
                        o[k][1] = fmaf(pr, v1, o[k][1]);
                    }
                }
            }
        }
        __syncthreads();   // stage `stage` and p_s are reused next iteration
    }
    cp_async_wait<0>();

    // ---- per-head totals
#pragma unroll
    for (int hh = 0; hh < C::kHeadsPerWarp; ++hh) {
        const int g = warp + 4 * hh;
        if (g < GT) {
            float l = l_lane[hh];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) {
                m_s[g] = m_run[hh];
                l_s[g] = l;
            }
        }
    }
    __syncthreads();

    if (nparts == 1) {
#pragma unroll
        for (int k = 0; k < C::kHeadsPerThread; ++k) {
            const int g = slice + C::kHeadSlices * k;
            if (g < G) {
                const float inv = 1.f / l_s[g];
                T *dst = out + (head0 + g) * D + 2 * pair;
                dst[0] = Elem<T>::from_f(o[k][0] * inv);
                dst[1] = Elem<T>::from_f(o[k][1] * inv);
            }
        }
    } else {
        const int P = p.max_partitions;
#pragma unroll
        for (int k = 0; k < C::kHeadsPerThread; ++k) {
            const int g = slice + C::kHeadSlices * k;
            if (g < G) {
                const int64_t row = (head0 + g) * P + part;
                float2 *dst = reinterpret_cast<float2 *>(p.ws_o + row * D + 2 * pair);
                *dst = make_float2(o[k][0], o[k][1]);
                if (pair == 0) {
                    p.ws_ml[2 * row] = m_s[g];
                    p.ws_ml[2 * row + 1] = l_s[g];
                }
            }
        }
    }
}

// Merge of partition partials: M = max m_p, L = sum l_p 2^(m_p - M),
// out = sum_p o_p 2^(m_p - M) / L. One CTA of 8 warps per (query head,
// sequence): every warp takes a strided subset of the partitions in one pass,
// keeping its own running max, sum and output (each lane owning 4 (head_dim 128)
// or 2 (head_dim 64) consecutive dimensions), and the 8 warps' results are
// combined through shared memory. (A first pass of warp 0 over the (m, l) pairs
// for M and L, with the other warps waiting, cost two round trips a row; a pass
// that rescaled after every partition kept one partition's loads in flight per
// warp and was slower still.)
constexpr int kReduceWarps = 8;
constexpr int kReduceThreads = 32 * kReduceWarps;

template <typename T, int VEC>
__device__ __forceinline__ void merge_row(const DecodeParams &p, int b, int h, int nparts, float *part_sum,
                                          float *ml_s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.head_dim, P = p.max_partitions;
    const int64_t row0 = ((int64_t)b * p.num_heads + h) * P;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + row0;
    const float *o = p.ws_o + row0 * D + lane * VEC;
    // one pass: the warp's running max m, sum l and output over its partitions, loaded
    // kBatch at a time (all loads of a batch in flight together) and rescaled once per
    // batch to the batch's max
    constexpr int kBatch = 8;
    float m = -INFINITY, l = 0.f, acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    for (int i0 = warp; i0 < nparts; i0 += kReduceWarps * kBatch) {
        float2 mi[kBatch];
        float x[kBatch][VEC];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int i = i0 + k * kReduceWarps;
            mi[k] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int v = 0; v < VEC; ++v) x[k][v] = 0.f;
            if (i < nparts) {
                mi[k] = ml[i];
                if constexpr (VEC == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(o + (int64_t)i * D);
                    x[k][0] = t.x;
                    x[k][1] = t.y;
                    x[k][2] = t.z;
                    x[k][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2 *>(o + (int64_t)i * D);
                    x[k][0] = t.x;
                    x[k][1] = t.y;
                }
            }
        }
        float mb = m;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, mi[k].x);
        if (mb == -INFINITY) continue;          // nothing visible yet
        const float a = fast_exp2(m - mb);      // m = -inf (nothing yet): 0
        l *= a;
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] *= a;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float c = mi[k].x == -INFINITY ? 0.f : fast_exp2(mi[k].x - mb);
            l = fmaf(mi[k].y, c, l);
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[v] = fmaf(x[k][v], c, acc[v]);
        }
        m = mb;
    }
    // the warps' results: M = the largest m, each warp's l and output scaled by 2^(m_w - M)
    if (lane == 0) {
        ml_s[2 * warp] = m;
        ml_s[2 * warp + 1] = l;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) part_sum[warp * 128 + lane * VEC + v] = acc[v];
    __syncthreads();
    if (threadIdx.x < D) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) M = fmaxf(M, ml_s[2 * w]);
        float t = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) {
            const float mw = ml_s[2 * w];
            const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
            L = fmaf(ml_s[2 * w + 1], f, L);
            t = fmaf(part_sum[w * 128 + threadIdx.x], f, t);
        }
        reinterpret_cast<T *>(p.out)[((int64_t)b * p.num_heads + h) * D + threadIdx.x] = Elem<T>::from_f(t / L);
    }
}

// Few partitions (at most kWarpRowMaxParts): one warp merges a whole
// (sequence, head) row, with no shared memory and no block barrier.
constexpr int kWarpRowMaxParts = 32;

// kPre > 0 (launches whose rows hold at most kPre partitions): the partials go out
// with the (m, l) pairs, so a row is one round trip; their slots are read even for
// rows the partition kernel wrote itself, so launches where many rows are whole
// (more partitions per row than kPre) keep the two round trips.
template <typename T, int VEC, int kPre>
__device__ __forceinline__ void merge_row_warp(const DecodeParams &p, int b, int h) {
    const int lane = threadIdx.x & 31;
    const int D = p.head_dim, P = p.max_partitions;
    const int64_t row0 = ((int64_t)b * p.num_heads + h) * P;
    // The (m, l) pairs are read together with the sequence's length (one round
    // trip, not two); entries past its partition count lie inside its row of the
    // workspace and are ignored. The partials themselves are read once the count
    // is known: rows written directly by the partition kernel read none.
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + row0;
    float2 mine = lane < P ? ml[lane] : make_float2(-INFINITY, 0.f);
    // the first kPre partials go out with them (slots past the row's count are read
    // but never used)
    const float *o = p.ws_o + row0 * D + lane * VEC;
    float pre[kPre > 0 ? kPre : 1][VEC];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
        if (i < P) {
            if constexpr (VEC == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(o + (int64_t)i * D);
                pre[i][0] = x.x;
                pre[i][1] = x.y;
                pre[i][2] = x.z;
                pre[i][3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2 *>(o + (int64_t)i * D);
                pre[i][0] = x.x;
                pre[i][1] = x.y;
            }
        }
    }
    const SeqSplit sp = seq_split(p, b);
    if (sp.direct) return;                      // the partition kernel wrote the row
    const int nparts = sp.shared + sp.priv;
    if (lane >= nparts) mine = make_float2(-INFINITY, 0.f);
    float M = mine.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float e = lane < nparts ? fast_exp2(mine.x - M) : 0.f;
    float L = mine.y * e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float c_mine = e / L;
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
        const float c = __shfl_sync(0xffffffffu, c_mine, i);
        if (i < nparts) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[v] = fmaf(c, pre[i][v], acc[v]);
        }
    }
#pragma unroll 4
    for (int i = kPre; i < nparts; ++i) {
        const float c = __shfl_sync(0xffffffffu, c_mine, i);
        if constexpr (VEC == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(o + (int64_t)i * D);
            acc[0] = fmaf(c, x.x, acc[0]);
            acc[1] = fmaf(c, x.y, acc[1]);
            acc[2] = fmaf(c, x.z, acc[2]);
            acc[3] = fmaf(c, x.w, acc[3]);
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(o + (int64_t)i * D);
            acc[0] = fmaf(c, x.x, acc[0]);
            acc[1] = fmaf(c, x.y, acc[1]);
        }
    }
    T *dst = reinterpret_cast<T *>(p.out) + ((int64_t)b * p.num_heads + h) * D + lane * VEC;
#pragma unroll
    for (int v = 0; v < VEC; ++v) dst[v] = Elem<T>::from_f(acc[v]);
}

template <typename T, int kPre>
__global__ __launch_bounds__(kReduceThreads) void decode_reduce_warp_kernel(const DecodeParams p) {
    // chain_next: the next call's partition kernel may launch and set itself up
    // meanwhile (it waits for this grid before it touches the workspace or the output)
    if (p.chain_next) asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t row = (int64_t)blockIdx.x * kReduceWarps + (threadIdx.x >> 5);
    if (row >= (int64_t)p.num_seqs * p.num_heads) return;
    const int b = (int)(row / p.num_heads), h = (int)(row % p.num_heads);
    if (p.head_dim == 128) merge_row_warp<T, 4, kPre>(p, b, h);
    else merge_row_warp<T, 2, kPre>(p, b, h);
}

template <typename T>
__global__ __launch_bounds__(kReduceThreads) void decode_reduce_kernel(const DecodeParams p) {
    // a no-op unless launched as a programmatic dependent of the partition kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ __align__(16) float part_sum[kReduceWarps * 128];
    __shared__ float ml_s[2 * kReduceWarps];
    const int h = blockIdx.x, b = blockIdx.y;
    const SeqSplit sp = seq_split(p, b);
    if (sp.direct) return;                      // the partition kernel wrote the row
    const int nparts = sp.shared + sp.priv;
    if (p.head_dim == 128) merge_row<T, 4>(p, b, h, nparts, part_sum, ml_s);
    else merge_row<T, 2>(p, b, h, nparts, part_sum, ml_s);
}

template <typename T, int D, int GT>
int launch_simt_t(const DecodeParams &p, cudaStream_t stream) {
    using C = SimtCfg<T, D, GT>;
    auto kern = decode_simt_kernel<T, D, GT>;
    static bool attr_set[kMaxDevices] = {};   // the opt-in is per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return -1;
        attr_set[dev] = true;
    }
    dim3 grid((unsigned)p.max_partitions, (unsigned)p.num_kv_heads, (unsigned)p.num_seqs);
    return launch_pdl(kern, grid, dim3(kThreads), C::kSmem, stream, p);
}

template <typename T, int D>
int launch_simt_g(const DecodeParams &p, cudaStream_t stream) {
    const int G = p.group;
    if (G <= 1) return launch_simt_t<T, D, 1>(p, stream);
    if (G <= 2) return launch_simt_t<T, D, 2>(p, stream);
    if (G <= 4) return launch_simt_t<T, D, 4>(p, stream);
    if (G <= 8) return launch_simt_t<T, D, 8>(p, stream);
    if (G <= 16) return launch_simt_t<T, D, 16>(p, stream);
    return -2;
}

template <typename T>
int launch_simt_d(const DecodeParams &p, cudaStream_t stream) {
    if (p.head_dim == 64) return launch_simt_g<T, 64>(p, stream);
    if (p.head_dim == 128) return launch_simt_g<T, 128>(p, stream);
    return -2;
}

}  // namespace

int launch_decode_simt(const DecodeParams &p, int dtype, cudaStream_t stream) {
    switch (dtype) {
    case PA_DTYPE_F32: return launch_simt_d<float>(p, stream);
    case PA_DTYPE_F16: return launch_simt_d<__half>(p, stream);
    case PA_DTYPE_BF16: return launch_simt_d<__nv_bfloat16>(p, stream);
    default: return -2;
    }
}

template <typename T>
int launch_reduce_t(const DecodeParams &p, cudaStream_t stream) {
    if (p.max_partitions <= kWarpRowMaxParts) {
        // rows of at most 4 partitions: their partials are loaded with the (m, l) pairs
        // (8B-shaped batch: 0.0974 -> 0.0965 ms a call; with up to 8 partitions, most rows
        // of the mixed-serving batch are whole and the early loads cost more than they save)
        const int64_t rows = (int64_t)p.num_seqs * p.num_heads;
        dim3 grid((unsigned)((rows + kReduceWarps - 1) / kReduceWarps));
        if (p.max_partitions <= 4)
            return launch_pdl(decode_reduce_warp_kernel<T, 4>, grid, dim3(kReduceThreads), 0, stream, p);
        return launch_pdl(decode_reduce_warp_kernel<T, 0>, grid, dim3(kReduceThreads), 0, stream, p);
    }
    // Launched plainly: measured on the long-context batch, early-launched CTAs of
    // this form slowed the partition kernel down (0.4608 vs 0.4515 ms).
    dim3 grid((unsigned)p.num_heads, (unsigned)p.num_seqs);
    decode_reduce_kernel<T><<<grid, kReduceThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_decode_reduce(const DecodeParams &p, int dtype, cudaStream_t stream) {
    switch (dtype) {
    case PA_DTYPE_F32: return launch_reduce_t<float>(p, stream);
    case PA_DTYPE_F16: return launch_reduce_t<__half>(p, stream);
    case PA_DTYPE_BF16: return launch_reduce_t<__nv_bfloat16>(p, stream);
    default: return -2;
    }
}

}  // namespace pa
