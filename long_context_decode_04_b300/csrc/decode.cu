// decode.cu -- split-KV exact decode: one partial (m, l, o) per KV chunk.
//
// What is computed (Attention glossary, jisaku.com/glossary/attention,
// "basic concepts and operating principle"): for the query of each
// (sequence b, query head h), scores s_j = scale * <q, k_j> over the
// attended keys, softmax weights, and the weighted mean of the values.
// The keys are cut into chunks; each chunk yields the partial
//   m = a reference point (>= max_j s_j - 8 ln 2), l = sum_j e^(s_j - m),
//   o = sum_j e^(s_j - m) v_j,
// and partials are merged by the log-sum-exp rule (Tree Attention
// explainer, aibr.jp/archives/143699, sections 1 and 3).  Decode reads the
// whole KV cache once per token and is bound by HBM bandwidth (Attention
// glossary, "the memory bandwidth and VRAM wall"), so the kernel is built
// to stream K and V at full bandwidth with the arithmetic hidden under it.
//
// Kernel layout (one CTA per SM, persistent):
//   * warp 8, lane 0 is the producer.  It pulls work items
//     (sequence, KV head, chunk) from a device-wide queue and stages the
//     chunk's K and V rows into shared memory, TILE keys at a time, with
//     one-dimensional bulk async copies into a 3-stage ring guarded by
//     mbarriers.  Each stage carries a small descriptor (item, first key,
//     key count, first/last flags) so the consumers need no schedule.
//   * warps 0-7 consume.  Each warp owns a 1/8 slice of every tile; inside
//     a warp, 8 lanes share one key (each lane holds 16 bytes x NCH of the
//     row), so 4 keys are processed per step.  All G query heads of the KV
//     head use each staged K/V row (grouped-query attention), with q held
//     in registers pre-multiplied by scale * log2(e).  The 8-lane dot
//     products are all-reduced with 3 xor shuffles.
//   * Each 8-lane group keeps its own online-softmax state (m, l, o) per
//     head and rescales lazily: only when a score exceeds the running
//     reference by more than 8 (log2 units) is the state rescaled, so the
//     weights stay below 2^8 and the result is unchanged in exact
//     arithmetic.  At the end of an item the 4 groups of a warp are merged
//     with shuffles and the 8 warps through shared memory, by the same
//     log-sum-exp rule, and the partial (or, with one chunk, the final
//     output and lse) is written.
//   * Every wait is bounded (kWaitLimitNs); on expiry the kernel records
//     TA_DEVERR_TIMEOUT, stops, and drains its own outstanding copies.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ta {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr float kRescaleLog2 = 8.0f;

enum : int { kFirst = 1, kLast = 2, kEnd = 4 };

struct TileDesc {
    int item;
    int j0;
    int n;
    int flags;
};

struct DecodeParams {
    const void *q, *k, *v;
    void *out;
    float *lse;
    int B, Hq, Hkv, S;
    float qscale;  // scale * log2(e)
    const int32_t *seqlens;
    int n_split, chunk, n_items;
    int final_out;    // 1: one chunk per item, write out/lse directly
    int32_t *status;  // [0] flags, [16] work-queue counter
    float *part_m, *part_l, *part_o;
};

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kPerChunk = 4;
    __device__ static void unpack(const uint4 &r, float *f)
    {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerChunk = 8;
    __device__ static void unpack(const uint4 &r, float *f)
    {
        f[0] = bf16_lo(r.x);
        f[1] = bf16_hi(r.x);
        f[2] = bf16_lo(r.y);
        f[3] = bf16_hi(r.y);
        f[4] = bf16_lo(r.z);
        f[5] = bf16_hi(r.z);
        f[6] = bf16_lo(r.w);
        f[7] = bf16_hi(r.w);
    }
};

__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

template <int D, int G, typename KV>
struct Cfg {
    static constexpr int RB = D * (int)sizeof(KV);  // bytes per K or V row
    static constexpr int NCH = RB / 128;            // 16-byte chunks per lane per row
    static constexpr int EPC = Elem<KV>::kPerChunk; // elements per chunk
    static constexpr int DPL = NCH * EPC;           // dims held by a lane
    static constexpr int KPW = 4096 / RB;           // keys per warp per stage
    static constexpr int TILE = kConsumerWarps * KPW;
    static constexpr int KV_OFF = TILE * RB;        // V tile offset inside a stage
    static constexpr int STAGE = 2 * TILE * RB;
    static constexpr int MERGE_FLOATS = kConsumerWarps * G * (D + 2);
    static constexpr size_t SMEM = (size_t)kStages * STAGE + (size_t)MERGE_FLOATS * 4 +
                                   (2 * kStages + 2) * 8 + kStages * sizeof(TileDesc) + 16;
    static_assert(NCH >= 1 && RB % 128 == 0, "row must be a multiple of 128 bytes");
    static_assert(KPW % 4 == 0, "a warp step covers 4 keys");
};

template <int D, int G, typename KV, typename OUT>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const DecodeParams p)
{
    using C = Cfg<D, G, KV>;
    extern __shared__ __align__(1024) unsigned char smem[];
    float *merge_o = reinterpret_cast<float *>(smem + kStages * C::STAGE);  // [W][G][D]
    float *merge_m = merge_o + kConsumerWarps * G * D;                       // [W][G]
    float *merge_l = merge_m + kConsumerWarps * G;                           // [W][G]
    uint64_t *bars = reinterpret_cast<uint64_t *>(merge_l + kConsumerWarps * G);
    uint64_t *full = bars;
    uint64_t *empty = bars + kStages;
    uint64_t *merge_in = bars + 2 * kStages;
    uint64_t *merge_out = merge_in + 1;
    TileDesc *desc = reinterpret_cast<TileDesc *>(bars + 2 * kStages + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(desc + kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(merge_in, kConsumerWarps);
        mbar_init(merge_out, kConsumerWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0)
            return;
        const uint64_t policy = l2_policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t used_mask = 0, parity_mask = 0;  // per stage: arrived on, and that phase's parity
        const size_t kv_head_stride = (size_t)p.S * D;
        bool ok = true;
        while (ok) {
            const int item = atomicAdd(&p.status[16], 1);
            if (item >= p.n_items) {
                if (item == p.n_items + (int)gridDim.x - 1)
                    atomicExch(&p.status[16], 0);  // last grab of the launch: reset the queue
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag))
                    break;
                desc[stage] = TileDesc{item, 0, 0, kEnd};
                mbar_arrive(&full[stage]);
                used_mask |= 1u << stage;
                parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
                break;
            }
            const int unit = item / p.n_split;
            const int split = item - unit * p.n_split;
            const int b = unit / p.Hkv;
            int L = p.S;
            if (p.seqlens) {
                L = p.seqlens[b];
                if (L < 0 || L > p.S) {
                    atomicOr(&p.status[0], TA_DEVERR_SEQLEN);
                    L = L < 0 ? 0 : p.S;
                }
            }
            const int c0 = split * p.chunk;
            const int c1 = min(c0 + p.chunk, L);
            const KV *kbase = static_cast<const KV *>(p.k) + (size_t)unit * kv_head_stride;
            const KV *vbase = static_cast<const KV *>(p.v) + (size_t)unit * kv_head_stride;
            int j0 = c0;
            int flags = kFirst;
            for (;;) {
                const int n = max(0, min(C::TILE, c1 - j0));
                const bool last = j0 + n >= c1;
                if (last)
                    flags |= kLast;
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                desc[stage] = TileDesc{item, j0, n, flags};
                unsigned char *dst = smem + stage * C::STAGE;
                if (n > 0) {
                    const uint32_t bytes = (uint32_t)n * C::RB;
                    mbar_arrive_expect_tx(&full[stage], 2 * bytes);
                    bulk_copy_g2s_hint(dst, kbase + (size_t)j0 * D, bytes, &full[stage], policy);
                    bulk_copy_g2s_hint(dst + C::KV_OFF, vbase + (size_t)j0 * D, bytes, &full[stage], policy);
                } else {
                    mbar_arrive(&full[stage]);
                }
                used_mask |= 1u << stage;
                parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (last)
                    break;
                j0 += n;
                flags = 0;
            }
        }
        // Drain: every copy this thread issued has landed before the CTA exits
        // (immediate on the normal path; bounded after an abort).
        int drain_abort = 0;
        for (int s = 0; s < kStages; ++s)
            if (used_mask & (1u << s))
                mbar_wait_bounded(&full[s], (parity_mask >> s) & 1u, &drain_abort);
        if (*abort_flag)
            atomicOr(&p.status[0], TA_DEVERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 3;  // key slot within a 4-key step
    const int t = lane & 7;   // lane within the 8-lane key group
    const int tid = threadIdx.x;
    constexpr unsigned kFull = 0xffffffffu;

    float qr[G][C::DPL];
    float o[G][C::DPL];
    float m_used[G], l[G];
    int stage = 0;
    uint32_t phase = 0;
    uint32_t merge_phase = 0;
    int b = 0, kvh = 0, split = 0;

    for (;;) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag))
            break;
        const TileDesc d = desc[stage];
        if (d.flags & kEnd)
            break;
        if (d.flags & kFirst) {
            const int unit = d.item / p.n_split;
            split = d.item - unit * p.n_split;
            b = unit / p.Hkv;
            kvh = unit - b * p.Hkv;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const KV *qrow = static_cast<const KV *>(p.q) + ((size_t)b * p.Hq + (size_t)kvh * G + h) * D;
#pragma unroll
                for (int i = 0; i < C::NCH; ++i) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + (t + 8 * i) * C::EPC);
                    float f[C::EPC];
                    Elem<KV>::unpack(raw, f);
#pragma unroll
                    for (int e = 0; e < C::EPC; ++e)
                        qr[h][i * C::EPC + e] = f[e] * p.qscale;
                }
                m_used[h] = -INFINITY;
                l[h] = 0.f;
#pragma unroll
                for (int e = 0; e < C::DPL; ++e)
                    o[h][e] = 0.f;
            }
        }

        const unsigned char *Ks = smem + stage * C::STAGE;
        const unsigned char *Vs = Ks + C::KV_OFF;
        const int kbeg = warp * C::KPW;
        const int kend = min(kbeg + C::KPW, d.n);
        for (int kk = kbeg; kk < kend; kk += 4) {
            const int key = kk + g;
            const bool valid = key < kend;
            float s[G];
#pragma unroll
            for (int h = 0; h < G; ++h)
                s[h] = 0.f;
            if (valid) {
#pragma unroll
                for (int i = 0; i < C::NCH; ++i) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(Ks + key * C::RB + (t + 8 * i) * 16);
                    float kf[C::EPC];
                    Elem<KV>::unpack(raw, kf);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < C::EPC; ++e)
                            s[h] = fmaf(qr[h][i * C::EPC + e], kf[e], s[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                s[h] += __shfl_xor_sync(kFull, s[h], 4);
                s[h] += __shfl_xor_sync(kFull, s[h], 2);
                s[h] += __shfl_xor_sync(kFull, s[h], 1);
            }
            if (valid) {
                float vf[C::DPL];
#pragma unroll
                for (int i = 0; i < C::NCH; ++i) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(Vs + key * C::RB + (t + 8 * i) * 16);
                    Elem<KV>::unpack(raw, vf + i * C::EPC);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    if (s[h] > m_used[h] + kRescaleLog2) {
                        const float a = fast_exp2(m_used[h] - s[h]);
                        l[h] *= a;
#pragma unroll
                        for (int e = 0; e < C::DPL; ++e)
                            o[h][e] *= a;
                        m_used[h] = s[h];
                    }
                    const float pw = fast_exp2(s[h] - m_used[h]);
                    l[h] += pw;
#pragma unroll
                    for (int e = 0; e < C::DPL; ++e)
                        o[h][e] = fmaf(pw, vf[e], o[h][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
        }
        if (!(d.flags & kLast))
            continue;

        // ---- end of item: merge the 4 key groups of this warp (xor 8, 16)
#pragma unroll
        for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float mo = __shfl_xor_sync(kFull, m_used[h], off);
                const float lo = __shfl_xor_sync(kFull, l[h], off);
                const float mn = fmaxf(m_used[h], mo);
                const float a_self = m_used[h] == -INFINITY ? 0.f : fast_exp2(m_used[h] - mn);
                const float a_oth = mo == -INFINITY ? 0.f : fast_exp2(mo - mn);
                l[h] = l[h] * a_self + lo * a_oth;
#pragma unroll
                for (int e = 0; e < C::DPL; ++e) {
                    const float oo = __shfl_xor_sync(kFull, o[h][e], off);
                    o[h][e] = o[h][e] * a_self + oo * a_oth;
                }
                m_used[h] = mn;
            }
        }
        // ---- merge the 8 warps through shared memory
        if (!mbar_wait_bounded(merge_out, merge_phase ^ 1, abort_flag))
            break;
        if (g == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int i = 0; i < C::NCH; ++i)
#pragma unroll
                    for (int e = 0; e < C::EPC; e += 4) {
                        float4 v4 = make_float4(o[h][i * C::EPC + e], o[h][i * C::EPC + e + 1],
                                                o[h][i * C::EPC + e + 2], o[h][i * C::EPC + e + 3]);
                        *reinterpret_cast<float4 *>(&merge_o[(warp * G + h) * D + (t + 8 * i) * C::EPC + e]) = v4;
                    }
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                merge_m[warp * G + h] = m_used[h];
                merge_l[warp * G + h] = l[h];
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(merge_in);
        if (!mbar_wait_bounded(merge_in, merge_phase, abort_flag))
            break;
        const bool final_out = p.final_out != 0;
        for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
            const int h = idx / D;
            const int dd = idx - h * D;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w)
                mx = fmaxf(mx, merge_m[w * G + h]);
            float ls = 0.f, os = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = merge_m[w * G + h];
                const float a = mw == -INFINITY ? 0.f : fast_exp2(mw - mx);
                ls = fmaf(a, merge_l[w * G + h], ls);
                os = fmaf(a, merge_o[(w * G + h) * D + dd], os);
            }
            const size_t row = (size_t)b * p.Hq + (size_t)kvh * G + h;
            if (final_out) {
                const float inv = ls > 0.f ? 1.0f / ls : 0.f;
                store_out(static_cast<OUT *>(p.out) + row * D + dd, os * inv);
                if (dd == 0 && p.lse)
                    p.lse[row] = ls > 0.f ? (mx + log2f(ls)) * kLn2 : -INFINITY;
            } else {
                const size_t pi = row * p.n_split + split;
                p.part_o[pi * D + dd] = os;
                if (dd == 0) {
                    p.part_m[pi] = mx == -INFINITY ? -INFINITY : mx * kLn2;
                    p.part_l[pi] = ls;
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(merge_out);
        merge_phase ^= 1;
    }
}

template <int D, int G, typename KV, typename OUT>
cudaError_t launch_typed(const DecodeLaunch &a, const DecodeParams &p)
{
    using C = Cfg<D, G, KV>;
    auto kern = decode_split_kernel<D, G, KV, OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess)
        return e;
    kern<<<a.plan.grid, kThreads, C::SMEM, a.stream>>>(p);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t dispatch_types(const DecodeLaunch &a, const DecodeParams &p)
{
    if (a.in_dtype == TA_BF16) {
        if (a.out_dtype == TA_BF16)
            return launch_typed<D, G, __nv_bfloat16, __nv_bfloat16>(a, p);
        return launch_typed<D, G, __nv_bfloat16, float>(a, p);
    }
    return launch_typed<D, G, float, float>(a, p);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch &a)
{
    DecodeParams p;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.out = a.out;
    p.lse = a.lse;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.S = a.S;
    p.qscale = a.scale * kLog2e;
    p.seqlens = a.seqlens;
    p.n_split = a.plan.n_split;
    p.chunk = a.plan.chunk;
    p.n_items = a.B * a.Hkv * a.plan.n_split;
    p.final_out = (a.plan.n_split == 1 && !a.force_partials) ? 1 : 0;
    p.status = a.status;
    p.part_m = a.part_m;
    p.part_l = a.part_l;
    p.part_o = a.part_o;
    const int G = a.Hq / a.Hkv;
    if (a.D == 128) {
        switch (G) {
        case 1: return dispatch_types<128, 1>(a, p);
        case 2: return dispatch_types<128, 2>(a, p);
        case 4: return dispatch_types<128, 4>(a, p);
        }
    } else if (a.D == 64) {
        switch (G) {
        case 1: return dispatch_types<64, 1>(a, p);
        case 2: return dispatch_types<64, 2>(a, p);
        case 4: return dispatch_types<64, 4>(a, p);
        case 8: return dispatch_types<64, 8>(a, p);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace ta
