// decode.cu -- split-KV exact decode: one partial (m, l, o) per KV chunk,
// and the log-sum-exp merge of a sequence's partials in the same launch.
//
// What is computed (Attention glossary, jisaku.com/glossary/attention,
// "basic concepts and operating principle"): for the query of each
// (sequence b, query head h), scores s_j = scale * <q, k_j> over the
// attended keys, softmax weights, and the weighted mean of the values.
// The keys are cut into chunks; each chunk yields the partial
//   m = a reference point (>= max_j s_j - 8 ln 2), l = sum_j e^(s_j - m),
//   o = sum_j e^(s_j - m) v_j,
// and partials are merged by the log-sum-exp rule (Tree Attention
// explainer, aibr.jp/archives/143699, sections 1 and 3):
//   m* = max_i m_i, l* = sum_i l_i e^(m_i - m*), o* = sum_i o_i e^(m_i - m*),
//   out = o* / l*, lse = m* + ln l*.
// Decode reads the whole KV cache once per token and is bound by HBM
// bandwidth (Attention glossary, "the memory bandwidth and VRAM wall"), so
// the kernel streams K and V at full bandwidth and keeps the arithmetic
// (about 4 FLOP per byte at G = 4) under it.
//
// Kernel layout (one persistent CTA per SM, 13 warps):
//   * warp 12, lane 0 is the producer.  It pulls work items
//     (sequence, KV head, chunk) from a device-wide queue and stages the
//     chunk's K and V rows into shared memory, kTile keys at a time, with
//     one-dimensional bulk async copies into a ring of stages guarded by
//     mbarriers.  Each stage carries a descriptor (item, first key, key
//     count, first/last flags) so the consumers need no schedule.
//   * warps 0-11 consume; warp w owns keys [8w, 8w + 8) of every tile, in
//     two steps of 4 keys.
//       scores: 8 lanes share a key, each holding 16 bytes x NCH of the
//         row; the G query heads of the KV head (grouped-query attention)
//         use each staged row, with q in registers pre-multiplied by
//         scale * log2(e), products taken two lanes of fp32 at a time
//         (packed f32x2 FMA) and the 8-lane sums closed by 3 xor shuffles.
//       online softmax: one running reference m per head for the whole
//         warp, raised lazily (only when a score exceeds it by more than
//         2^8, with a warp vote), so the weights stay below 2^8 and the
//         result is exact up to rounding.
//       PV: the weights go through shared memory, and every lane owns
//         D/32 output dimensions of every head, accumulated with packed
//         f32x2 FMAs over the warp's keys.
//     At the end of an item the 12 warps are merged through shared memory
//     by the log-sum-exp rule and the item's partial (or, with one chunk,
//     the final output and lse) is written.
//   * Fused merge: the CTA that finishes the last chunk of a (sequence,
//     KV head) -- found with an atomic ticket, never by waiting -- merges
//     that unit's partials and writes out and lse, so a decode is one
//     launch.  (Larger split counts merge in a separate kernel.)
//   * Every wait is bounded (kWaitLimitNs); on expiry the kernel records
//     TA_DEVERR_TIMEOUT, stops, and drains its own outstanding copies.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ta {
namespace {

constexpr int kConsumerWarps = 12;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kKeysPerWarp = 8;                        // per stage
constexpr int kTile = kConsumerWarps * kKeysPerWarp;  // keys per stage
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned kFull = 0xffffffffu;

static_assert(kTile == kDecodeTileKeys, "scheduler and kernel disagree on the tile");

enum : int { kFirst = 1, kLast = 2, kEnd = 4 };
enum : int { kModeFinal = 0, kModePartials = 1, kModeFused = 2 };

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
    int mode;
    int32_t *status;    // [0] flags, [16] work-queue counter
    int32_t *counters;  // [B * Hkv] finished chunks per unit (fused mode)
    float *part_m, *part_l, *part_o;
};

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kPerChunk = 4;
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerChunk = 8;
};

__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// 16 bytes of K or V as floats.
__device__ __forceinline__ void unpack16(const uint4 &r, float (&f)[4], float *)
{
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
}
__device__ __forceinline__ void unpack16(const uint4 &r, float (&f)[8], __nv_bfloat16 *)
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

template <int D, int G, typename KV>
struct Cfg {
    static constexpr int RB = D * (int)sizeof(KV);  // bytes per K or V row
    static constexpr int NCH = RB / 128;            // 16-byte chunks per lane per row (8 lanes per key)
    static constexpr int EPC = Elem<KV>::kPerChunk; // elements per chunk
    static constexpr int QPL = NCH * EPC;           // q elements held by a lane per head
    static constexpr int DPL = D / 32;              // output dims owned by a lane (PV)
    static constexpr int VB = DPL * (int)sizeof(KV);// V bytes read by a lane per key
    static constexpr int KV_OFF = kTile * RB;       // V tile offset inside a stage
    static constexpr int STAGE = 2 * kTile * RB;
    static constexpr int STAGES = (196608 / STAGE) > 6 ? 6 : (196608 / STAGE);
    static constexpr int MERGE_FLOATS = kConsumerWarps * G * (D + 2);
    static constexpr int PBUF_FLOATS = kConsumerWarps * 2 * 4 * G;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE + (size_t)(MERGE_FLOATS + PBUF_FLOATS) * 4 +
                                   (2 * STAGES + 4) * 8 + STAGES * sizeof(TileDesc) + 16;
    static_assert(NCH >= 1 && RB % 128 == 0, "row must be a multiple of 128 bytes");
    static_assert(STAGES >= 2, "need at least two stages");
    static_assert(DPL % 2 == 0, "lanes own an even number of output dims");
};

template <int D, int G, typename KV, typename OUT>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const DecodeParams p)
{
    using C = Cfg<D, G, KV>;
    extern __shared__ __align__(1024) unsigned char smem[];
    float *merge_o = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE);  // [W][G][D]
    float *merge_m = merge_o + kConsumerWarps * G * D;                         // [W][G]
    float *merge_l = merge_m + kConsumerWarps * G;                             // [W][G]
    float *pbuf = merge_l + kConsumerWarps * G;                                // [W][2][4][G]
    uint64_t *bars = reinterpret_cast<uint64_t *>(pbuf + C::PBUF_FLOATS);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::STAGES;
    uint64_t *merge_in = bars + 2 * C::STAGES;
    uint64_t *merge_out = merge_in + 1;
    uint64_t *written = merge_in + 2;  // consumers' partial stores done (fused mode)
    uint64_t *ticket = merge_in + 3;   // the ticket's outcome is in *ticket_flag
    TileDesc *desc = reinterpret_cast<TileDesc *>(bars + 2 * C::STAGES + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(desc + C::STAGES);
    volatile int *ticket_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(merge_in, kConsumerWarps);
        mbar_init(merge_out, kConsumerWarps);
        mbar_init(written, kConsumerThreads);
        mbar_init(ticket, 1);
        *abort_flag = 0;
        *ticket_flag = 0;
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
        uint32_t used_mask = 0, parity_mask = 0;  // per stage: armed, and that phase's parity
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
                const int n = max(0, min(kTile, c1 - j0));
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
                if (++stage == C::STAGES) {
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
        for (int s = 0; s < C::STAGES; ++s)
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

    float qr[G][C::QPL];       // q * scale * log2(e), this lane's slice
    float2 o[G][C::DPL / 2];   // this lane's output dims, unnormalised
    float m_run[G], l[G];      // warp-uniform reference; this lane group's sum
    int stage = 0;
    uint32_t phase = 0;
    uint32_t merge_phase = 0, ticket_phase = 0;
    int b = 0, kvh = 0, split = 0, unit = 0;
    int pslot = 0;
    float *my_pbuf = pbuf + warp * (2 * 4 * G);

    for (;;) {
        bool ok = mbar_wait_bounded(&full[stage], phase, abort_flag);
        if (!__all_sync(kFull, ok))
            break;
        const TileDesc d = desc[stage];
        if (d.flags & kEnd)
            break;
        if (d.flags & kFirst) {
            unit = d.item / p.n_split;
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
                    unpack16(raw, f, (KV *)nullptr);
#pragma unroll
                    for (int e = 0; e < C::EPC; ++e)
                        qr[h][i * C::EPC + e] = f[e] * p.qscale;
                }
                m_run[h] = -INFINITY;
                l[h] = 0.f;
#pragma unroll
                for (int e = 0; e < C::DPL / 2; ++e)
                    o[h][e] = make_float2(0.f, 0.f);
            }
        }

        const unsigned char *Ks = smem + stage * C::STAGE;
        const unsigned char *Vs = Ks + C::KV_OFF;
        const int kbeg = warp * kKeysPerWarp;
#pragma unroll
        for (int st4 = 0; st4 < kKeysPerWarp; st4 += 4) {
            if (kbeg + st4 >= d.n)
                break;  // warp-uniform
            const int key = kbeg + st4 + g;
            const bool valid = key < d.n;
            // ---- scores of this lane group's key for the G heads
            float2 acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h)
                acc[h] = make_float2(0.f, 0.f);
            if (valid) {
#pragma unroll
                for (int i = 0; i < C::NCH; ++i) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(Ks + key * C::RB + (t + 8 * i) * 16);
                    float kf[C::EPC];
                    unpack16(raw, kf, (KV *)nullptr);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < C::EPC; e += 2)
                            acc[h] = __ffma2_rn(make_float2(qr[h][i * C::EPC + e], qr[h][i * C::EPC + e + 1]),
                                                make_float2(kf[e], kf[e + 1]), acc[h]);
                }
            }
            float s[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float x = acc[h].x + acc[h].y;
                x += __shfl_xor_sync(kFull, x, 4);
                x += __shfl_xor_sync(kFull, x, 2);
                x += __shfl_xor_sync(kFull, x, 1);
                s[h] = valid ? x : -INFINITY;
            }
            // ---- lazy, warp-uniform rescale of the running reference
            bool need = false;
#pragma unroll
            for (int h = 0; h < G; ++h)
                need |= s[h] > m_run[h] + kRescaleLog2;
            if (__any_sync(kFull, need)) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float mx = s[h];
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                    if (mx > m_run[h] + kRescaleLog2) {
                        const float a = m_run[h] == -INFINITY ? 0.f : fast_exp2(m_run[h] - mx);
                        l[h] *= a;
#pragma unroll
                        for (int e = 0; e < C::DPL / 2; ++e)
                            o[h][e] = make_float2(o[h][e].x * a, o[h][e].y * a);
                        m_run[h] = mx;
                    }
                }
            }
            float pw[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                pw[h] = valid ? fast_exp2(s[h] - m_run[h]) : 0.f;
                l[h] += pw[h];
            }
            // ---- PV: the 4 keys' weights through shared memory, lanes own dims
            float *slot = my_pbuf + pslot * (4 * G);
            if (t == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    slot[g * G + h] = pw[h];
            }
            __syncwarp();
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
                const int key2 = kbeg + st4 + gg;
                if (key2 >= d.n)
                    break;  // warp-uniform
                float vf[C::DPL];
                const unsigned char *vrow = Vs + key2 * C::RB + lane * C::VB;
                if constexpr (sizeof(KV) == 2) {
                    if constexpr (C::DPL == 4) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(vrow);
                        vf[0] = bf16_lo(w.x);
                        vf[1] = bf16_hi(w.x);
                        vf[2] = bf16_lo(w.y);
                        vf[3] = bf16_hi(w.y);
                    } else {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(vrow);
                        vf[0] = bf16_lo(w);
                        vf[1] = bf16_hi(w);
                    }
                } else {
                    if constexpr (C::DPL == 4) {
                        const float4 w = *reinterpret_cast<const float4 *>(vrow);
                        vf[0] = w.x;
                        vf[1] = w.y;
                        vf[2] = w.z;
                        vf[3] = w.w;
                    } else {
                        const float2 w = *reinterpret_cast<const float2 *>(vrow);
                        vf[0] = w.x;
                        vf[1] = w.y;
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pk = slot[gg * G + h];
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e)
                        o[h][e] = __ffma2_rn(make_float2(pk, pk), make_float2(vf[2 * e], vf[2 * e + 1]), o[h][e]);
                }
            }
            pslot ^= 1;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);
        if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
        }
        if (!(d.flags & kLast))
            continue;

        // ---- end of item: the lane groups' sums, then merge the 12 warps
#pragma unroll
        for (int h = 0; h < G; ++h) {
            l[h] += __shfl_xor_sync(kFull, l[h], 8);
            l[h] += __shfl_xor_sync(kFull, l[h], 16);
        }
        ok = mbar_wait_bounded(merge_out, merge_phase ^ 1, abort_flag);
        if (!__all_sync(kFull, ok))
            break;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = merge_o + (warp * G + h) * D + lane * C::DPL;
#pragma unroll
            for (int e = 0; e < C::DPL / 2; ++e)
                *reinterpret_cast<float2 *>(dst + 2 * e) = o[h][e];
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                merge_m[warp * G + h] = m_run[h];
                merge_l[warp * G + h] = l[h];
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(merge_in);
        ok = mbar_wait_bounded(merge_in, merge_phase, abort_flag);
        if (!__all_sync(kFull, ok))
            break;
        const size_t row0 = (size_t)b * p.Hq + (size_t)kvh * G;
        for (int idx = tid; idx < G * D; idx += kConsumerThreads) {
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
            const size_t row = row0 + h;
            if (p.mode == kModeFinal) {
                const float inv = ls > 0.f ? 1.0f / ls : 0.f;
                store_out(static_cast<OUT *>(p.out) + row * D + dd, os * inv);
                if (dd == 0 && p.lse)
                    p.lse[row] = ls > 0.f ? (mx + fast_log2(ls)) * kLn2 : -INFINITY;
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
        if (p.mode != kModeFused)
            continue;

        // ---- fused merge: the CTA that writes a unit's last partial merges it
        __threadfence();
        mbar_arrive(written);
        if (tid == 0) {
            int last = 0;
            if (mbar_wait_bounded(written, ticket_phase, abort_flag)) {
                const int done = atomicAdd(&p.counters[unit], 1);
                if (done == p.n_split - 1) {
                    last = 1;
                    p.counters[unit] = 0;  // ready for the next launch
                    __threadfence();
                }
            }
            *ticket_flag = last;
            mbar_arrive(ticket);
        }
        ok = mbar_wait_bounded(ticket, ticket_phase, abort_flag);
        ticket_phase ^= 1;
        if (!__all_sync(kFull, ok))
            break;
        if (!*ticket_flag)
            continue;
        const int ns = p.n_split;
        for (int idx = tid; idx < G * D; idx += kConsumerThreads) {
            const int h = idx / D;
            const int dd = idx - h * D;
            const size_t row = row0 + h;
            const float *pm = p.part_m + row * ns;
            const float *pl = p.part_l + row * ns;
            const float *po = p.part_o + row * ns * D + dd;
            float mx = -INFINITY;
            for (int n = 0; n < ns; ++n)
                mx = fmaxf(mx, __ldcg(pm + n));
            float ls = 0.f, os = 0.f;
            if (mx != -INFINITY) {
                for (int n = 0; n < ns; ++n) {
                    const float mn = __ldcg(pm + n);
                    const float a = mn == -INFINITY ? 0.f : fast_exp2((mn - mx) * kLog2e);
                    ls = fmaf(a, __ldcg(pl + n), ls);
                    os = fmaf(a, __ldcg(po + (size_t)n * D), os);
                }
            }
            const float inv = ls > 0.f ? 1.0f / ls : 0.f;
            store_out(static_cast<OUT *>(p.out) + row * D + dd, os * inv);
            if (dd == 0 && p.lse)
                p.lse[row] = ls > 0.f ? mx + fast_log2(ls) * kLn2 : -INFINITY;
        }
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
    if (a.force_partials)
        p.mode = kModePartials;
    else if (a.plan.n_split == 1)
        p.mode = kModeFinal;
    else
        p.mode = decode_merges_itself(a.plan.n_split, a.B * a.Hkv) ? kModeFused : kModePartials;
    p.status = a.status;
    p.counters = a.counters;
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
