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
// Kernel layout (one persistent CTA per SM, 16 warps):
//   * warp 15 is the producer (lane 0 decides, the 32 lanes share the
//     copies of a tile).  It pulls work items
//     (sequence, KV head, chunk) from a device-wide queue and stages the
//     chunk's K and V rows into shared memory, a tile at a time, with
//     one-dimensional bulk async copies into a ring of stages guarded by
//     mbarriers.  Each stage carries a descriptor (item, first key, key
//     count, first/last flags) so the consumers need no schedule.
//   * warps 0-14 consume; warp w owns keys [KPW w, KPW w + KPW) of every
//     tile (KPW = 8 keys, two steps of 4; 4 for 512-byte rows), so a tile
//     is 120 (or 60) keys.
//       scores: 8 lanes share a key, each holding 16 bytes x NCH of the
//         row; the G query heads of the KV head (grouped-query attention)
//         use each staged row.  For bf16 K the products use the
//         mixed-precision FMA (bf16 x bf16 + fp32), so neither q nor K is
//         widened; the 8 lanes' partial sums of the G heads are reduced by
//         a reduce-scatter over 3 xor shuffles (G/2 + G/4 + ... exchanges),
//         after which each lane holds one head's full score.
//       online softmax: one running reference m per head for the whole
//         warp, raised lazily (only when a score exceeds it by more than
//         2^8, with a warp vote), so the weights stay below 2^8 and the
//         result is exact up to rounding.  Each lane takes one exp.
//       PV: the weights go through shared memory (one vector load per key),
//         and every lane owns D/32 output dimensions of every head,
//         accumulated in fp32 over the warp's keys.
//     At the end of an item the 15 warps are merged through shared memory
//     by the log-sum-exp rule and the item's partial (or, with one chunk,
//     the final output and lse) is written.
//   * Fused merge: the CTA that finishes the last chunk of a (sequence,
//     KV head) -- found with an atomic ticket, never by waiting -- merges
//     that unit's partials and writes out and lse, so a decode is one
//     launch.  (Larger split counts merge in a separate kernel.)
//   * Every wait is bounded (kWaitLimitNs); on expiry the kernel records
//     TA_DEVERR_TIMEOUT, stops, and drains its own outstanding copies.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace ta {
namespace {

constexpr int kConsumerWarps = 15;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // 16 warps: 128 registers a thread
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned kFull = 0xffffffffu;


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
    ChunkMap cm;  // work item -> (unit, chunk) and the chunk's keys
    int mode;
    int32_t *status;    // [0] flags, [16] work-queue counter
    int32_t *counters;  // [B * Hkv] finished chunks per unit (fused mode)
    float *part_m, *part_l, *part_o;
    uint64_t wait_ns;   // time limit of a pipeline wait
    int test_stall;     // test hook: the producer first waits on a barrier nothing ends
    // Paged KV cache (block_table != nullptr): k, v are [num_pages, Hkv,
    // page_size, D] and key j of sequence b lives in page
    // block_table[b * pages_per_seq + j / page_size] at row j % page_size.
    const int32_t *block_table;
    int page_size, pages_per_seq, num_pages;
    // pi-Attention key set (pi_period > 0): the query at i = L - 1 attends
    // the window [max(0, i - pi_window), i] and the keys i - m * pi_period
    // (m >= 1) before it; the chunks cut the ascending list of those keys.
    int pi_window, pi_period;
    // fp8 K/V: per (sequence, KV head) dequantisation factors, or nullptr (1)
    const float *k_scale, *v_scale;
    // pi_tma: K and V of each (sequence, KV head) seen as rows of
    // pi_period keys, [B*Hkv, ceil(S / period), period * D] with a box of
    // D x TILE: the box at x = r * D, y = m gathers keys r + (m + t) * period,
    // t < TILE, in one copy.
    int pi_tma;
    CUtensorMap pi_kmap, pi_vmap;
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
template <>
struct Elem<__nv_fp8_e4m3> {
    static constexpr int kPerChunk = 16;
};

__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// acc += a.lo * b.lo + a.hi * b.hi for packed bf16 pairs a, b: the
// mixed-precision FMA takes bf16 operands and an fp32 accumulator, so
// neither operand is widened (each step is exactly fmaf of the widened
// values).
__device__ __forceinline__ void fma_bf16(float &acc, uint32_t a, uint32_t b)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
}

// Where the scores of a step land after the 8-lane reduce-scatter.  A lane
// group has NV = KPG * G (key, head) dot products; lane t ends with NVL of
// them, score index (t / RED) * NVL + j, key kk = index / G, head
// h = index % G, and RED lanes hold each one when NV < 8.
template <int KPG_, int G>
struct Lay {
    static constexpr int KPG = KPG_;
    static constexpr int NV = KPG * G;
    static constexpr int NVL = NV >= 8 ? NV / 8 : 1;
    static constexpr int RED = NV >= 8 ? 1 : 8 / NV;
    __host__ __device__ static constexpr int idx_of(int t, int j) { return (t / RED) * NVL + j; }
    __host__ __device__ static constexpr int kk_of(int t, int j) { return idx_of(t, j) / G; }
    __host__ __device__ static constexpr int h_of(int t, int j) { return idx_of(t, j) % G; }
    // Whether xor-ing the lane index with `mask` keeps the head of every
    // value j (masks 8 and 16 only change the group).
    __host__ __device__ static constexpr bool preserves_head(int mask)
    {
        if (mask >= 8)
            return true;
        for (int tt = 0; tt < 8; ++tt)
            for (int j = 0; j < NVL; ++j)
                if (h_of(tt, j) != h_of(tt ^ mask, j))
                    return false;
        return true;
    }
    // A lane of group 0 that holds head h (as its value j_of_head(h), key 0).
    __host__ __device__ static constexpr int lane_of_head(int h)
    {
        for (int tt = 0; tt < 8; ++tt)
            for (int j = 0; j < NVL; ++j)
                if (h_of(tt, j) == h && kk_of(tt, j) == 0 && tt % RED == 0)
                    return tt;
        return 0;
    }
    __host__ __device__ static constexpr int j_of_head(int h)
    {
        for (int tt = 0; tt < 8; ++tt)
            for (int j = 0; j < NVL; ++j)
                if (h_of(tt, j) == h && kk_of(tt, j) == 0 && tt % RED == 0)
                    return j;
        return 0;
    }
};

// acc += sum of the 4 products of two packed f16 pairs a, b (fp32 accumulator).
__device__ __forceinline__ void fma_f16(float &acc, uint32_t a, uint32_t b)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
}

// Two e4m3 values (low byte first) to a packed f16 pair (exact: e4m3 is a
// subset of f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
    return r;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w)
{
    float2 r;
    asm("{\n\t.reg .f16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\t"
        "cvt.f32.f16 %1, hi;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(w));
    return r;
}

// The G weights of one key from shared memory (one vector load).
template <int G>
__device__ __forceinline__ void load_weights(const float *src, float (&pk)[G])
{
    if constexpr (G == 1) {
        pk[0] = *src;
    } else if constexpr (G == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(src);
        pk[0] = x.x;
        pk[1] = x.y;
    } else {
#pragma unroll
        for (int i = 0; i < G; i += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + i);
            pk[i] = x.x;
            pk[i + 1] = x.y;
            pk[i + 2] = x.z;
            pk[i + 3] = x.w;
        }
    }
}

// The DPL consecutive values of a V row that this lane owns, as floats.
template <int DPL>
__device__ __forceinline__ void load_v_slice(const unsigned char *src, float (&vf)[DPL], __nv_bfloat16 *)
{
    if constexpr (DPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        vf[0] = bf16_lo(w.x);
        vf[1] = bf16_hi(w.x);
        vf[2] = bf16_lo(w.y);
        vf[3] = bf16_hi(w.y);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
        vf[0] = bf16_lo(w);
        vf[1] = bf16_hi(w);
    }
}
template <int DPL>
__device__ __forceinline__ void load_v_slice(const unsigned char *src, float (&vf)[DPL], __nv_fp8_e4m3 *)
{
    static_assert(DPL == 4, "fp8 rows are 128 bytes: 4 dims a lane");
    const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
    const float2 a = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)(w & 0xffffu)));
    const float2 b = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)(w >> 16)));
    vf[0] = a.x;
    vf[1] = a.y;
    vf[2] = b.x;
    vf[3] = b.y;
}
template <int DPL>
__device__ __forceinline__ void load_v_slice(const unsigned char *src, float (&vf)[DPL], float *)
{
    if constexpr (DPL == 4) {
        const float4 w = *reinterpret_cast<const float4 *>(src);
        vf[0] = w.x;
        vf[1] = w.y;
        vf[2] = w.z;
        vf[3] = w.w;
    } else {
        const float2 w = *reinterpret_cast<const float2 *>(src);
        vf[0] = w.x;
        vf[1] = w.y;
    }
}

template <int D, int G, typename KV>
struct Cfg {
    static constexpr int RB = D * (int)sizeof(KV);  // bytes per K or V row
    static constexpr int NCH = RB / 128;            // 16-byte chunks per lane per row (8 lanes per key)
    static constexpr int EPC = Elem<KV>::kPerChunk; // elements per chunk
    // 32-bit q words a lane holds per head: bf16 pairs or fp32 values as
    // loaded; for fp8 K/V, f16 pairs (16 dims per chunk)
    static constexpr int QPL_W = NCH * (sizeof(KV) == 1 ? 8 : 4);
    static constexpr int DPL = D / 32;              // output dims owned by a lane (PV)
    static constexpr int VB = DPL * (int)sizeof(KV);// V bytes read by a lane per key
    static constexpr int PB = (G * (DPL + 1) > 24) ? 2 : 4;  // keys per PV load batch (register budget)
    static constexpr int KPW = RB > 256 ? 4 : 8;    // keys per consumer warp per stage
    static constexpr int TILE = kConsumerWarps * KPW;  // keys per stage
    static constexpr int KV_OFF = TILE * RB;        // V tile offset inside a stage
    static constexpr int STAGE = 2 * TILE * RB;
    static constexpr int STAGES = (196608 / STAGE) > 6 ? 6 : (196608 / STAGE);
    static constexpr int MERGE_FLOATS = kConsumerWarps * G * (D + 2);
    static constexpr int PBUF_FLOATS = kConsumerWarps * KPW * G;
    static constexpr int FM_FLOATS = 2 * G * kFusedMergeMaxSplits;  // partial m, l of one unit
    static constexpr size_t SMEM = (size_t)STAGES * STAGE + (size_t)(MERGE_FLOATS + PBUF_FLOATS + FM_FLOATS) * 4 +
                                   (2 * STAGES + 5) * 8 + STAGES * sizeof(TileDesc) + 16 + 1024;
    static_assert(NCH >= 1 && RB % 128 == 0, "row must be a multiple of 128 bytes");
    static_assert(STAGES >= 2, "need at least two stages");
    static_assert(kDecodeTileKeysCC % TILE == 0, "chunks of the CUDA-core shapes are whole tiles");
    static_assert(DPL % 2 == 0, "lanes own an even number of output dims");
};

template <int D, int G, typename KV, typename OUT>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const __grid_constant__ DecodeParams p)
{
    using C = Cfg<D, G, KV>;
    // stage buffers start on a 1024-byte boundary (tensor copies need 128)
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    float *merge_o = reinterpret_cast<float *>(smem + C::STAGES * C::STAGE);  // [W][G][D]
    float *merge_m = merge_o + kConsumerWarps * G * D;                         // [W][G]
    float *merge_l = merge_m + kConsumerWarps * G;                             // [W][G]
    float *pbuf = merge_l + kConsumerWarps * G;                                // [W][KPW][G]
    float *fm_m = pbuf + C::PBUF_FLOATS;                                       // [G][n_split]
    float *fm_l = fm_m + G * kFusedMergeMaxSplits;                             // [G][n_split]
    uint64_t *bars = reinterpret_cast<uint64_t *>(fm_l + G * kFusedMergeMaxSplits);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::STAGES;
    uint64_t *merge_in = bars + 2 * C::STAGES;
    uint64_t *merge_out = merge_in + 1;
    uint64_t *written = merge_in + 2;  // consumers' partial stores done (fused mode)
    uint64_t *ticket = merge_in + 3;   // the ticket's outcome is in *ticket_flag
    uint64_t *fm_ready = merge_in + 4; // fm_m / fm_l staged (fused merge)
    TileDesc *desc = reinterpret_cast<TileDesc *>(bars + 2 * C::STAGES + 5);
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
        mbar_init(fm_ready, kConsumerThreads);
        *abort_flag = 0;
        *ticket_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        // Lane 0 takes the decisions (work queue, ring waits, expected bytes,
        // descriptors); every lane computes the same schedule and the 32
        // lanes share the bulk copies of a tile (gathered rows of the
        // pi-Attention set or a paged cache need one copy per run of rows).
        const bool leader = lane == 0;
        const uint64_t policy = l2_policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t used_mask = 0, parity_mask = 0;  // per stage: armed, and that phase's parity
        const size_t kv_head_stride = (size_t)p.S * D;
        bool ok = true;
        if (p.test_stall) {
            // test hook: a wait that nothing ends (phase 0 of a barrier only
            // this warp arms), so the launch's time limit runs out
            int w = 1;
            if (leader)
                w = mbar_wait_bounded(&full[0], 0, abort_flag, p.wait_ns);
            ok = __shfl_sync(kFull, w, 0) != 0;
        }
        // A CTA's first item is its block index; later ones come from the
        // device-wide queue, which counts the grabs after the first (the
        // last grab, item n_items + gridDim.x - 1, resets it).
        bool first_grab = true;
        while (ok) {
            int item = 0;
            if (leader)
                item = first_grab ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&p.status[16], 1);
            first_grab = false;
            item = __shfl_sync(kFull, item, 0);
            if (item >= p.n_items) {
                bool w = true;
                if (leader) {
                    if (item == p.n_items + (int)gridDim.x - 1)
                        atomicExch(&p.status[16], 0);  // last grab of the launch: reset the queue
                    w = mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.wait_ns);
                    if (w) {
                        desc[stage] = TileDesc{item, 0, 0, kEnd};
                        mbar_arrive(&full[stage]);
                    }
                }
                if (__shfl_sync(kFull, w, 0)) {
                    used_mask |= 1u << stage;
                    parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
                }
                break;
            }
            const int unit = p.cm.unit_of(item);
            const int split = p.cm.split_of(item);
            const int b = unit / p.Hkv;
            int L = p.S;
            if (p.seqlens) {
                L = p.seqlens[b];
                if (L < 0 || L > p.S) {
                    if (leader)
                        atomicOr(&p.status[0], TA_DEVERR_SEQLEN);
                    L = L < 0 ? 0 : p.S;
                }
            }
            // the keys this sequence attends, as an ascending list of N
            // positions: n_skip periodic keys r, r + pi, ... then the window
            int N = L, w0 = 0, r0 = 0, n_skip = 0;
            if (p.pi_period > 0 && L > 0) {
                const int i = L - 1;
                w0 = max(0, i - p.pi_window);
                r0 = i % p.pi_period;
                n_skip = w0 > r0 ? (w0 - 1 - r0) / p.pi_period + 1 : 0;
                N = n_skip + (i - w0 + 1);
            }
            const int c0 = p.cm.start_of(split);
            const int c1 = min(c0 + p.cm.len_of(split), N);
            const KV *kbase = static_cast<const KV *>(p.k) + (size_t)unit * kv_head_stride;
            const KV *vbase = static_cast<const KV *>(p.v) + (size_t)unit * kv_head_stride;
            int j0 = c0;
            int flags = kFirst;
            for (;;) {
                const int n = max(0, min(C::TILE, c1 - j0));
                const bool last = j0 + n >= c1;
                if (last)
                    flags |= kLast;
                bool w = true;
                if (leader) {
                    w = mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.wait_ns);
                    if (w) {
                        desc[stage] = TileDesc{item, j0, n, flags};
                        if (n > 0)
                            mbar_arrive_expect_tx(&full[stage], 2 * (uint32_t)n * C::RB);
                        else
                            mbar_arrive(&full[stage]);
                    }
                }
                if (!__shfl_sync(kFull, w, 0)) {
                    ok = false;
                    break;
                }
                unsigned char *dst = smem + stage * C::STAGE;
                if (n > 0 && p.pi_period > 0) {
                    // periodic keys one row each (one run when the period is 1),
                    // then the window as one contiguous run
                    const int skip_end = min(j0 + n, n_skip);
                    if (p.pi_tma && n == C::TILE && skip_end == j0 + n) {
                        // a whole tile of periodic keys: one strided box each
                        if (leader) {
                            tc::tma_load_3d(dst, &p.pi_kmap, r0 * D, j0, unit, &full[stage]);
                            tc::tma_load_3d(dst + C::KV_OFF, &p.pi_vmap, r0 * D, j0, unit, &full[stage]);
                        }
                    } else if (p.pi_period == 1) {
                        if (leader && j0 < skip_end) {
                            const uint32_t bytes = (uint32_t)(skip_end - j0) * C::RB;
                            bulk_copy_g2s_hint(dst, kbase + (size_t)(r0 + j0) * D, bytes, &full[stage], policy);
                            bulk_copy_g2s_hint(dst + C::KV_OFF, vbase + (size_t)(r0 + j0) * D, bytes, &full[stage],
                                               policy);
                        }
                    } else {
                        for (int pos = j0 + lane; pos < skip_end; pos += 32) {  // one row per lane
                            const size_t key = (size_t)r0 + (size_t)pos * p.pi_period;
                            const uint32_t so = (uint32_t)(pos - j0) * C::RB;
                            bulk_copy_g2s_hint(dst + so, kbase + key * D, C::RB, &full[stage], policy);
                            bulk_copy_g2s_hint(dst + C::KV_OFF + so, vbase + key * D, C::RB, &full[stage], policy);
                        }
                    }
                    const int pos = max(j0, skip_end);
                    if (leader && pos < j0 + n) {
                        const size_t key = (size_t)w0 + (size_t)(pos - n_skip);
                        const uint32_t so = (uint32_t)(pos - j0) * C::RB;
                        const uint32_t bytes = (uint32_t)(j0 + n - pos) * C::RB;
                        bulk_copy_g2s_hint(dst + so, kbase + key * D, bytes, &full[stage], policy);
                        bulk_copy_g2s_hint(dst + C::KV_OFF + so, vbase + key * D, bytes, &full[stage], policy);
                    }
                } else if (n > 0 && !p.block_table) {
                    if (leader) {
                        const uint32_t bytes = (uint32_t)n * C::RB;
                        bulk_copy_g2s_hint(dst, kbase + (size_t)j0 * D, bytes, &full[stage], policy);
                        bulk_copy_g2s_hint(dst + C::KV_OFF, vbase + (size_t)j0 * D, bytes, &full[stage], policy);
                    }
                } else if (n > 0) {
                    // paged: one copy per page segment of the tile, segment s
                    // issued by lane s % 32 (segment 0 starts at j0, the
                    // others at page starts)
                    const int kvh = unit - b * p.Hkv;
                    const int32_t *bt = p.block_table + (size_t)b * p.pages_per_seq;
                    const int pg0 = j0 / p.page_size;
                    const int n_seg = (j0 + n - 1) / p.page_size - pg0 + 1;
                    for (int sg = lane; sg < n_seg; sg += 32) {
                        const int pg = pg0 + sg;
                        const int j = sg == 0 ? j0 : pg * p.page_size;
                        const int off = j - pg * p.page_size;
                        const int cnt = min(p.page_size - off, j0 + n - j);
                        int page = bt[pg];
                        if (page < 0 || page >= p.num_pages) {
                            atomicOr(&p.status[0], TA_DEVERR_PAGE);
                            page = 0;  // stay in bounds; the output is flagged invalid
                        }
                        const size_t row = ((size_t)page * p.Hkv + kvh) * p.page_size + off;
                        const uint32_t bytes = (uint32_t)cnt * C::RB;
                        const uint32_t so = (uint32_t)(j - j0) * C::RB;
                        bulk_copy_g2s_hint(dst + so, static_cast<const KV *>(p.k) + row * D, bytes, &full[stage],
                                           policy);
                        bulk_copy_g2s_hint(dst + C::KV_OFF + so, static_cast<const KV *>(p.v) + row * D, bytes,
                                           &full[stage], policy);
                    }
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
        // Drain: every copy this warp issued has landed before the CTA exits
        // (immediate on the normal path; bounded after an abort).
        __syncwarp();
        if (leader) {
            int drain_abort = 0;
            for (int s = 0; s < C::STAGES; ++s)
                if (used_mask & (1u << s))
                    mbar_wait_bounded(&full[s], (parity_mask >> s) & 1u, &drain_abort);
            if (*abort_flag)
                atomicOr(&p.status[0], TA_DEVERR_TIMEOUT);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Score layout.  A warp's KPW keys of a tile are processed in one step:
    // lane group g (8 lanes) takes keys kbeg + g*KPG + kk, kk < KPG.  Each
    // group reduces its NV = KPG*G (key, head) dot products by a
    // reduce-scatter, after which lane t holds NVL of them (score index
    // (t / RED) * NVL + j, RED lanes holding each when NV < 8).
    using L = Lay<C::KPW / 4, G>;
    const int g = lane >> 3;  // lane group
    const int t = lane & 7;   // lane within the group
    const int tid = threadIdx.x;

    uint32_t qw[G][C::QPL_W];  // this lane's q slice: bf16 pairs, or fp32 bits
    float o[G][C::DPL];        // this lane's output dims of every head, unnormalised
    float m_run[L::NVL];       // running reference (log2 units) of this lane's heads, warp-uniform per head
    float l_run[L::NVL];       // this lane's share of those heads' weight sums
    int stage = 0;
    uint32_t phase = 0;
    uint32_t merge_phase = 0, ticket_phase = 0, fm_phase = 0;
    int b = 0, kvh = 0, split = 0, unit = 0;
    float qs = p.qscale;  // scale * log2(e), times the key dequantisation factor
    float *slot = pbuf + warp * (C::KPW * G);  // this warp's weights [KPW][G]
    int my_kidx[L::NVL], my_h[L::NVL];          // key (within the warp's KPW) and head of value j
#pragma unroll
    for (int j = 0; j < L::NVL; ++j) {
        my_kidx[j] = g * L::KPG + L::kk_of(t, j);
        my_h[j] = L::h_of(t, j);
    }

    for (;;) {
        bool ok = mbar_wait_bounded(&full[stage], phase, abort_flag, p.wait_ns);
        if (!__all_sync(kFull, ok))
            break;
        const TileDesc d = desc[stage];
        if (d.flags & kEnd)
            break;
        if (d.flags & kFirst) {
            unit = p.cm.unit_of(d.item);
            split = p.cm.split_of(d.item);
            b = unit / p.Hkv;
            kvh = unit - b * p.Hkv;
            qs = p.k_scale ? p.qscale * p.k_scale[unit] : p.qscale;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if constexpr (sizeof(KV) == 1) {
                    // bf16 q, as f16 pairs for the mixed-precision products
                    // with f16-widened e4m3 keys
                    const __nv_bfloat16 *qrow =
                        static_cast<const __nv_bfloat16 *>(p.q) + ((size_t)b * p.Hq + (size_t)kvh * G + h) * D;
#pragma unroll
                    for (int i = 0; i < C::NCH; ++i) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(qrow + (t + 8 * i) * C::EPC);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const uint4 raw = src[u];
                            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                uint32_t hv;
                                asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hv) : "f"(bf16_hi(wv[w])), "f"(bf16_lo(wv[w])));
                                qw[h][8 * i + 4 * u + w] = hv;
                                // a query outside the fp16 range: its scores are not the exact ones
                                if (bf16x2_beyond_f16(wv[w]))
                                    atomicOr(&p.status[0], TA_DEVERR_RANGE);
                            }
                        }
                    }
                } else {
                    const KV *qrow = static_cast<const KV *>(p.q) + ((size_t)b * p.Hq + (size_t)kvh * G + h) * D;
#pragma unroll
                    for (int i = 0; i < C::NCH; ++i) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + (t + 8 * i) * C::EPC);
                        qw[h][4 * i + 0] = raw.x;
                        qw[h][4 * i + 1] = raw.y;
                        qw[h][4 * i + 2] = raw.z;
                        qw[h][4 * i + 3] = raw.w;
                    }
                }
#pragma unroll
                for (int e = 0; e < C::DPL; ++e)
                    o[h][e] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < L::NVL; ++j) {
                m_run[j] = -INFINITY;
                l_run[j] = 0.f;
            }
        }

        const unsigned char *Ks = smem + stage * C::STAGE;
        const unsigned char *Vs = Ks + C::KV_OFF;
        const int kbeg = warp * C::KPW;
        // FULL: all KPW keys of this warp are present (every tile but a
        // chunk's last), so no key needs a bounds check.
        auto step = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const int nvalid = FULL ? C::KPW : min(C::KPW, d.n - kbeg);
            // ---- <q_h, k> partial sums over this lane's slice of each row
            float v[L::NV];
#pragma unroll
            for (int i = 0; i < L::NV; ++i)
                v[i] = 0.f;
#pragma unroll
            for (int kk = 0; kk < L::KPG; ++kk) {
                const int kidx = g * L::KPG + kk;
                if (FULL || kidx < nvalid) {
#pragma unroll
                    for (int i = 0; i < C::NCH; ++i) {
                        const uint4 kr =
                            *reinterpret_cast<const uint4 *>(Ks + (kbeg + kidx) * C::RB + (t + 8 * i) * 16);
                        const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
                        if constexpr (sizeof(KV) == 1) {
                            // 16 e4m3 keys -> 8 f16 pairs, once for all heads
                            uint32_t kh[8];
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                kh[2 * w] = e4m3x2_to_f16x2((uint16_t)(kw[w] & 0xffffu));
                                kh[2 * w + 1] = e4m3x2_to_f16x2((uint16_t)(kw[w] >> 16));
                            }
#pragma unroll
                            for (int h = 0; h < G; ++h)
#pragma unroll
                                for (int w = 0; w < 8; ++w)
                                    fma_f16(v[kk * G + h], qw[h][8 * i + w], kh[w]);
                        } else {
#pragma unroll
                            for (int h = 0; h < G; ++h)
#pragma unroll
                                for (int w = 0; w < 4; ++w) {
                                    if constexpr (sizeof(KV) == 2)
                                        fma_bf16(v[kk * G + h], qw[h][4 * i + w], kw[w]);
                                    else
                                        v[kk * G + h] = fmaf(__uint_as_float(qw[h][4 * i + w]),
                                                             __uint_as_float(kw[w]), v[kk * G + h]);
                                }
                        }
                    }
                }
            }
            // ---- 8-lane reduce-scatter (then all-reduce while NV < 8)
            int n = L::NV;
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                const int mask = 4 >> r;
                if (n > 1) {
                    const bool upper = (t & mask) != 0;
#pragma unroll
                    for (int i = 0; i < n / 2; ++i) {
                        const float send = upper ? v[i] : v[i + n / 2];
                        const float keep = upper ? v[i + n / 2] : v[i];
                        v[i] = keep + __shfl_xor_sync(kFull, send, mask);
                    }
                    n /= 2;
                } else {
                    v[0] += __shfl_xor_sync(kFull, v[0], mask);
                }
            }
            float sc[L::NVL];
            bool need = false;
#pragma unroll
            for (int j = 0; j < L::NVL; ++j) {
                sc[j] = (FULL || my_kidx[j] < nvalid) ? v[j] * qs : -INFINITY;  // log2 units
                need |= sc[j] > m_run[j] + kRescaleLog2;
            }
            // ---- lazy rescale of the running references (warp vote)
            if (__any_sync(kFull, need)) {
                float alpha[L::NVL];
#pragma unroll
                for (int j = 0; j < L::NVL; ++j) {
                    float mx = sc[j];
#pragma unroll
                    for (int mask = 1; mask < 32; mask <<= 1)
                        if (L::preserves_head(mask))
                            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mask));
                    alpha[j] = 1.f;
                    if (mx > m_run[j] + kRescaleLog2) {
                        alpha[j] = m_run[j] == -INFINITY ? 0.f : fast_exp2(m_run[j] - mx);
                        m_run[j] = mx;
                        l_run[j] *= alpha[j];
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float a = __shfl_sync(kFull, alpha[L::j_of_head(h)], L::lane_of_head(h));
#pragma unroll
                    for (int e = 0; e < C::DPL; ++e)
                        o[h][e] *= a;
                }
            }
            // ---- weights: one exp per score, into shared memory for PV
#pragma unroll
            for (int j = 0; j < L::NVL; ++j) {
                const float pw = (FULL || my_kidx[j] < nvalid) ? fast_exp2(sc[j] - m_run[j]) : 0.f;
                l_run[j] += pw;
                if (t % L::RED == 0)
                    slot[my_kidx[j] * G + my_h[j]] = pw;
            }
            __syncwarp();
            // ---- PV: lanes own D/32 dims of every head; keys C::PB at a time
#pragma unroll
            for (int k0 = 0; k0 < C::KPW; k0 += C::PB) {
                float pk[C::PB][G];
                float vf[C::PB][C::DPL];
#pragma unroll
                for (int kk = 0; kk < C::PB; ++kk) {
                    if (FULL || k0 + kk < nvalid) {
                        load_weights<G>(slot + (k0 + kk) * G, pk[kk]);
                        load_v_slice<C::DPL>(Vs + (kbeg + k0 + kk) * C::RB + lane * C::VB, vf[kk], (KV *)nullptr);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < C::PB; ++kk) {
                    if (FULL || k0 + kk < nvalid) {
#pragma unroll
                        for (int h = 0; h < G; ++h)
#pragma unroll
                            for (int e = 0; e < C::DPL; ++e)
                                o[h][e] = fmaf(pk[kk][h], vf[kk][e], o[h][e]);
                    }
                }
            }
        };
        if (d.n >= kbeg + C::KPW)
            step(std::true_type{});
        else if (d.n > kbeg)
            step(std::false_type{});
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);
        if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
        }
        if (!(d.flags & kLast))
            continue;

        // ---- end of item: each head's weight sum over the warp, then merge
        // the consumer warps
#pragma unroll
        for (int j = 0; j < L::NVL; ++j) {
            if (t % L::RED != 0)
                l_run[j] = 0.f;  // redundant copies count once
#pragma unroll
            for (int mask = 1; mask < 32; mask <<= 1)
                if (L::preserves_head(mask))
                    l_run[j] += __shfl_xor_sync(kFull, l_run[j], mask);
        }
        if (p.v_scale) {
            const float vs = p.v_scale[unit];  // value dequantisation factor
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < C::DPL; ++e)
                    o[h][e] *= vs;
        }
        ok = mbar_wait_bounded(merge_out, merge_phase ^ 1, abort_flag, p.wait_ns);
        if (!__all_sync(kFull, ok))
            break;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = merge_o + (warp * G + h) * D + lane * C::DPL;
#pragma unroll
            for (int e = 0; e < C::DPL; e += 2)
                *reinterpret_cast<float2 *>(dst + e) = make_float2(o[h][e], o[h][e + 1]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if (lane == L::lane_of_head(h)) {
                merge_m[warp * G + h] = m_run[L::j_of_head(h)];
                merge_l[warp * G + h] = l_run[L::j_of_head(h)];
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(merge_in);
        ok = mbar_wait_bounded(merge_in, merge_phase, abort_flag, p.wait_ns);
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
            if (mbar_wait_bounded(written, ticket_phase, abort_flag, p.wait_ns)) {
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
        ok = mbar_wait_bounded(ticket, ticket_phase, abort_flag, p.wait_ns);
        ticket_phase ^= 1;
        if (!__all_sync(kFull, ok))
            break;
        if (!*ticket_flag)
            continue;
        // Stage the unit's partial m and l in shared memory, then every thread
        // owns 4 consecutive dims of one head, with its loads of o in flight
        // together.
        const int ns = p.n_split;
        for (int i = tid; i < G * ns; i += kConsumerThreads) {
            const int h = i / ns;
            const size_t pi = (row0 + h) * ns + (i - h * ns);
            fm_m[i] = __ldcg(p.part_m + pi);
            fm_l[i] = __ldcg(p.part_l + pi);
        }
        mbar_arrive(fm_ready);
        ok = mbar_wait_bounded(fm_ready, fm_phase, abort_flag, p.wait_ns);
        fm_phase ^= 1;
        if (!__all_sync(kFull, ok))
            break;
        for (int idx = tid; idx < G * D / 4; idx += kConsumerThreads) {
            const int h = idx / (D / 4);
            const int d4 = (idx - h * (D / 4)) * 4;
            const float *mh = fm_m + h * ns;
            const float *lh = fm_l + h * ns;
            float mx = -INFINITY;
            for (int n = 0; n < ns; ++n)
                mx = fmaxf(mx, mh[n]);
            float ls = 0.f;
            float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
            if (mx != -INFINITY) {
                const float4 *po = reinterpret_cast<const float4 *>(p.part_o + (row0 + h) * ns * D + d4);
#pragma unroll 4
                for (int n = 0; n < ns; ++n) {
                    const float mn = mh[n];
                    const float a = mn == -INFINITY ? 0.f : fast_exp2((mn - mx) * kLog2e);
                    const float4 x = __ldcg(po + (size_t)n * (D / 4));
                    ls = fmaf(a, lh[n], ls);
                    os.x = fmaf(a, x.x, os.x);
                    os.y = fmaf(a, x.y, os.y);
                    os.z = fmaf(a, x.z, os.z);
                    os.w = fmaf(a, x.w, os.w);
                }
            }
            const float inv = ls > 0.f ? 1.0f / ls : 0.f;
            OUT *dst = static_cast<OUT *>(p.out) + (row0 + h) * D + d4;
            store_out(dst + 0, os.x * inv);
            store_out(dst + 1, os.y * inv);
            store_out(dst + 2, os.z * inv);
            store_out(dst + 3, os.w * inv);
            if (d4 == 0 && p.lse)
                p.lse[row0 + h] = ls > 0.f ? mx + fast_log2(ls) * kLn2 : -INFINITY;
        }
    }
    // A consumer warp that gave up (or saw another give up) records it: the
    // producer may have returned before the wait that failed.
    if (lane == 0 && *abort_flag)
        atomicOr(&p.status[0], TA_DEVERR_TIMEOUT);
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
    if (a.kv_fp8) {
        if constexpr (D == 128 && G <= 4) {
            if (a.out_dtype == TA_BF16)
                return launch_typed<D, G, __nv_fp8_e4m3, __nv_bfloat16>(a, p);
            return launch_typed<D, G, __nv_fp8_e4m3, float>(a, p);
        }
        return cudaErrorInvalidValue;
    }
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
    if (cudaError_t inj = injected_launch_failure())
        return inj;
    if (decode_tc_eligible(a))
        return launch_decode_tc(a);
    if (decode_fp8_tc_eligible(a))
        return launch_decode_fp8_tc(a);
    if (a.kv_nvfp4)
        return cudaErrorNotSupported;  // NVFP4 caches run on the tensor-core kernel only
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
    p.cm = ChunkMap{a.B * a.Hkv, a.plan.chunk};
    p.n_items = a.B * a.Hkv * a.plan.n_split;
    if (a.force_partials)
        p.mode = kModePartials;
    else if (a.plan.n_split == 1)
        p.mode = kModeFinal;
    else
        p.mode = decode_merges_itself(a.plan.n_split, a.B * a.Hkv) ? kModeFused : kModePartials;
    p.status = a.status;
    p.wait_ns = a.wait_ns;
    p.test_stall = a.test_stall;
    p.counters = a.counters;
    p.part_m = a.part_m;
    p.part_l = a.part_l;
    p.part_o = a.part_o;
    p.block_table = a.block_table;
    p.page_size = a.page_size;
    p.pages_per_seq = a.pages_per_seq;
    p.num_pages = a.num_pages;
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.pi_window = a.pi_window;
    p.pi_period = a.pi_period;
    p.pi_tma = 0;
    if (a.pi_period > 1) {
        const bool bf16 = a.in_dtype == TA_BF16;
        const uint64_t es = bf16 ? 2 : 4;
        const uint64_t dims[3] = {(uint64_t)a.pi_period * a.D, ((uint64_t)a.S + a.pi_period - 1) / a.pi_period,
                                  (uint64_t)a.B * a.Hkv};
        const uint64_t strides[2] = {(uint64_t)a.pi_period * a.D * es, (uint64_t)a.S * a.D * es};
        const uint32_t box[3] = {(uint32_t)a.D, (uint32_t)(a.D * es > 256 ? 60 : 120), 1};
        // the boxes only ever cover keys below S of one (sequence, KV head)
        p.pi_tma = encode_tmap_3d(&p.pi_kmap, a.k, bf16, dims, strides, box, false) &&
                   encode_tmap_3d(&p.pi_vmap, a.v, bf16, dims, strides, box, false);
    }
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
