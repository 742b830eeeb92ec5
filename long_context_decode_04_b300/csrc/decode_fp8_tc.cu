// decode_fp8_tc.cu -- split-KV exact decode over an FP8 (E4M3) KV cache for
// grouped-query attention, with both contractions on the tensor cores.
//
// What is computed is the decode of decode_tc.cu (Attention glossary,
// jisaku.com/glossary/attention, "basic concepts and operating principle";
// partials merged by the log-sum-exp rule of the Tree Attention explainer,
// aibr.jp/archives/143699, sections 1 and 3) over a cache stored in low
// precision and computed in higher precision (the ThriftAttention page,
// hyperion-consulting.io, "the rise of FP4" and the COMPUTE layer): K and V
// are E4M3 codes with one fp32 dequantisation factor per (sequence, KV
// head) each, q is bf16.  The K factor scales the scores, the V factor the
// partial.  Same chunks of whole 128-key tiles, same partials.
//
// The tensor cores take 16-bit operands, so each tile is widened on chip:
// E4M3 is a subset of fp16, and cvt.rn.f16x2.e4m3x2 widens two codes
// exactly.  The raw codes arrive by TMA in a ring of stages that is
// released as soon as a tile is widened, so most of the ring is in flight.
//   S^T [128 keys x 16] = K [128 x D] . Q^T   A = K in TMEM (fp16, written by
//                                            the converting threads, one key
//                                            row per TMEM lane), B = q as fp16
//                                            (K-major, 128-byte swizzle)
//   O_t^T [D x 32]      = V^T . P^T          A = V as fp16 in shared memory
//                                            (MN-major, 128-byte swizzle),
//                                            B = P, one row per (softmax
//                                            warp, head), hi then lo parts
// Queries are used as fp16 values: exact for bf16 values of magnitude in
// [2^-17, 65280] (and zero); one of magnitude 2^16 or more does not fit,
// and the producer records TA_DEVERR_RANGE.
//
// Kernel layout (one persistent CTA per SM, 12 warps):
//   * warp 0: producer.  Work items (sequence, KV head, chunk) from the
//     device-wide queue; the item's G query rows widened to fp16 into one of
//     two Q buffers; raw K and V tiles (128 rows of 128 codes) by TMA into a
//     3-stage ring.
//   * warp 1: TMEM (512 columns: S and O double buffers, three K buffers)
//     and the score products; warp 2: the value products; warp 3 (fused
//     mode): the ticket thread of the merge.
//   * warps 4-7: softmax and accumulation, as in decode_tc.cu (each warp its
//     own online softmax over its 32 keys, per-warp references raised
//     lazily, the four warps merged at the item end).
//   * warps 8-11 (TMEM lane quadrants 0-3): widen a tile: thread r writes
//     key row r of K into TMEM, and the threads write V as fp16 into shared
//     memory (zero for keys past the tile's end); then the raw stage is free.
//   * Every wait is bounded (kWaitLimitNs); on expiry the kernel records
//     TA_DEVERR_TIMEOUT, stops, lets its copies and MMAs land and frees its
//     TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "decode_tc_common.cuh"
#include "tcgen05.cuh"

namespace ta {
namespace {

constexpr int kD = 128;
constexpr int kTile = kDecodeTileKeysTC;  // 128 keys a tile
constexpr int kRows = 128;                // MMA rows: one key a row
constexpr int kN = 16;                  // score-product N: the group's heads, zero-padded
constexpr int kON = 2 * kN;             // value-product N: (warp, head) columns, hi then lo
constexpr int kConvBufs = 3;                      // widened tiles (K in TMEM, V in shared memory)
// The raw ring holds tiles as they arrive by TMA, in the cache's format:
//   E4M3:  K then V, each 128 rows of 128 one-byte codes (128-byte swizzle);
//   NVFP4: K codes, V codes (each 128 keys x 64 bytes seen as 64 rows of 128
//          bytes, two keys a row, 128-byte swizzle), then K and V block
//          scales (each 128 keys x 8 bytes seen as 8 rows of 128 bytes).
template <bool NV4>
struct Raw;
template <>
struct Raw<false> {
    static constexpr int kKBytes = kTile * kD;     // 16 KiB
    static constexpr int kStage = 2 * kKBytes;     // 32 KiB
    static constexpr int kStages = 3;
};
template <>
struct Raw<true> {
    static constexpr int kCodes = kTile * kD / 2;  // 8 KiB
    static constexpr int kScales = kTile * kD / 16;  // 1 KiB
    static constexpr int kStage = 2 * kCodes + 2 * kScales;  // 18 KiB
    static constexpr int kStages = 5;
};
constexpr int kMaxRawStages = 5;
constexpr int kRawRegion = 98304;                 // room for either ring
constexpr int kHalf = kRows * 128;                // one 64-dim half of an fp16 V tile
constexpr int kVBytes = 2 * kHalf;                // 32 KiB
constexpr int kQHalf = kN * 128;
constexpr int kQBytes = 2 * kQHalf;
constexpr int kPHalf = kON * 128;
constexpr int kPBytes = 2 * kPHalf;
constexpr int kVOff = 0;                          // kConvBufs fp16 V tiles
constexpr int kQOff = kVOff + kConvBufs * kVBytes;  // two fp16 Q operands
constexpr int kPOff = kQOff + 2 * kQBytes;        // two P operands
constexpr int kRawOff = kPOff + 2 * kPBytes;      // the raw ring
constexpr int kMiscOff = kRawOff + kRawRegion;
constexpr int kDescRing = 8;
constexpr int kSoftWarp0 = 4;
constexpr int kConvWarp0 = 8;
constexpr int kSoftThreads = 128;
constexpr int kThreads = 384;
constexpr uint32_t kOCol = 2 * kN;                // S at TMEM columns 0, 16; O at 32, 64
constexpr uint32_t kKCol = kOCol + 2 * kON;       // K at 96, 160, 224
constexpr uint32_t kTmemCols = 512;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kRescaleLog2 = 8.0f;
// partial outputs in flight per round of the fused merge (the register
// budget of 256 threads allows sixteen float4, that of 384 threads eight)
constexpr int kMergeBatch = 8;

enum : int { kFirst = 1, kLast = 2, kEnd = 4 };
constexpr int kModeFinal = tcd::kModeFinal, kModePartials = tcd::kModePartials, kModeFused = tcd::kModeFused;

struct TileDesc {
    int item;
    int j0;
    int n;
    int flags;
};

struct Misc {
    uint64_t raw_full[kMaxRawStages];   // raw codes landed (TMA bytes), descriptor written
    uint64_t raw_empty[kMaxRawStages];  // raw codes widened (128 converting threads)
    uint64_t conv_full[kConvBufs];   // K in TMEM and V as fp16 (128 converting threads)
    uint64_t conv_empty[kConvBufs];  // the value product of the tile read them (MMA commit)
    uint64_t s_full[2];              // S in TMEM (MMA commit) and its descriptor (score issuer)
    uint64_t p_full[2][4];           // a warp's P (32 threads)
    uint64_t p_all[2];               // all four warps' P and factors (128 threads)
    uint64_t o_full[2];
    uint64_t o_empty[2];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t grp_bar;
    uint64_t mma_done;
    TileDesc desc[kDescRing];        // tile t's descriptor at t % kDescRing
    float alpha[4][4][4];            // [tile % 4][warp][head]
    tcd::ItemSmem isum;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmem = (size_t)kMiscOff + sizeof(Misc) + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory per CTA");
static_assert(Raw<false>::kStages * Raw<false>::kStage <= kRawRegion && Raw<true>::kStages * Raw<true>::kStage <= kRawRegion,
              "raw rings");
static_assert(Raw<false>::kKBytes % 1024 == 0 && Raw<true>::kCodes % 1024 == 0 && Raw<true>::kStage % 1024 == 0 &&
                  kRawOff % 1024 == 0, "raw tiles on 1024-byte boundaries (swizzle atoms)");
static_assert(kTile * 4 % kSoftThreads == 0, "V widening tasks per thread");

struct Fp8Params {
    // E4M3: codes (D, S, B*Hkv), box 128 x 128; NVFP4: codes (128 bytes,
    // S/2, B*Hkv), box 128 x 64, and block scales (128 bytes, S/16, B*Hkv),
    // box 128 x 8
    CUtensorMap kmap, vmap, ksmap, vsmap;
    const __nv_bfloat16 *q;
    void *out;
    float *lse;
    int B, Hq, Hkv, S;
    float qscale;  // scale * log2(e)
    const int32_t *seqlens;
    int n_split, chunk, n_items;
    ChunkMap cm;  // work item -> (unit, chunk) and the chunk's keys
    int mode;
    int32_t *status;
    int32_t *counters;
    float *part_m, *part_l, *part_o;
    uint64_t wait_ns;  // time limit of a pipeline wait
    int test_stall;    // test hook: the producer first waits on a barrier nothing ends
    const float *k_scale, *v_scale;  // per (sequence, KV head), or nullptr (1)
};


// Two E4M3 codes (low byte first) to a packed fp16 pair (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
    return r;
}

// Four codes of a word to two fp16 pairs.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    lo = e4m3x2_to_f16x2(w & 0xffffu);
    hi = e4m3x2_to_f16x2(w >> 16);
}

// Eight E2M1 codes of a word (element 2i in the low nibble of byte i) to
// four fp16 pairs, each multiplied by the fp16 pair s2: an E2M1 value (2
// significant bits) times an E4M3 scale (4) is exact in fp16 (11), and in
// its range (at most 6 * 448 in magnitude, at least 2^-10 when not 0).
__device__ __forceinline__ void e2m1x8_scaled(uint32_t w, uint32_t s2, uint32_t (&d)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        ".reg .b32 c0, c1, c2, c3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 c0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 c1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 c2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 c3, b3;\n\t"
        "mul.rn.f16x2 %0, c0, %5;\n\t"
        "mul.rn.f16x2 %1, c1, %5;\n\t"
        "mul.rn.f16x2 %2, c2, %5;\n\t"
        "mul.rn.f16x2 %3, c3, %5;\n\t}"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(w), "r"(s2));
}

// Two E4M3 block scales (the low two bytes of `two`) as two fp16 pairs,
// each holding its value twice.
__device__ __forceinline__ void e4m3_scales2(uint32_t two, uint32_t &s0, uint32_t &s1)
{
    const uint32_t h = e4m3x2_to_f16x2(two & 0xffffu);
    s0 = __byte_perm(h, 0u, 0x1010);
    s1 = __byte_perm(h, 0u, 0x3232);
}

template <int G, typename OUT, bool NV4>
__global__ void __launch_bounds__(kThreads, 1) decode_fp8_tc_kernel(const __grid_constant__ Fp8Params p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Misc *ms = reinterpret_cast<Misc *>(smem + kMiscOff);
    volatile int *abort_flag = &ms->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Zero what no widening or query write covers: the Q operands (rows
    // G..15) and the P operands.
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < (kRawOff - kQOff) / 16; i += kThreads)
        *reinterpret_cast<uint4 *>(smem + kQOff + i * 16) = z4;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

    using RC = Raw<NV4>;
    constexpr int kRawStages = RC::kStages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(&ms->raw_full[s], 1);
            mbar_init(&ms->raw_empty[s], kSoftThreads);
        }
        for (int i = 0; i < kConvBufs; ++i) {
            mbar_init(&ms->conv_full[i], kSoftThreads);
            mbar_init(&ms->conv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms->s_full[i], 2);
            for (int w = 0; w < 4; ++w)
                mbar_init(&ms->p_full[i][w], 32);
            mbar_init(&ms->p_all[i], kSoftThreads);
            mbar_init(&ms->o_full[i], 1);
            mbar_init(&ms->o_empty[i], kSoftThreads);
            mbar_init(&ms->q_full[i], 1);
            mbar_init(&ms->q_empty[i], 1);
        }
        mbar_init(&ms->grp_bar, 4);
        mbar_init(&ms->mma_done, 2);  // both MMA issuers commit
        ms->abort = 0;
        tcd::init_item_smem(&ms->isum);
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&ms->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = ms->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const bool leader = lane == 0;
        if (leader) {
            tc::prefetch_tensormap(&p.kmap);
            tc::prefetch_tensormap(&p.vmap);
        }
        const uint64_t policy = l2_policy_evict_first();
        int stage = 0, ti = 0, ic = 0;
        uint32_t uses[kMaxRawStages] = {};
        uint32_t q_uses[2] = {0u, 0u};
        // The item's G query rows as fp16 into Q buffer ic % 2: 16-byte chunk c
        // of head h (8 dims) to row h of the operand, 128-byte swizzle.
        auto widen_q = [&](int item) -> bool {
            const int unit = p.cm.unit_of(item);
            const int qb = ic & 1;
            int w = 1;
            if (leader && q_uses[qb] > 0)
                w = mbar_wait_bounded(&ms->q_empty[qb], (q_uses[qb] - 1) & 1, abort_flag, p.wait_ns);
            if (!__shfl_sync(kFull, w, 0))
                return false;
            unsigned char *qd = smem + kQOff + qb * kQBytes;
            const __nv_bfloat16 *qsrc = p.q + (size_t)unit * G * kD;
            bool big = false;
            for (int i = lane; i < G * 16; i += 32) {
                const int h = i >> 4, c = i & 15;
                const uint4 x = *reinterpret_cast<const uint4 *>(qsrc + h * kD + c * 8);
                const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
                uint32_t hv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    hv[k] = tc::pack_f16x2(bf16_lo(wv[k]), bf16_hi(wv[k]));
                    big |= bf16x2_beyond_f16(wv[k]);
                }
                *reinterpret_cast<uint4 *>(qd + (c >> 3) * kQHalf + h * 128 + ((((c & 7) ^ h) & 7) << 4)) =
                    make_uint4(hv[0], hv[1], hv[2], hv[3]);
            }
            if (big)  // a query outside the fp16 range: its scores are not the exact ones
                atomicOr(&p.status[0], TA_DEVERR_RANGE);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (leader)
                mbar_arrive(&ms->q_full[qb]);
            ++q_uses[qb];
            ++ic;
            return true;
        };
        bool ok = true;
        if (p.test_stall) {
            // test hook: a wait that nothing ends (phase 0 of a barrier only
            // this warp arms), so the launch's time limit runs out
            int w = 1;
            if (leader)
                w = mbar_wait_bounded(&ms->raw_full[0], 0, abort_flag, p.wait_ns);
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
                int w = 1;
                if (leader) {
                    if (item == p.n_items + (int)gridDim.x - 1)
                        atomicExch(&p.status[16], 0);  // last grab of the launch: reset the queue
                    if (uses[stage] > 0)
                        w = mbar_wait_bounded(&ms->raw_empty[stage], (uses[stage] - 1) & 1, abort_flag, p.wait_ns);
                    if (w) {
                        ms->desc[ti & (kDescRing - 1)] = TileDesc{item, 0, 0, kEnd};
                        mbar_arrive(&ms->raw_full[stage]);
                    }
                }
                if (__shfl_sync(kFull, w, 0))
                    ++uses[stage];
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
            const int c0 = p.cm.start_of(split);
            const int c1 = min(c0 + p.cm.len_of(split), L);
            int j0 = c0, flags = kFirst;
            for (;;) {
                const int n = max(0, min(kTile, c1 - j0));
                const bool last = j0 + n >= c1;
                if (last)
                    flags |= kLast;
                int w = 1;
                if (leader) {
                    if (uses[stage] > 0)
                        w = mbar_wait_bounded(&ms->raw_empty[stage], (uses[stage] - 1) & 1, abort_flag, p.wait_ns);
                    if (w) {
                        ms->desc[ti & (kDescRing - 1)] = TileDesc{item, j0, n, flags};
                        uint64_t *fb = &ms->raw_full[stage];
                        if (n > 0) {
                            // rows past S read as zero; V rows in [n, 128) are
                            // written as zero by the converting threads
                            unsigned char *rd = smem + kRawOff + stage * RC::kStage;
                            mbar_arrive_expect_tx(fb, (uint32_t)RC::kStage);
                            if constexpr (!NV4) {
                                tc::tma_load_3d_hint(rd, &p.kmap, 0, j0, unit, fb, policy);
                                tc::tma_load_3d_hint(rd + RC::kKBytes, &p.vmap, 0, j0, unit, fb, policy);
                            } else {
                                // tiles start on multiples of 128 keys: whole
                                // code rows (2 keys) and scale rows (16 keys)
                                tc::tma_load_3d_hint(rd, &p.kmap, 0, j0 / 2, unit, fb, policy);
                                tc::tma_load_3d_hint(rd + RC::kCodes, &p.vmap, 0, j0 / 2, unit, fb, policy);
                                tc::tma_load_3d_hint(rd + 2 * RC::kCodes, &p.ksmap, 0, j0 / 16, unit, fb, policy);
                                tc::tma_load_3d_hint(rd + 2 * RC::kCodes + RC::kScales, &p.vsmap, 0, j0 / 16, unit, fb,
                                                     policy);
                            }
                        } else {
                            mbar_arrive(fb);
                        }
                    }
                }
                if (!__shfl_sync(kFull, w, 0)) {
                    ok = false;
                    break;
                }
                ++uses[stage];
                ++ti;
                if (flags & kFirst) {
                    // the item's queries, once its first copy is in flight
                    if (!widen_q(item))
                        ok = false;
                }
                if (!ok)
                    break;
                if (++stage == kRawStages)
                    stage = 0;
                if (last)
                    break;
                j0 += n;
                flags = 0;
            }
        }
        __syncwarp();
        if (leader) {
            int drain_abort = 0;
            for (int s = 0; s < kRawStages; ++s)
                if (uses[s] > 0)
                    mbar_wait_bounded(&ms->raw_full[s], (uses[s] - 1) & 1, &drain_abort);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA issuers
        if (lane == 0) {
            const uint32_t sbase = smem_u32(smem);
            int t = 0;
            if (warp == 1) {
                // score products: S_t^T = K Q^T, K from TMEM, 8 steps of 16 dims
                constexpr uint32_t kIdS = tc::idesc_f16_f32(kRows, kN, false);
                int ic = 0;
                for (;;) {
                    if (!mbar_wait_bounded(&ms->conv_full[t % kConvBufs], (t / kConvBufs) & 1, abort_flag, p.wait_ns))
                        break;
                    const TileDesc d = ms->desc[t & (kDescRing - 1)];
                    // S and P buffers of this parity are free once the value
                    // product of tile t - 2 is done
                    if (t >= 2 && !mbar_wait_bounded(&ms->o_full[t & 1], ((t - 2) >> 1) & 1, abort_flag, p.wait_ns))
                        break;
                    if (d.flags & kEnd) {
                        mbar_arrive(&ms->s_full[t & 1]);  // tells the softmax warps to stop
                        mbar_arrive(&ms->s_full[t & 1]);
                        break;
                    }
                    const int qb = ic & 1;
                    if ((d.flags & kFirst) && !mbar_wait_bounded(&ms->q_full[qb], (ic >> 1) & 1, abort_flag, p.wait_ns))
                        break;
                    tc::fence_after_sync();
                    const uint32_t s_tm = tmem + (t & 1) * kN;
                    const uint32_t k_tm = tmem + kKCol + (t % kConvBufs) * (kD / 2);
                    const uint32_t qa = sbase + kQOff + qb * kQBytes;
                    // descriptor of the first K step; a later step adds its
                    // offset / 16 to the start-address field (no carry below
                    // 256 KiB), so no MMA rebuilds one
                    const uint64_t qdesc = tc::sw128_desc(qa, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t qo = (kk >> 2) * kQHalf + (kk & 3) * 32;
                        tc::mma_ts(s_tm, k_tm + kk * 8, qdesc + (qo >> 4), kIdS, kk > 0 ? 1u : 0u);
                    }
                    // the commit arrives when S is in TMEM; the plain arrive
                    // releases the descriptor this thread acquired
                    tc::commit(&ms->s_full[t & 1]);
                    mbar_arrive(&ms->s_full[t & 1]);
                    if (d.flags & kLast) {
                        tc::commit(&ms->q_empty[qb]);
                        ++ic;
                    }
                    ++t;
                }
            } else {
                // value products: O_t^T = V^T P^T, V fp16 MN-major, P K-major
                constexpr uint32_t kIdPV = tc::idesc_f16_f32_major(kRows, kON, true, false);
                for (;;) {
                    if (!mbar_wait_bounded(&ms->conv_full[t % kConvBufs], (t / kConvBufs) & 1, abort_flag, p.wait_ns))
                        break;
                    if (ms->desc[t & (kDescRing - 1)].flags & kEnd)
                        break;
                    if (!mbar_wait_bounded(&ms->o_empty[t & 1], ((t >> 1) & 1) ^ 1, abort_flag, p.wait_ns))
                        break;
                    const uint32_t o_tm = tmem + kOCol + (t & 1) * kON;
                    const uint32_t vb = sbase + kVOff + (t % kConvBufs) * kVBytes;
                    const uint32_t pb = sbase + kPOff + (t & 1) * kPBytes;
                    bool ok = true;
                    const uint64_t vdesc = tc::sw128_desc(vb, kHalf, 1024), pdesc = tc::sw128_desc(pb, 16, 1024);
#pragma unroll
                    for (int w = 0; w < 4 && ok; ++w) {
                        ok = mbar_wait_bounded(&ms->p_full[t & 1][w], (t >> 1) & 1, abort_flag, p.wait_ns);
                        if (!ok)
                            break;
                        tc::fence_after_sync();
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int kk = 2 * w + i;
                            const uint32_t po = (kk >> 2) * kPHalf + (kk & 3) * 32;
                            tc::mma_ss(o_tm, vdesc + (uint64_t)(kk * (2048 >> 4)), pdesc + (po >> 4), kIdPV,
                                       kk > 0 ? 1u : 0u);
                        }
                    }
                    if (!ok)
                        break;
                    tc::commit(&ms->o_full[t & 1]);
                    tc::commit(&ms->conv_empty[t % kConvBufs]);
                    ++t;
                }
            }
            tc::commit(&ms->mma_done);
            int drain_abort = 0;
            mbar_wait_bounded(&ms->mma_done, 0, &drain_abort);
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        // ------------------------------------------------------------ widening
        const int cq = warp - kConvWarp0;  // TMEM lane quadrant (warp % 4)
        const int ct = cq * 32 + lane;     // key row (K), and work index (V)
        const uint32_t lane_base = (uint32_t)(cq * 32) << 16;
        int t = 0, stage = 0;
        uint32_t rph = 0;
        for (;;) {
            bool w = mbar_wait_bounded(&ms->raw_full[stage], rph, abort_flag, p.wait_ns);
            const TileDesc d = ms->desc[t & (kDescRing - 1)];
            const int cv = t % kConvBufs;
            w = w && mbar_wait_bounded(&ms->conv_empty[cv], ((t / kConvBufs) & 1) ^ 1, abort_flag, p.wait_ns);
            if (!__all_sync(kFull, w))
                break;
            if (d.flags & kEnd) {
                mbar_arrive(&ms->conv_full[cv]);  // the issuers read the end from the descriptor
                break;
            }
            const unsigned char *rk = smem + kRawOff + stage * RC::kStage;
            const uint32_t k_tm = tmem + lane_base + kKCol + cv * (kD / 2);
            unsigned char *vd = smem + kVOff + cv * kVBytes;
            if constexpr (!NV4) {
                const unsigned char *rv = rk + RC::kKBytes;
                // K row ct into TMEM lane ct: 128 codes -> 64 fp16 pairs (the raw
                // rows are swizzled, so the 32 lanes' chunks fall in 8 bank groups)
                uint32_t kr[32];
                uint32_t kh[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(rk + ct * kD + ((c ^ (ct & 7)) << 4));
                    kr[4 * c + 0] = x.x;
                    kr[4 * c + 1] = x.y;
                    kr[4 * c + 2] = x.z;
                    kr[4 * c + 3] = x.w;
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        e4m3x4_to_f16(kr[16 * half + i], kh[2 * i], kh[2 * i + 1]);
                    tc::tmem_st32(k_tm + 32 * half, kh);
                }
                // V: task i = (row r, quarter qq) -> the 32 codes of dims 32qq ..
                // + 31 (raw 16-byte chunks 2qq, 2qq + 1, swizzled) as four
                // 16-byte fp16 chunks 4 (qq & 1) .. + 3 of half qq / 2 (zero
                // past the tile's end).  All loads first.
                constexpr int kV4Tasks = kTile * 4 / kSoftThreads;  // 4 a thread
                uint4 vx[kV4Tasks][2];
#pragma unroll
                for (int k = 0; k < kV4Tasks; ++k) {
                    const int i = ct + k * kSoftThreads;
                    const int r = i >> 2, qq = i & 3;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        vx[k][j] = r < d.n ? *reinterpret_cast<const uint4 *>(rv + r * kD + (((2 * qq + j) ^ (r & 7)) << 4))
                                           : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int k = 0; k < kV4Tasks; ++k) {
                    const int i = ct + k * kSoftThreads;
                    const int r = i >> 2, qq = i & 3;
                    unsigned char *dst = vd + (qq >> 1) * kHalf + r * 128;
                    const int fc0 = 4 * (qq & 1);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 x = vx[k][c >> 1];
                        const uint32_t lo = (c & 1) ? x.z : x.x, hi = (c & 1) ? x.w : x.y;
                        uint32_t f[4];
                        e4m3x4_to_f16(lo, f[0], f[1]);
                        e4m3x4_to_f16(hi, f[2], f[3]);
                        *reinterpret_cast<uint4 *>(dst + (((fc0 + c) ^ (r & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                    }
                }
            } else {
                const unsigned char *rv = rk + RC::kCodes;
                const unsigned char *rks = rk + 2 * RC::kCodes;
                const unsigned char *rvs = rks + RC::kScales;
                // K row ct into TMEM lane ct: 64 code bytes (half of swizzled
                // raw row ct / 2) and 8 block scales -> 64 fp16 pairs
                {
                    const int y = ct >> 1, hf = ct & 1;
                    uint32_t kr[16];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(rk + y * 128 + (((4 * hf + c) ^ (y & 7)) << 4));
                        kr[4 * c + 0] = x.x;
                        kr[4 * c + 1] = x.y;
                        kr[4 * c + 2] = x.z;
                        kr[4 * c + 3] = x.w;
                    }
                    const uint2 sc = *reinterpret_cast<const uint2 *>(rks + (ct >> 4) * 128 + (ct & 15) * 8);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t kh[32];
                        uint32_t s2[4];  // blocks 4 * half .. + 3, each as an fp16 pair
                        const uint32_t sw = half ? sc.y : sc.x;
                        e4m3_scales2(sw, s2[0], s2[1]);
                        e4m3_scales2(sw >> 16, s2[2], s2[3]);
#pragma unroll
                        for (int b4 = 0; b4 < 4; ++b4) {
                            // block b = 4 * half + b4: 16 elements = words 2b, 2b + 1
                            const int blk = 4 * half + b4;
                            uint32_t d0[4], d1[4];
                            e2m1x8_scaled(kr[2 * blk], s2[b4], d0);
                            e2m1x8_scaled(kr[2 * blk + 1], s2[b4], d1);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                kh[8 * b4 + i] = d0[i];
                                kh[8 * b4 + 4 + i] = d1[i];
                            }
                        }
                        tc::tmem_st32(k_tm + 32 * half, kh);
                    }
                }
                // V: task i = (row r, quarter qq) -> the 32 elements of dims
                // 32qq .. + 31 (16 code bytes, blocks 2qq and 2qq + 1) as four
                // 16-byte fp16 chunks 4 (qq & 1) .. + 3 of half qq / 2 (zero
                // past the tile's end).  All loads first.
                constexpr int kV4Tasks = kTile * 4 / kSoftThreads;  // 4 a thread
                uint4 vx[kV4Tasks];
                uint32_t vs[kV4Tasks];
#pragma unroll
                for (int k = 0; k < kV4Tasks; ++k) {
                    const int i = ct + k * kSoftThreads;
                    const int r = i >> 2, qq = i & 3;
                    const int y = r >> 1;
                    const int c16 = 4 * (r & 1) + qq;  // 16-byte chunk of the 128-byte raw row
                    // (a row past the tile's end is written as zero: its block
                    // scales may be anything, NaN included)
                    vx[k] = r < d.n ? *reinterpret_cast<const uint4 *>(rv + y * 128 + ((c16 ^ (y & 7)) << 4))
                                    : make_uint4(0u, 0u, 0u, 0u);
                    vs[k] = r < d.n ? *reinterpret_cast<const uint16_t *>(rvs + (r >> 4) * 128 + (r & 15) * 8 + 2 * qq)
                                    : 0u;
                }
#pragma unroll
                for (int k = 0; k < kV4Tasks; ++k) {
                    const int i = ct + k * kSoftThreads;
                    const int r = i >> 2, qq = i & 3;
                    unsigned char *dst = vd + (qq >> 1) * kHalf + r * 128;
                    const int fc0 = 4 * (qq & 1);
                    uint32_t s0, s1;
                    e4m3_scales2(vs[k], s0, s1);
                    const uint32_t w[4] = {vx[k].x, vx[k].y, vx[k].z, vx[k].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t f[4];
                        e2m1x8_scaled(w[c], c < 2 ? s0 : s1, f);
                        *reinterpret_cast<uint4 *>(dst + (((fc0 + c) ^ (r & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                    }
                }
            }
            tc::tmem_wait_st();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc::fence_before_sync();
            mbar_arrive(&ms->conv_full[cv]);
            mbar_arrive(&ms->raw_empty[stage]);
            ++t;
            if (++stage == kRawStages) {
                stage = 0;
                rph ^= 1;
            }
        }
    } else if (warp >= kSoftWarp0) {
        // ------------------------------------------------------------ softmax + accumulation
        const int q4 = warp - kSoftWarp0;  // TMEM lane quadrant (warp % 4)
        const int row = q4 * 32 + lane;    // key row of a tile; output dimension
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        uint32_t gph = 0;
        int t = 0;
        float mw[G], l_run[G], o[4][G];
        int unit = 0, split = 0, b = 0, kvh = 0;
        float qs = p.qscale;
        const tcd::ItemOut io{p.out,     p.lse,    p.Hq,       p.mode,     p.n_split, p.part_m,
                              p.part_l,  p.part_o, p.counters, abort_flag, p.wait_ns};
        float *const stage_area = ms->isum.stage;
        tcd::PendingTicket pt;
        bool ended = false;
        auto group_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ms->grp_bar);
            const bool w = mbar_wait_bounded(&ms->grp_bar, gph, abort_flag, p.wait_ns);
            gph ^= 1;
            return __all_sync(kFull, w);
        };
        auto accumulate = [&](int x) -> bool {
            bool w = mbar_wait_bounded(&ms->o_full[x & 1], (x >> 1) & 1, abort_flag, p.wait_ns);
            w = w && mbar_wait_bounded(&ms->p_all[x & 1], (x >> 1) & 1, abort_flag, p.wait_ns);  // the factors
            if (!__all_sync(kFull, w))
                return false;
            tc::fence_after_sync();
            uint32_t r[32];
            tc::tmem_ld32(tmem + lane_base + kOCol + (x & 1) * kON, r);
            tc::tmem_wait_ld(r);
#pragma unroll
            for (int w2 = 0; w2 < 4; ++w2)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int c = w2 * G + g;
                    const float ov = __uint_as_float(r[c]) + __uint_as_float(r[kN + c]);
                    o[w2][g] = fmaf(o[w2][g], ms->alpha[x & 3][w2][g], ov);
                }
            tc::fence_before_sync();
            mbar_arrive(&ms->o_empty[x & 1]);
            return true;
        };
        for (;;) {
            const bool w = mbar_wait_bounded(&ms->s_full[t & 1], (t >> 1) & 1, abort_flag, p.wait_ns);  // S, descriptor
            if (!__all_sync(kFull, w))
                break;
            const TileDesc d = ms->desc[t & (kDescRing - 1)];
            if (d.flags & kEnd) {
                ended = true;
                break;
            }
            if (d.flags & kFirst) {
                unit = p.cm.unit_of(d.item);
                split = p.cm.split_of(d.item);
                b = unit / p.Hkv;
                kvh = unit - b * p.Hkv;
                qs = p.k_scale ? p.qscale * p.k_scale[unit] : p.qscale;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    mw[g] = -INFINITY;
                    l_run[g] = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < 4; ++w2)
                        o[w2][g] = 0.f;
                }
            }
            tc::fence_after_sync();
            uint32_t sr[G];
            tc::tmem_ld_small<G>(tmem + lane_base + (t & 1) * kN, sr);
            const bool valid = row < d.n;
            float s[G], mx[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                s[g] = valid ? __uint_as_float(sr[g]) * qs : -INFINITY;  // log2 units
                mx[g] = s[g];
            }
            // lazy per-warp reference: raised only when a score exceeds it by
            // more than 2^8 (warp vote), so the weights stay below 2^8
            float alpha[G], pw[G];
            bool need = false;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                alpha[g] = 1.f;
                need |= s[g] > mw[g] + kRescaleLog2;
            }
            if (__any_sync(kFull, need)) {
#pragma unroll
                for (int mask = 16; mask >= 1; mask >>= 1)
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        mx[g] = fmaxf(mx[g], __shfl_xor_sync(kFull, mx[g], mask));
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (mx[g] > mw[g] + kRescaleLog2) {
                        alpha[g] = mw[g] == -INFINITY ? 0.f : fast_exp2(mw[g] - mx[g]);
                        l_run[g] *= alpha[g];
                        mw[g] = mx[g];
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                pw[g] = mw[g] == -INFINITY ? 0.f : fast_exp2(s[g] - mw[g]);
                l_run[g] += pw[g];
            }
            if (lane < G) {
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (lane == g)
                        ms->alpha[t & 3][q4][g] = alpha[g];
            }
            // P^T: rows w*G + g (hi) and 16 + w*G + g (lo), column `row`,
            // fp16 (the type of V), 128-byte swizzle
            unsigned char *pbase = smem + kPOff + (t & 1) * kPBytes;
            const int cb = (row & 63) * 2;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int rh = q4 * G + g, rl = kN + rh;
                const int base = (row >> 6) * kPHalf + (cb & 15);
                const __half hi = __float2half_rn(pw[g]);
                const __half lo = __float2half_rn(pw[g] - __half2float(hi));
                *reinterpret_cast<__half *>(pbase + base + rh * 128 + ((((cb >> 4) ^ rh) & 7) << 4)) = hi;
                *reinterpret_cast<__half *>(pbase + base + rl * 128 + ((((cb >> 4) ^ rl) & 7) << 4)) = lo;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc::fence_before_sync();
            mbar_arrive(&ms->p_full[t & 1][q4]);
            mbar_arrive(&ms->p_all[t & 1]);
            if (!(d.flags & kFirst) && !accumulate(t - 1))
                break;
            const int tt = t;
            ++t;
            if (!(d.flags & kLast))
                continue;
            if (!accumulate(tt))
                break;

            // ---- end of item: the partial, the result, and in fused mode the merge
            if (!tcd::finish_item<G, OUT, kMergeBatch>(io, &ms->isum, stage_area, q4, lane, unit, split, b, kvh, p.v_scale ? p.v_scale[unit] : 1.f, mw, l_run,
                                          o, pt, group_sync))
                break;
        }
        if (ended)
            tcd::finish_pending<G, OUT, kMergeBatch>(io, &ms->isum, stage_area, q4, lane, pt, group_sync, smem + kRawOff,
                                                     (size_t)kRawRegion);
        if (p.mode == kModeFused)
            tcd::end_tickets(&ms->isum, row);
    } else if (warp == 3) {
        // ------------------------------------------------------------ ticket thread
        if (lane == 0 && p.mode == kModeFused) {
            const tcd::ItemOut io{p.out,     p.lse,    p.Hq,       p.mode,     p.n_split, p.part_m,
                                  p.part_l,  p.part_o, p.counters, abort_flag, p.wait_ns};
            tcd::ticket_loop(io, &ms->isum);
        }
        __syncwarp();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(&p.status[0], TA_DEVERR_TIMEOUT);
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int G, typename OUT, bool NV4>
cudaError_t launch_typed(const DecodeLaunch &a, const Fp8Params &p)
{
    auto kern = decode_fp8_tc_kernel<G, OUT, NV4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess)
        return e;
    kern<<<a.plan.grid, kThreads, kSmem, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool decode_fp8_tc_eligible(const DecodeLaunch &a)
{
    const int G = a.Hq / a.Hkv;
    return (a.kv_fp8 || a.kv_nvfp4) && a.D == kD && (G == 2 || G == 4) && !a.block_table && a.pi_period == 0;
}

cudaError_t launch_decode_fp8_tc(const DecodeLaunch &a)
{
    const int G = a.Hq / a.Hkv;
    Fp8Params p;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
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
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    const uint64_t units = (uint64_t)a.B * a.Hkv;
    if (!a.kv_nvfp4) {
        // K, V codes [B, Hkv, S, D] as (D, S, B*Hkv), one byte each, box 128 x
        // 128, 128-byte swizzle (16-byte chunk c of row r lands at chunk c ^ (r % 8))
        const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.S, units};
        const uint64_t strides[2] = {(uint64_t)kD, (uint64_t)a.S * kD};
        const uint32_t box[3] = {(uint32_t)kD, (uint32_t)kTile, 1};
        if (!encode_tmap_3d_u8(&p.kmap, a.k, dims, strides, box, true) ||
            !encode_tmap_3d_u8(&p.vmap, a.v, dims, strides, box, true))
            return cudaErrorInvalidValue;
        p.ksmap = p.vsmap = p.kmap;  // unused
    } else {
        // NVFP4 codes [B, Hkv, S, D/2] as (128 bytes, S/2, B*Hkv): two keys a
        // row, box 64 rows (128 keys), 128-byte swizzle; block scales [B, Hkv,
        // S, D/16] as (128 bytes, S/16, B*Hkv), box 8 rows (128 keys).  S is a
        // multiple of 16 (checked by the entry point).
        const uint64_t cdims[3] = {128, (uint64_t)a.S / 2, units};
        const uint64_t cstr[2] = {128, (uint64_t)a.S * (kD / 2)};
        const uint32_t cbox[3] = {128, (uint32_t)kTile / 2, 1};
        const uint64_t sdims[3] = {128, (uint64_t)a.S / 16, units};
        const uint64_t sstr[2] = {128, (uint64_t)a.S * (kD / 16)};
        const uint32_t sbox[3] = {128, (uint32_t)kTile / 16, 1};
        if (!encode_tmap_3d_u8(&p.kmap, a.k, cdims, cstr, cbox, true) ||
            !encode_tmap_3d_u8(&p.vmap, a.v, cdims, cstr, cbox, true) ||
            !encode_tmap_3d_u8(&p.ksmap, a.k_bs, sdims, sstr, sbox, false) ||
            !encode_tmap_3d_u8(&p.vsmap, a.v_bs, sdims, sstr, sbox, false))
            return cudaErrorInvalidValue;
    }
    const bool bf16_out = a.out_dtype == TA_BF16;
    if (a.kv_nvfp4) {
        if (G == 2)
            return bf16_out ? launch_typed<2, __nv_bfloat16, true>(a, p) : launch_typed<2, float, true>(a, p);
        return bf16_out ? launch_typed<4, __nv_bfloat16, true>(a, p) : launch_typed<4, float, true>(a, p);
    }
    if (G == 2)
        return bf16_out ? launch_typed<2, __nv_bfloat16, false>(a, p) : launch_typed<2, float, false>(a, p);
    return bf16_out ? launch_typed<4, __nv_bfloat16, false>(a, p) : launch_typed<4, float, false>(a, p);
}

}  // namespace ta
