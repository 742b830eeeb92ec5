// prefill.cu -- fused causal prefill on the tensor cores (tcgen05 / TMEM).
//
// What is computed (Attention glossary, jisaku.com/glossary/attention,
// "basic concepts and operating principle"): for query row i of each
// (sequence b, head h), scores s_ij = scale * <q_i, k_j> over keys j <= i
// (causal, top-left aligned), softmax weights, and the weighted mean of the
// values, plus lse_i = ln sum_j exp(s_ij).  The Grayskull SRAM attention
// explainer (aibr.jp/archives/146339, section 3) fuses the score matmul,
// the scaling and the softmax into one kernel so that no intermediate goes
// back to DRAM; here the score tile S and the output accumulator O live in
// tensor memory and never leave the SM.
//
// One CTA owns two 128-row query tiles (rows q0 .. q0 + 255) of one
// (b, h) and walks the 128-key K/V tiles up to the causal diagonal:
//   warp 8   TMA producer: loads both Q tiles once, then K tiles into a
//            3-stage and V tiles into a 2-stage shared-memory ring (128-byte
//            swizzle, two 64-column boxes per tile), each ring refilled as
//            soon as it has a free stage (a V tile never before its K tile).
//            It also allocates and frees the TMEM.
//   warp 9   MMA issuer (one thread): per K tile j and query tile t,
//              PV_t(j-1): O_t += P_t(j-1) V_{j-1}  (P from TMEM, V MN-major)
//              S_t(j)   = Q_t K_j^T                (both K-major)
//            Tensor-core operations of one thread run in issue order, so
//            S_t(j) overwrites the TMEM that holds P_t(j-1) only after the
//            PV that reads it, and the commit that signals S_t(j) also
//            guarantees that O_t holds every PV before it.
//   warps 10-11  V converters: each staged V tile is rewritten in place
//            from bf16 to fp16 (same swizzled layout) before the PV that
//            reads it.  P is stored as fp16, whose 11-bit significand keeps
//            the weights' rounding error near 2^-12 (bf16 would give 2^-9,
//            enough to move early causal rows by several 1e-3), and a
//            tcgen05 kind::f16 MMA takes A and B of one type.  bf16 values
//            with |v| <= 65280 convert exactly (subnormal fp16 results lose
//            at most 2^-25 absolute); larger ones set TA_DEVERR_RANGE.
//   warps 0-3 / 4-7   softmax for query tile 0 / 1, one thread per row:
//            read the S row from TMEM, apply the causal mask on the diagonal
//            tile, keep the running reference m (rescaled lazily: only when
//            the row maximum exceeds it by more than 2^8, and then also
//            O_t in TMEM), write P = 2^(s*scale*log2e - m) as fp16 into the
//            first 64 columns of the S tile, and accumulate two row sums:
//            l over P as computed (for lse) and lr over P as rounded to fp16,
//            the weights the PV product uses (for the output, which is then a
//            weighted mean whose weights sum to one exactly; their fp16
//            rounding moves it by at most ~2^-12 of the value range).  The two
//            warpgroups ping-pong: while one does its softmax the tensor cores
//            run the other's PV and QK^T.
//            Epilogue: out = O / lr in bf16 or fp32, lse = (m + log2 l) * ln 2.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// Every wait is bounded; on expiry TA_DEVERR_TIMEOUT is recorded, all roles
// stop, outstanding copies and MMAs are drained and the TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace ta {
namespace {

constexpr int kBM = 128;      // query rows per tile
constexpr int kBN = 128;      // keys per K/V tile
constexpr int kHD = 128;      // head dim
constexpr int kThreads = 384; // 12 warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kConvWarp0 = 10;  // warps 10, 11
constexpr int kConvThreads = 64;
constexpr uint32_t kTileBytes = kBM * kHD * 2;  // 32 KiB (one bf16 tile)
constexpr uint32_t kHalfBytes = kTileBytes / 2; // one 64-column box
constexpr uint32_t kQOff = 0;                   // 2 Q tiles
constexpr int kKStages = 3;                     // K runs a tile ahead of V
constexpr int kVStages = 2;
constexpr uint32_t kKOff = 2 * kTileBytes;      // K ring
constexpr uint32_t kVOff = kKOff + kKStages * kTileBytes;  // V ring
constexpr uint32_t kBarOff = kVOff + kVStages * kTileBytes;
constexpr size_t kSmemBytes = kBarOff + 256 + 1024;  // + alignment slack
constexpr float kRescaleLog2 = 8.0f;

struct PrefillParams {
    // batched: q [B*H, S, D], k/v [B*Hkv, S, D] (z = (b, head), y = token);
    // packed variable lengths: q [T, H, D], k/v [T, Hkv, D] seen as
    // {D, T, heads} (z = head, y = token).  bf16, box {64, 128, 1}.
    CUtensorMap qmap;
    CUtensorMap kmap;
    CUtensorMap vmap;
    void *out;              // bf16 or fp32 (the kernel's OUT type)
    float *lse;
    int S, H, G, n_qt, BH;  // S: keys per sequence (batched) or max_seqlen (packed)
    float c;                // scale * log2(e)
    int32_t *status;
    const int32_t *cu_seqlens;  // packed: [BH / H + 1] token offsets; nullptr: batched
    int T;                      // packed: total tokens
    uint64_t wait_ns;           // time limit of a pipeline wait
    int test_stall;             // test hook: the producer first waits on a barrier nothing ends
};

struct Bars {
    uint64_t q_full;
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages];
    uint64_t v_conv[kVStages];
    uint64_t v_empty[kVStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_full[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

// l += the two fp16 weights of a packed pair, each widened exactly
// (mixed-precision FMA with f16 operands and an fp32 accumulator)
__device__ __forceinline__ float add_f16x2(float acc, uint32_t w)
{
    float r;
    asm("{\n\t.reg .f16 lo, hi, one;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "mov.b16 one, 0x3C00;\n\t"
        "fma.rn.f32.f16 %0, lo, one, %2;\n\t"
        "fma.rn.f32.f16 %0, hi, one, %0;\n\t}"
        : "=f"(r)
        : "r"(w), "f"(acc));
    return r;
}

// Packed fp32 pairs (two lanes of one 64-bit register, one instruction per pair).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f2_unpack(uint64_t w)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(w));
    return r;
}

// a * b + c on both lanes
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint4 out_pack4(const float *x, __nv_bfloat16 *)
{
    return make_uint4(tc::pack_bf16x2(x[0], x[1]), tc::pack_bf16x2(x[2], x[3]), tc::pack_bf16x2(x[4], x[5]),
                      tc::pack_bf16x2(x[6], x[7]));
}

// Eight score-product MMAs (K steps of 16) in one asm block: the predicate
// of the accumulate flag is set once, and steps 1-7 add their offsets (in
// 16-byte units of the start-address field) to the first step's
// descriptors.  Steps: (kk >> 2) * 16 KiB + (kk & 3) * 32 bytes.
__device__ __forceinline__ void mma_ss_x8(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc, uint32_t acc0)
{
    asm volatile(
        "{\n\t.reg .pred p0, p1;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "setp.ne.b32 p1, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
        "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t"
        "add.s64 a, %1, 4;\n\tadd.s64 b, %2, 4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t"
        "add.s64 a, %1, 6;\n\tadd.s64 b, %2, 6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t"
        "add.s64 a, %1, 1024;\n\tadd.s64 b, %2, 1024;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t"
        "add.s64 a, %1, 1026;\n\tadd.s64 b, %2, 1026;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t"
        "add.s64 a, %1, 1028;\n\tadd.s64 b, %2, 1028;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t"
        "add.s64 a, %1, 1030;\n\tadd.s64 b, %2, 1030;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p1;\n\t}"
        ::"r"(d), "l"(a0), "l"(b0), "r"(idesc), "r"(acc0), "r"(1u)
        : "memory");
}

// Eight value-product MMAs: A (P) from TMEM columns a + 8 kk, B (V) steps of
// 2 KiB (128 in 16-byte units).
__device__ __forceinline__ void mma_ts_x8(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc, uint32_t acc0)
{
    asm volatile(
        "{\n\t.reg .pred p0, p1;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "setp.ne.b32 p1, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
        "add.u32 a, %1, 8;\n\tadd.s64 b, %2, 128;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t"
        "add.u32 a, %1, 16;\n\tadd.s64 b, %2, 256;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t"
        "add.u32 a, %1, 24;\n\tadd.s64 b, %2, 384;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t"
        "add.u32 a, %1, 32;\n\tadd.s64 b, %2, 512;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t"
        "add.u32 a, %1, 40;\n\tadd.s64 b, %2, 640;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t"
        "add.u32 a, %1, 48;\n\tadd.s64 b, %2, 768;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t"
        "add.u32 a, %1, 56;\n\tadd.s64 b, %2, 896;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, p1;\n\t}"
        ::"r"(d), "r"(a0), "l"(b0), "r"(idesc), "r"(acc0), "r"(1u)
        : "memory");
}

template <typename OUT>
__global__ void __launch_bounds__(kThreads, 1) prefill_causal_kernel(const __grid_constant__ PrefillParams p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Bars *bars = reinterpret_cast<Bars *>(smem + kBarOff);
    volatile int *abort_flag = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Heaviest query tiles first: they walk the most K/V tiles.
    const int qt = p.n_qt - 1 - (int)(blockIdx.x / p.BH);
    const int bh = (int)(blockIdx.x % p.BH);
    const int q0 = qt * 2 * kBM;
    const int bh_kv = (bh / p.H) * (p.H / p.G) + (bh % p.H) / p.G;
    // This CTA's sequence: L tokens starting at token y0 of the maps' y axis,
    // at z = zq (queries) and zkv (keys, values).
    int L = p.S, y0 = 0, zq = bh, zkv = bh_kv;
    if (p.cu_seqlens) {
        const int seq = bh / p.H, h = bh - seq * p.H;
        const int a = p.cu_seqlens[seq], e = p.cu_seqlens[seq + 1];
        if (threadIdx.x == 0 && qt == 0 && (a < 0 || e < a || e > p.T || e - a > p.S))
            atomicOr(p.status, TA_DEVERR_SEQLEN);
        y0 = max(0, min(a, p.T));
        L = max(0, min(e, p.T) - y0);
        zq = h;
        zkv = h / p.G;
        if (q0 >= L)
            return;  // past this sequence's end: the whole CTA leaves before any set-up
    }
    const bool active1 = q0 + kBM < L;
    const int diag0 = 2 * qt, diag1 = 2 * qt + 1;
    const int nk = (active1 ? diag1 : diag0) + 1;  // K/V tiles this CTA walks

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_conv[s], kConvThreads);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], kBM);
            mbar_init(&bars->o_full[s], 1);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kProducerWarp) {
        tc::tmem_alloc(&bars->tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::prefetch_tensormap(&p.qmap);
            tc::prefetch_tensormap(&p.kmap);
            tc::prefetch_tensormap(&p.vmap);
            // test hook: a wait that nothing ends (phase 0 of a barrier only
            // this thread arms), so the launch's time limit runs out and the
            // CTA issues nothing
            const bool go = !p.test_stall || mbar_wait_bounded(&bars->k_full[0], 0, abort_flag, p.wait_ns);
            const int n_q = active1 ? 2 : 1;
            if (go) {
                mbar_arrive_expect_tx(&bars->q_full, n_q * kTileBytes);
                for (int t = 0; t < n_q; ++t) {
                    unsigned char *dst = smem + kQOff + t * kTileBytes;
                    tc::tma_load_3d(dst, &p.qmap, 0, y0 + q0 + t * kBM, zq, &bars->q_full);
                    tc::tma_load_3d(dst + kHalfBytes, &p.qmap, 64, y0 + q0 + t * kBM, zq, &bars->q_full);
                }
            }
            // K and V tiles each go as soon as their own ring has a free
            // stage (V tile j never before K tile j): a K tile is needed by
            // the score product of its step, while the V ring frees only
            // after the value product of two steps back, so a K copy must
            // not queue behind a V stage.  The thread polls both rings and
            // naps briefly when neither moved; it gives up when nothing moved
            // for the launch's time limit or another role gave up.
            int k_armed[kKStages] = {0, 0, 0}, v_armed[kVStages] = {0, 0};
            bool ok = go;
            int kn = 0, vn = 0;  // next K tile, next V tile
            uint64_t idle_since = 0;
            uint32_t spins = 0;
            while (ok && vn < nk) {
                bool moved = false;
                if (kn < nk) {
                    const int st = kn % kKStages, use = kn / kKStages;
                    if (use == 0 || mbar_test_wait(&bars->k_empty[st], (use - 1) & 1)) {
                        unsigned char *kd = smem + kKOff + st * kTileBytes;
                        mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
                        tc::tma_load_3d(kd, &p.kmap, 0, y0 + kn * kBN, zkv, &bars->k_full[st]);
                        tc::tma_load_3d(kd + kHalfBytes, &p.kmap, 64, y0 + kn * kBN, zkv, &bars->k_full[st]);
                        ++k_armed[st];
                        ++kn;
                        moved = true;
                    }
                }
                if (vn < kn) {
                    const int st = vn % kVStages, use = vn / kVStages;
                    if (use == 0 || mbar_test_wait(&bars->v_empty[st], (use - 1) & 1)) {
                        unsigned char *vd = smem + kVOff + st * kTileBytes;
                        mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
                        tc::tma_load_3d(vd, &p.vmap, 0, y0 + vn * kBN, zkv, &bars->v_full[st]);
                        tc::tma_load_3d(vd + kHalfBytes, &p.vmap, 64, y0 + vn * kBN, zkv, &bars->v_full[st]);
                        ++v_armed[st];
                        ++vn;
                        moved = true;
                    }
                }
                if (moved) {
                    idle_since = 0;
                    spins = 0;
                    continue;
                }
                __nanosleep(64);
                if ((++spins & 15) == 0) {
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint64_t now = globaltimer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > p.wait_ns) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                }
            }
            {
                // Every copy issued lands before the CTA exits, whether or
                // not some role gave up: a role may give up after this
                // thread has issued its last copy, so the drain cannot
                // depend on the abort flag (on the normal path the waits
                // end as soon as the last copies land).
                int drain_abort = 0;
                if (go)
                    mbar_wait_bounded(&bars->q_full, 0, &drain_abort);
                for (int st = 0; st < kKStages; ++st)
                    if (k_armed[st] > 0)
                        mbar_wait_bounded(&bars->k_full[st], (k_armed[st] - 1) & 1, &drain_abort);
                for (int st = 0; st < kVStages; ++st)
                    if (v_armed[st] > 0)
                        mbar_wait_bounded(&bars->v_full[st], (v_armed[st] - 1) & 1, &drain_abort);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t kIdescPV = tc::idesc_f16_f32(kBM, kHD, true);
            const uint32_t sbase = smem_u32(smem);
            // Matrix descriptors of the tiles' first K steps; a later step or
            // stage adds its byte offset / 16 to the start-address field (the
            // addresses stay below 256 KiB, so the field never carries).  The
            // tensor pipe takes only a few operations ahead of this thread, so
            // every instruction it spends between two MMAs can leave the pipe
            // idle: nothing is recomputed per MMA.
            const uint64_t qdesc0 = tc::sw128_desc(sbase + kQOff, 16, 1024);
            const uint64_t kdesc0 = tc::sw128_desc(sbase + kKOff, 16, 1024);
            const uint64_t vdesc0 = tc::sw128_desc(sbase + kVOff, kHalfBytes, 1024);
            bool ok = mbar_wait_bounded(&bars->q_full, 0, abort_flag, p.wait_ns);
            tc::fence_after_sync();
            for (int j = 0; ok && j <= nk; ++j) {
                const int st = j % kKStages;
                if (j < nk) {
                    ok = mbar_wait_bounded(&bars->k_full[st], (j / kKStages) & 1, abort_flag, p.wait_ns);
                    if (!ok)
                        break;
                    tc::fence_after_sync();
                }
                bool v_ready = false;
                for (int t = 0; t < 2 && ok; ++t) {
                    const int diag = t == 0 ? diag0 : diag1;
                    const bool t_active = t == 0 || active1;
                    const uint32_t s_tmem = tmem + t * kBN;
                    const uint32_t o_tmem = tmem + 2 * kBN + t * kHD;
                    if (j > 0 && t_active && j - 1 <= diag) {
                        // O_t += P_t(j-1) V_{j-1}
                        ok = mbar_wait_bounded(&bars->p_full[t], (j - 1) & 1, abort_flag, p.wait_ns);
                        if (ok && !v_ready) {
                            ok = mbar_wait_bounded(&bars->v_conv[(j - 1) % kVStages], ((j - 1) / kVStages) & 1,
                                                   abort_flag, p.wait_ns);
                            v_ready = true;
                        }
                        if (!ok)
                            break;
                        tc::fence_after_sync();
                        const uint64_t vdesc = vdesc0 + (uint64_t)(((j - 1) % kVStages) * (kTileBytes >> 4));
                        // B = V rows [16kk, 16kk+16): MN-major, the two
                        // 64-column halves are 16 KiB apart (LBO), 8-key
                        // groups 1 KiB apart (SBO).
                        mma_ts_x8(o_tmem, s_tmem, vdesc, kIdescPV, j - 1 > 0 ? 1u : 0u);
                        if (j > diag)
                            tc::commit(&bars->o_full[t]);  // last PV of this tile
                    }
                    if (j < nk && t_active && j <= diag) {
                        // S_t = Q_t K_j^T
                        const uint64_t qdesc = qdesc0 + (uint64_t)(t * (kTileBytes >> 4));
                        const uint64_t kdesc = kdesc0 + (uint64_t)(st * (kTileBytes >> 4));
                        mma_ss_x8(s_tmem, qdesc, kdesc, kIdescS, 0u);
                        tc::commit(&bars->s_full[t]);
                    }
                }
                if (!ok)
                    break;
                if (j < nk)
                    tc::commit(&bars->k_empty[st]);  // S of tile j issued for both query tiles
                if (j > 0)
                    tc::commit(&bars->v_empty[(j - 1) % kVStages]);  // and PV of tile j - 1
            }
            // Every MMA this thread issued completes before the TMEM is freed.
            tc::commit(&bars->mma_done);
            int drain_abort = 0;
            mbar_wait_bounded(&bars->mma_done, 0, &drain_abort);
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        // ------------------------------------------------------------ V bf16 -> fp16
        const int ct = threadIdx.x - kConvWarp0 * 32;
        uint32_t vmax = 0;  // largest |v| bit pattern seen, per 16-bit half
        for (int j = 0; j < nk; ++j) {
            const int st = j % kVStages;
            bool ok = mbar_wait_bounded(&bars->v_full[st], (j / kVStages) & 1, abort_flag, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            uint4 *vt = reinterpret_cast<uint4 *>(smem + kVOff + st * kTileBytes);
#pragma unroll 4
            for (int i = ct; i < (int)(kTileBytes / 16); i += kConvThreads) {
                uint4 w = vt[i];
                vmax = __vmaxu2(vmax, w.x & 0x7fff7fffu);
                vmax = __vmaxu2(vmax, w.y & 0x7fff7fffu);
                vmax = __vmaxu2(vmax, w.z & 0x7fff7fffu);
                vmax = __vmaxu2(vmax, w.w & 0x7fff7fffu);
                w.x = tc::bf16x2_to_f16x2(w.x);
                w.y = tc::bf16x2_to_f16x2(w.y);
                w.z = tc::bf16x2_to_f16x2(w.z);
                w.w = tc::bf16x2_to_f16x2(w.w);
                vt[i] = w;
            }
            // generic-proxy writes, read next by the tensor cores (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&bars->v_conv[st]);
        }
        if ((vmax & 0xffffu) > 0x477fu || (vmax >> 16) > 0x477fu)
            atomicOr(p.status, TA_DEVERR_RANGE);
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = warp >> 2;  // query tile
        const int r = threadIdx.x & (kBM - 1);
        const int qrow0 = q0 + t * kBM;
        if (qrow0 < L) {
            const int diag = qrow0 / kBN;
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t s_tmem = tmem + lane_base + t * kBN;
            const uint32_t o_tmem = tmem + lane_base + 2 * kBN + t * kHD;
            const float c = p.c;
            // l: the row sum of the weights as computed (for lse); lr: the
            // same weights as rounded to fp16, the values the PV product
            // multiplies (for the normalisation of O, so that the output is
            // a weighted mean whose weights sum to one exactly)
            float m_used = -INFINITY, l = 0.f, lr = 0.f;
            bool ok = true;
            for (int j = 0; j <= diag; ++j) {
                ok = mbar_wait_bounded(&bars->s_full[t], j & 1, abort_flag, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc::fence_after_sync();
                // all four TMEM loads in flight before the first wait
                uint32_t u[4][32];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    tc::tmem_ld32(s_tmem + ch * 32, u[ch]);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    tc::tmem_wait_ld(u[ch]);
                float s[kBN];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        s[ch * 32 + i] = __uint_as_float(u[ch][i]);
                if (j == diag) {
#pragma unroll
                    for (int i = 0; i < kBN; ++i)
                        if (i > r)
                            s[i] = -INFINITY;
                }
                // row maximum: four chains of three-input max
                float mq[4] = {fmaxf(s[0], s[1]), fmaxf(s[2], s[3]), fmaxf(s[4], s[5]), fmaxf(s[6], s[7])};
#pragma unroll
                for (int i = 8; i < kBN; i += 8) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        mq[c] = fmax3(mq[c], s[i + 2 * c], s[i + 2 * c + 1]);
                }
                const float mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
                const float mcand = mx * c;
                const bool resc = mcand > m_used + kRescaleLog2;
                float alpha = 1.f;
                if (resc) {
                    alpha = fast_exp2(m_used - mcand);
                    m_used = mcand;
                }
                // two columns at a time in packed fp32 pairs: the exponent
                // s * scale * log2(e) - m, then the sum of the weights
                const uint64_t c2 = f2_pack(c, c), negm2 = f2_pack(-m_used, -m_used);
                uint64_t ls2 = f2_pack(0.f, 0.f);
                float lsr[2] = {0.f, 0.f};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 e = f2_unpack(
                            f2_fma(f2_pack(s[half * 64 + 2 * i], s[half * 64 + 2 * i + 1]), c2, negm2));
                        const float p0 = fast_exp2(e.x);
                        const float p1 = fast_exp2(e.y);
                        const uint32_t w = tc::pack_f16x2(p0, p1);
                        pk[i] = w;
                        ls2 = f2_add(ls2, f2_pack(p0, p1));
                        lsr[i & 1] = add_f16x2(lsr[i & 1], w);
                    }
                    tc::tmem_st32(s_tmem + half * 32, pk);
                }
                const float2 ls = f2_unpack(ls2);
                l = l * alpha + (ls.x + ls.y);
                lr = lr * alpha + (lsr[0] + lsr[1]);
                if (j > 0 && __any_sync(0xffffffffu, resc)) {
                    // O_t holds every PV up to j-1 (see the MMA issuer);
                    // bring it to the new reference.
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t ou[2][32];
#pragma unroll
                        for (int ch = 0; ch < 2; ++ch)
                            tc::tmem_ld32(o_tmem + (2 * half + ch) * 32, ou[ch]);
#pragma unroll
                        for (int ch = 0; ch < 2; ++ch) {
                            tc::tmem_wait_ld(ou[ch]);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                ou[ch][i] = __float_as_uint(__uint_as_float(ou[ch][i]) * alpha);
                            tc::tmem_st32(o_tmem + (2 * half + ch) * 32, ou[ch]);
                        }
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                mbar_arrive(&bars->p_full[t]);
            }
            if (ok) {
                ok = mbar_wait_bounded(&bars->o_full[t], 0, abort_flag, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok) {
                tc::fence_after_sync();
                const int row = qrow0 + r;
                const float inv = 1.0f / lr;
                // output row: [b*H + h][S][D] batched, [T][H][D] packed; lse
                // [b*H + h][S] batched, [H][T] packed
                OUT *const obase = static_cast<OUT *>(p.out);
                OUT *orow = p.cu_seqlens ? obase + ((size_t)(y0 + row) * p.H + zq) * kHD
                                         : obase + ((size_t)bh * p.S + row) * kHD;
                const size_t lse_at = p.cu_seqlens ? (size_t)zq * p.T + y0 + row : (size_t)bh * p.S + row;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t u[32];
                    tc::tmem_ld32(o_tmem + ch * 32, u);
                    tc::tmem_wait_ld(u);
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __uint_as_float(u[i]) * inv;
                    if (row < L) {
                        // streaming stores: the output is not read again here,
                        // so its lines leave L2 first instead of lingering dirty
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
                        if constexpr (sizeof(OUT) == 2) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                __stcs(dst + i, out_pack4(o + 8 * i, (__nv_bfloat16 *)nullptr));
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                __stcs(dst + i, make_uint4(__float_as_uint(o[4 * i]), __float_as_uint(o[4 * i + 1]),
                                                           __float_as_uint(o[4 * i + 2]),
                                                           __float_as_uint(o[4 * i + 3])));
                        }
                    }
                }
                if (row < L && p.lse)
                    __stcs(p.lse + lse_at, (m_used + fast_log2(l)) * kLn2);
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.status, TA_DEVERR_TIMEOUT);
    if (warp == kProducerWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host

// 3-D map over a [rows3, S, D] bf16 tensor, box {64, 128, 1}, 128-byte
// swizzle; out-of-range rows read as zero.
bool make_map(CUtensorMap *m, const void *base, int S, int rows3)
{
    const uint64_t dims[3] = {(uint64_t)kHD, (uint64_t)S, (uint64_t)rows3};
    const uint64_t strides[2] = {(uint64_t)kHD * 2, (uint64_t)S * kHD * 2};
    const uint32_t box[3] = {64, (uint32_t)kBM, 1};
    return encode_tmap_3d(m, base, true, dims, strides, box, true);
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch &a)
{
    if (a.D != kHD)
        return cudaErrorNotSupported;
    if (cudaError_t inj = injected_launch_failure())
        return inj;
    PrefillParams p;
    if (!a.cu_seqlens) {
        if (!make_map(&p.qmap, a.q, a.S, a.B * a.H) || !make_map(&p.kmap, a.k, a.S, a.B * a.Hkv) ||
            !make_map(&p.vmap, a.v, a.S, a.B * a.Hkv))
            return cudaErrorInvalidValue;
    } else {
        // the packed tensors as {D, T, heads}: token stride heads * D, head stride D
        const uint64_t qdims[3] = {(uint64_t)kHD, (uint64_t)a.T, (uint64_t)a.H};
        const uint64_t qstr[2] = {(uint64_t)a.H * kHD * 2, (uint64_t)kHD * 2};
        const uint64_t kdims[3] = {(uint64_t)kHD, (uint64_t)a.T, (uint64_t)a.Hkv};
        const uint64_t kstr[2] = {(uint64_t)a.Hkv * kHD * 2, (uint64_t)kHD * 2};
        const uint32_t box[3] = {64, (uint32_t)kBM, 1};
        if (!encode_tmap_3d(&p.qmap, a.q, true, qdims, qstr, box, true) ||
            !encode_tmap_3d(&p.kmap, a.k, true, kdims, kstr, box, true) ||
            !encode_tmap_3d(&p.vmap, a.v, true, kdims, kstr, box, true))
            return cudaErrorInvalidValue;
    }
    p.out = a.out;
    p.lse = a.lse;
    p.S = a.S;  // packed: max_seqlen
    p.H = a.H;
    p.G = a.H / a.Hkv;
    p.n_qt = (a.S + 2 * kBM - 1) / (2 * kBM);
    p.BH = a.B * a.H;  // packed: B = number of sequences
    p.c = a.scale * kLog2e;
    p.status = a.status;
    p.cu_seqlens = a.cu_seqlens;
    p.T = a.cu_seqlens ? a.T : 0;
    p.wait_ns = a.wait_ns;
    p.test_stall = a.test_stall;
    auto kern = a.out_dtype == TA_F32 ? prefill_causal_kernel<float> : prefill_causal_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess)
        return e;
    const long long grid = (long long)p.n_qt * p.BH;
    kern<<<(unsigned)grid, kThreads, kSmemBytes, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ta
