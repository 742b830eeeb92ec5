// decode_tc_common.cuh -- the end of a work item, shared by the two
// tensor-core decodes (decode_tc.cu: bf16 cache; decode_fp8_tc.cu: E4M3
// and NVFP4 caches).
//
// Both kernels run a warpgroup of four softmax warps; warp w keeps, for
// each of the G query heads of the item's KV head, its own running
// reference mw (log2 units), weight sum l_run and, per thread (output
// dimension `row`), the four warps' unnormalised outputs o[w][g].  At the
// end of an item these are merged by the log-sum-exp rule (Tree Attention
// explainer, aibr.jp/archives/143699, sections 1 and 3: the reduction along
// the sequence axis is associative) into the item's partial (m, l, o), which
// is either the result (one chunk), or written to the partials, and in
// fused mode the CTA that writes a unit's last partial merges all of them
// (learning that it is the last one item later, so no item waits for it).
// Which CTA that is comes from a GPU-scope acquire-release increment of
// the unit's counter, which stalls its thread for about a microsecond: a
// warp of its own (the ticket thread) takes it, off the softmax warps' path.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ta {
namespace tcd {

constexpr int kD = 128;
constexpr int kSoftThreads = 128;
constexpr unsigned kFull = 0xffffffffu;

enum : int { kModeFinal = 0, kModePartials = 1, kModeFused = 2 };

__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Where an item's result goes.
struct ItemOut {
    void *out;       // [B*Hq, D] OUT
    float *lse;      // [B*Hq] or nullptr
    int Hq;
    int mode;
    int n_split;
    float *part_m, *part_l, *part_o;  // [R, n_split], [R, n_split], [R, n_split, D]
    int32_t *counters;                // [B*Hkv] finished chunks per unit (fused mode)
    volatile int *abort;              // the launch's give-up flag
    uint64_t wait_ns;                 // time limit of a pipeline wait
};

template <int G>
constexpr int stage_floats() { return G * kFusedMergeMaxSplits + 2 * G; }

// Shared memory of the item end: the four warps' sums and references, the
// ticket channel to the ticket thread, the decision of a deferred ticket
// (below), and the merge's area for the weights of the partials.  (The area
// is its own: the weight buffers of the value product are not free for it,
// since the entries of a warp's rows outside its own 32 keys must stay
// zero.)
struct ItemSmem {
    uint64_t tk_req;   // a ticket asked for: the 128 softmax threads, each after its partial stores
    uint64_t tk_done;  // the ticket is taken and its result is in tk_old (the ticket thread)
    uint64_t mg_bar;   // the last merge's partial outputs landed (one bulk copy, phase 0 only)
    float lred[4][4];  // [warp][head] weight sums
    float mred[4][4];  // [warp][head] references
    int merge_unit;    // unit whose partials are all written (-1: none)
    int tk_unit;       // the unit of the ticket asked for; -1: no more tickets
    int tk_old;        // the unit counter's value before the ticket's increment
    float stage[stage_floats<4>()];
};

// Called by one thread before the kernel's first __syncthreads.
__device__ __forceinline__ void init_item_smem(ItemSmem *sm)
{
    mbar_init(&sm->tk_req, kSoftThreads);
    mbar_init(&sm->tk_done, 1);
    mbar_init(&sm->mg_bar, 1);
    sm->merge_unit = -1;
    sm->tk_unit = -1;
}

// A ticket asked for and not yet looked at (kept by softmax thread 0).  In
// fused mode the CTA that writes a unit's last partial merges that unit;
// the ticket says whether this CTA's was the last.  Its result is read at
// the next item's end (or after the last item), so no item waits for it.
struct PendingTicket {
    int unit = -1;   // -1: none pending
    uint32_t n = 0;  // tickets asked for so far (the phase of tk_done)
};

// The ticket thread (one thread of an otherwise idle warp, fused mode
// only): for each ticket asked for, the acquire-release increment of the
// unit's counter.  The 128 arrivals on tk_req order every softmax thread's
// partial stores before the increment (whose release publishes them to the
// merging CTA); its acquire, passed on through tk_done, orders the other
// CTAs' partials before this CTA's merge reads them.  Its waits last as long
// as an item, so they are bounded by the larger of the launch's limit and
// the default, and end early when the launch gives up.
__device__ __forceinline__ void ticket_loop(const ItemOut &io, ItemSmem *sm)
{
    const uint64_t limit = io.wait_ns > kWaitLimitNs ? io.wait_ns : kWaitLimitNs;
    for (uint32_t n = 0;; ++n) {
        if (!mbar_wait_bounded(&sm->tk_req, n & 1, io.abort, limit))
            return;
        const int u = *reinterpret_cast<volatile int *>(&sm->tk_unit);
        if (u < 0)
            return;
        sm->tk_old = atomic_add_acq_rel_gpu(&io.counters[u], 1);
        mbar_arrive(&sm->tk_done);
    }
}

// The merge of a unit whose partials are all written: out = sum_n e^(m_n -
// max) o_n / sum_n e^(m_n - max) l_n, lse = max + ln(that sum), over the
// unit's ns partials of each of its G heads.  Warp h loads head h's
// references (natural log) and sums and turns them into weights (kept in
// shared memory) and the weighted sum; every thread adds its 4 output
// dimensions of all ns partials, kBatch independent loads a round (as many
// as the kernel's register budget allows), the first round issued before
// the weights are known.
//
// After the CTA's last item its copy ring is idle: there (bulk != nullptr,
// room for the G x ns partial outputs) the outputs come by one bulk copy
// into shared memory, issued before the weights are computed, instead of
// rounds of loads.
template <int G, typename OUT, int kBatch, typename Sync>
__device__ __forceinline__ bool merge_unit(const ItemOut &io, ItemSmem *sm, float *stage, int q4, int lane,
                                           size_t row0, Sync &&group_sync, unsigned char *bulk = nullptr)
{
    const int row = q4 * 32 + lane;
    const int ns = io.n_split;
    constexpr int kCols = G * kD / 4;  // output columns of 4 dimensions
    static_assert(kCols <= kSoftThreads && kFusedMergeMaxSplits <= 128, "one column a thread, 4 partials a lane");

    float *sw = stage;          // [G][ns] weights
    float *shd = stage + G * ns; // [G][2] maximum, weighted sum
    // Thread `row` owns column `row` (head h, dimensions d4 .. d4 + 3).  Its
    // first kBatch partial outputs are loaded before the weights are known,
    // so that round trip overlaps the one of the references.
    const bool has_col = row < kCols;
    const int h = row / (kD / 4);
    const int d4 = (row - h * (kD / 4)) * 4;
    const float4 *po = reinterpret_cast<const float4 *>(io.part_o + (row0 + h) * ns * kD + d4);
    float4 x[kBatch];
    if (bulk) {
        if (row == 0) {
            // The copy runs in the async proxy: this fence orders before it the
            // ring's last generic-proxy accesses and the other CTAs' partial
            // stores, which the ticket's acquire made visible to this thread.
            asm volatile("fence.proxy.async;" ::: "memory");
            const uint32_t bytes = (uint32_t)(G * ns * kD * sizeof(float));
            mbar_arrive_expect_tx(&sm->mg_bar, bytes);
            bulk_copy_g2s(bulk, io.part_o + row0 * ns * kD, bytes, &sm->mg_bar);
        }
    } else if (has_col) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            x[i] = i < ns ? __ldcg(po + (size_t)i * (kD / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // warp q4 < G: head q4's references and sums (at most four a lane) ->
    // its maximum, the weights e^(m_n - max) and the weighted sum of l_n
    if (q4 < G) {
        const size_t base = (row0 + q4) * ns;
        float mv[4], lv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int n = lane + 32 * k;
            mv[k] = n < ns ? __ldcg(io.part_m + base + n) : -INFINITY;
            lv[k] = n < ns ? __ldcg(io.part_l + base + n) : 0.f;
        }
        float mx = fmax3(mv[0], mv[1], fmaxf(mv[2], mv[3]));
#pragma unroll
        for (int mask = 16; mask >= 1; mask >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mask));
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int n = lane + 32 * k;
            const float a = mv[k] == -INFINITY ? 0.f : fast_exp2((mv[k] - mx) * kLog2e);
            if (n < ns)
                sw[q4 * ns + n] = a;
            lsum = fmaf(a, lv[k], lsum);
        }
#pragma unroll
        for (int mask = 16; mask >= 1; mask >>= 1)
            lsum += __shfl_xor_sync(kFull, lsum, mask);
        if (lane == 0) {
            shd[2 * q4] = mx;
            shd[2 * q4 + 1] = lsum;
        }
    }
    if (!group_sync())
        return false;
    if (bulk && !mbar_wait_bounded(&sm->mg_bar, 0, io.abort, io.wait_ns))
        return false;
    if (has_col && bulk) {
        const float *wh = sw + h * ns;
        const float4 *so = reinterpret_cast<const float4 *>(bulk) + h * ns * (kD / 4) + d4 / 4;
        float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int n = 0; n < ns; ++n) {
            const float4 y = so[n * (kD / 4)];
            const float a = wh[n];
            os.x = fmaf(a, y.x, os.x);
            os.y = fmaf(a, y.y, os.y);
            os.z = fmaf(a, y.z, os.z);
            os.w = fmaf(a, y.w, os.w);
        }
        const float mx = shd[2 * h], lsum = shd[2 * h + 1];
        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
        OUT *dst = static_cast<OUT *>(io.out) + (row0 + h) * kD + d4;
        store_out(dst + 0, os.x * inv);
        store_out(dst + 1, os.y * inv);
        store_out(dst + 2, os.z * inv);
        store_out(dst + 3, os.w * inv);
        if (d4 == 0 && io.lse)
            io.lse[row0 + h] = lsum > 0.f ? mx + fast_log2(lsum) * kLn2 : -INFINITY;
    } else if (has_col) {
        const float *wh = sw + h * ns;
        float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int n0 = 0;;) {
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const float a = n0 + i < ns ? wh[n0 + i] : 0.f;
                os.x = fmaf(a, x[i].x, os.x);
                os.y = fmaf(a, x[i].y, os.y);
                os.z = fmaf(a, x[i].z, os.z);
                os.w = fmaf(a, x[i].w, os.w);
            }
            n0 += kBatch;
            if (n0 >= ns)
                break;
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                x[i] = n0 + i < ns ? __ldcg(po + (size_t)(n0 + i) * (kD / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float mx = shd[2 * h], lsum = shd[2 * h + 1];
        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
        OUT *dst = static_cast<OUT *>(io.out) + (row0 + h) * kD + d4;
        store_out(dst + 0, os.x * inv);
        store_out(dst + 1, os.y * inv);
        store_out(dst + 2, os.z * inv);
        store_out(dst + 3, os.w * inv);
        if (d4 == 0 && io.lse)
            io.lse[row0 + h] = lsum > 0.f ? mx + fast_log2(lsum) * kLn2 : -INFINITY;
    }
    // the staging area is read above; the softmax warps write the next tile's
    // weights to the same buffers only after this rendezvous
    return group_sync();
}

// Thread 0 publishes the decision of its pending ticket (called before a
// rendezvous, after which every thread reads sm->merge_unit).  If the wait
// for the ticket gives up, the launch's give-up flag is set and no merge is
// made.
__device__ __forceinline__ void publish_ticket(const ItemOut &io, ItemSmem *sm, int row, PendingTicket &pt)
{
    if (row != 0)
        return;
    int u = -1;
    if (pt.unit >= 0) {
        if (mbar_wait_bounded(&sm->tk_done, (pt.n - 1) & 1, io.abort, io.wait_ns) &&
            *reinterpret_cast<volatile int *>(&sm->tk_old) == io.n_split - 1) {
            u = pt.unit;
            io.counters[u] = 0;  // ready for the next launch
        }
        pt.unit = -1;
    }
    sm->merge_unit = u;
}

// After the softmax warpgroup's last item (every thread, fused mode): tells
// the ticket thread that no ticket follows.  The last ticket has been read
// by then (finish_pending), so tk_unit is free.
__device__ __forceinline__ void end_tickets(ItemSmem *sm, int row)
{
    if (row == 0)
        *reinterpret_cast<volatile int *>(&sm->tk_unit) = -1;
    mbar_arrive(&sm->tk_req);
}

// The end of an item for softmax thread `row` (warp q4 of the warpgroup):
// the four warps' states merged into the item's partial, which is the
// result (one chunk) or is written to the partials; a unit whose partials
// a deferred ticket found complete is merged; in fused mode this item's
// ticket is taken (and left pending).  vscale multiplies the partial's
// output (a value dequantisation factor, 1 for bf16 caches).  group_sync()
// is a rendezvous of the four warps that returns false when the launch gave
// up.  Returns false on give-up.
template <int G, typename OUT, int kBatch, typename Sync>
__device__ __forceinline__ bool finish_item(const ItemOut &io, ItemSmem *sm, float *stage, int q4, int lane, int unit,
                                            int split, int b, int kvh, float vscale, const float (&mw)[G],
                                            const float (&l_run)[G], const float (&o)[4][G], PendingTicket &pt,
                                            Sync &&group_sync)
{
    const int row = q4 * 32 + lane;
    // the four warps' states, merged
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float v = l_run[g];
#pragma unroll
        for (int mask = 16; mask >= 1; mask >>= 1)
            v += __shfl_xor_sync(kFull, v, mask);
        if (lane == g) {
            sm->lred[q4][g] = v;
            sm->mred[q4][g] = mw[g];
        }
    }
    if (io.mode == kModeFused)
        publish_ticket(io, sm, row, pt);
    if (!group_sync())
        return false;
    float ls[G], mt[G], of[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        mt[g] = fmax3(sm->mred[0][g], sm->mred[1][g], fmaxf(sm->mred[2][g], sm->mred[3][g]));
        ls[g] = 0.f;
        of[g] = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
            const float m2 = sm->mred[w2][g];
            const float be = m2 == -INFINITY ? 0.f : fast_exp2(m2 - mt[g]);
            ls[g] = fmaf(sm->lred[w2][g], be, ls[g]);
            of[g] = fmaf(o[w2][g], be, of[g]);
        }
        of[g] *= vscale;
    }
    const size_t row0 = (size_t)b * io.Hq + (size_t)kvh * G;
    if (io.mode == kModeFinal) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float inv = ls[g] > 0.f ? 1.0f / ls[g] : 0.f;
            store_out(static_cast<OUT *>(io.out) + (row0 + g) * kD + row, of[g] * inv);
            if (row == g && io.lse)
                io.lse[row0 + g] = ls[g] > 0.f ? (mt[g] + fast_log2(ls[g])) * kLn2 : -INFINITY;
        }
        return true;
    }
    const int ns = io.n_split;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const size_t pi = (row0 + g) * ns + split;
        io.part_o[pi * kD + row] = of[g];
        if (row == g) {
            io.part_m[pi] = mt[g] == -INFINITY ? -INFINITY : mt[g] * kLn2;
            io.part_l[pi] = ls[g];
        }
    }
    if (io.mode != kModeFused)
        return true;
    // the unit an earlier ticket found complete (read after the rendezvous)
    const int mu = *reinterpret_cast<volatile int *>(&sm->merge_unit);
    // (unit u = b * Hkv + kvh has output rows u * G .. u * G + G - 1)
    if (mu >= 0 && !merge_unit<G, OUT, kBatch>(io, sm, stage, q4, lane, (size_t)mu * G, group_sync))
        return false;
    // This item's ticket: thread 0 names the unit and every thread arrives
    // after its own partial stores; the ticket thread takes it.  Its result
    // is read at the next item's end.
    if (row == 0) {
        *reinterpret_cast<volatile int *>(&sm->tk_unit) = unit;
        pt.unit = unit;
        ++pt.n;
    }
    mbar_arrive(&sm->tk_req);
    return true;
}

// After the last item: the decision of the last pending ticket, and its
// merge (through `ring`, the idle copy ring of ring_bytes, when the unit's
// partial outputs fit there).
template <int G, typename OUT, int kBatch, typename Sync>
__device__ __forceinline__ bool finish_pending(const ItemOut &io, ItemSmem *sm, float *stage, int q4, int lane,
                                               PendingTicket &pt, Sync &&group_sync, unsigned char *ring,
                                               size_t ring_bytes)
{
    if (io.mode != kModeFused)
        return true;
    publish_ticket(io, sm, q4 * 32 + lane, pt);
    if (!group_sync())
        return false;
    const int mu = *reinterpret_cast<volatile int *>(&sm->merge_unit);
    if (mu >= 0) {
        const bool fits = (size_t)G * io.n_split * kD * sizeof(float) <= ring_bytes;
        const bool ok = merge_unit<G, OUT, kBatch>(io, sm, stage, q4, lane, (size_t)mu * G, group_sync,
                                                   fits ? ring : nullptr);
        if (fits) {
            // the copy lands before the CTA leaves, even when the merge gave up
            int drain_abort = 0;
            mbar_wait_bounded(&sm->mg_bar, 0, &drain_abort);
        }
        return ok;
    }
    return true;
}

}  // namespace tcd
}  // namespace ta
