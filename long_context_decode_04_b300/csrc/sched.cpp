// sched.cpp -- the KV-chunk scheduler: how many chunks to split each
// (sequence, KV head) into, and how the partials are merged.
//
// Split-KV decode is the one-GPU form of the sequence-axis split of the
// Tree Attention explainer (aibr.jp/archives/143699, sections 1 and 3):
// each chunk is reduced locally and the results are combined by an
// associative tree.  The pages give no rule for the chunk size; the rule
// here keeps every SM busy: the persistent decode kernel runs
// sm_count * ctas_per_sm CTAs, and the chunk count is chosen so that the
// (sequence, KV head, chunk) work items fill those CTAs evenly.  Chunks are
// whole numbers of the decode kernel's tiles (128 keys for the tensor-core
// shapes, 120 for the CUDA-core kernel).
#include <algorithm>
#include <climits>

#include "internal.h"

namespace ta {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int decode_ctas_per_sm() { return 1; }

bool decode_shape_supported(int D, int G, ta_dtype in_dtype)
{
    if (in_dtype != TA_F32 && in_dtype != TA_BF16)
        return false;
    if (D == 64)
        return G == 1 || G == 2 || G == 4 || G == 8;
    if (D == 128)
        return G == 1 || G == 2 || G == 4;
    return false;
}

size_t combine_scratch_bytes(int R, int N, int D)
{
    // Levels write (m, l, o) intermediates into two ping-pong buffers sized
    // for the first level's output, each region 256-byte aligned.
    if (N <= kFanin)
        return 0;
    const int64_t n1 = ceil_div(N, kFanin);
    auto align = [](int64_t x) { return (x + 255) / 256 * 256; };
    const int64_t one = align(4 * (int64_t)R * n1) * 2 + align(4 * (int64_t)R * n1 * D);
    return (size_t)(2 * one);
}

ta_status plan_decode(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                      int sm_count, ta_decode_plan *plan, const char **why)
{
    *why = "";
    if (!plan) {
        *why = "plan pointer is NULL";
        return TA_ERR_INVALID_ARG;
    }
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || D < 1) {
        *why = "B, Hq, Hkv, S and D must all be >= 1";
        return TA_ERR_INVALID_ARG;
    }
    if (Hq % Hkv != 0) {
        *why = "Hq must be a multiple of Hkv";
        return TA_ERR_INVALID_ARG;
    }
    if (sm_count < 1) {
        *why = "sm_count must be >= 1";
        return TA_ERR_INVALID_ARG;
    }
    if (chunk < 0 || n_split < 0) {
        *why = "chunk and n_split overrides must be >= 0";
        return TA_ERR_INVALID_ARG;
    }
    const int64_t units = (int64_t)B * Hkv;           // independent (sequence, KV head) pairs
    const int64_t tile = decode_tile_keys(D, Hq / Hkv);
    const int64_t slots = (int64_t)sm_count * decode_ctas_per_sm();
    auto chunk_for = [&](int64_t ns) {
        // a whole number of the kernel's tiles, at least two
        int64_t c = ceil_div(ceil_div(S, ns), tile) * tile;
        c = std::max<int64_t>(c, 2 * tile);
        return std::min<int64_t>(c, S);
    };
    int64_t c;
    if (chunk > 0) {
        c = std::min<int64_t>(chunk, S);
    } else if (n_split > 0) {
        c = ceil_div(S, std::min<int64_t>(n_split, S));
    } else if (varlen) {
        // Lengths are only known on the device: over-decompose to about four
        // work items per CTA slot so the dynamic item queue balances them.
        c = chunk_for(std::max<int64_t>(1, ceil_div(4 * slots, units)));
    } else {
        // Every item has the same length: pick the chunk count that
        // minimises (waves of items over the CTA slots) x (keys per item +
        // a fixed per-item cost of 64 keys), preferring fewer chunks on ties.
        int64_t best_c = chunk_for(1), best_cost = INT64_MAX;
        const int64_t max_ns = std::min<int64_t>(ceil_div(S, 2 * tile), 8 * ceil_div(slots, units) + 1);
        for (int64_t ns = 1; ns <= std::max<int64_t>(1, max_ns); ++ns) {
            const int64_t cc = chunk_for(ns);
            const int64_t real_ns = ceil_div(S, cc);
            const int64_t waves = ceil_div(units * real_ns, slots);
            const int64_t cost = waves * (cc + 64);
            if (cost < best_cost) {
                best_cost = cost;
                best_c = cc;
            }
        }
        c = best_c;
    }
    const int64_t ns = ceil_div(S, c);
    const int64_t items = units * ns;
    if (items > INT_MAX || (int64_t)B * Hq * ns > INT_MAX / 2) {
        *why = "too many split-KV work items";
        return TA_ERR_INVALID_ARG;
    }
    int levels = 0;
    if (ns > 1 && !decode_merges_itself((int)ns, (int)std::min<int64_t>(units, INT_MAX))) {
        int64_t n = ns;
        levels = 1;
        while (n > kFanin) {
            n = ceil_div(n, kFanin);
            ++levels;
        }
    }
    const int64_t R = (int64_t)B * Hq;
    auto align = [](int64_t x) { return (x + 255) / 256 * 256; };
    int64_t ws = kStatusBytes;  // status word + work-queue counter
    if (ns > 1) {
        ws = kCtrlBytes;  // + the chunk counters
        ws += align(4 * R * ns) * 2 + align(4 * R * ns * D);
        ws += (int64_t)combine_scratch_bytes((int)R, (int)ns, D);
    }
    plan->n_split = (int32_t)ns;
    plan->chunk = (int32_t)c;
    plan->levels = levels;
    plan->fanin = kFanin;
    plan->grid = (int32_t)std::min<int64_t>(items, slots);
    plan->sm_count = sm_count;
    plan->workspace_bytes = (size_t)ws;
    return TA_OK;
}

}  // namespace ta
