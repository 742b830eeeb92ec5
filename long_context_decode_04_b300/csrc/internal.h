// internal.h -- declarations shared by the host-side files of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ta.h"

namespace ta {

constexpr int kFanin = 64;            // partials merged by one warp per level
constexpr int kStatusBytes = 256;     // status word region at the workspace start
// Keys of one decode tile, the unit the chunks are whole multiples of: 128
// (the MMA's M) for the tensor-core kernels' shapes, D = 128 with G = 2 or 4
// query heads per KV head; 120 (15 warps of 8 keys) for the CUDA-core kernel.
constexpr int kDecodeTileKeysTC = 128;
constexpr int kDecodeTileKeysCC = 120;
inline int decode_tile_keys(int D, int G) { return D == 128 && (G == 2 || G == 4) ? kDecodeTileKeysTC : kDecodeTileKeysCC; }
// A split decode's workspace starts with a fixed control region that no
// other use of the workspace writes: the status word and work-queue counter
// (first 256 bytes), then one chunk counter per (sequence, KV head).
// Every completed launch leaves the region zero.
constexpr int kCtrlBytes = 16384;
constexpr int kMaxFusedUnits = (kCtrlBytes - kStatusBytes) / 4;
// Up to this many chunks per (sequence, KV head), and kMaxFusedUnits units,
// the decode kernel merges the partials itself.
constexpr int kFusedMergeMaxSplits = 128;
// Time limit of a pipeline wait inside the kernels when the caller sets none.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

inline uint64_t wait_limit_or_default(uint64_t ns) { return ns ? ns : kDefaultWaitLimitNs; }

struct DecodeLaunch {
    const void *q, *k, *v;
    void *out;
    float *lse;
    int B, Hq, Hkv, S, D;
    float scale;
    const int32_t *seqlens;
    ta_dtype in_dtype, out_dtype;
    ta_decode_plan plan;
    int32_t *status;       // device status word
    int32_t *counters;     // [B * Hkv] finished chunks per unit, zero between launches
    float *part_m, *part_l, *part_o;   // [R, n_split], [R, n_split], [R, n_split, D]
    bool force_partials;               // write partials even when n_split == 1
    const int32_t *block_table;        // paged KV cache, or nullptr (contiguous [B, Hkv, S, D])
    int page_size, pages_per_seq, num_pages;
    int pi_window, pi_period;          // pi-Attention key set (period 0: every key)
    bool kv_fp8;                       // K/V are e4m3 bytes (q bf16), dequantised by
    const float *k_scale, *v_scale;    //   per (sequence, KV head) factors
    bool kv_nvfp4;                     // K/V are NVFP4 codes [.., D/2] with E4M3 block
    const void *k_bs, *v_bs;           //   scales [.., D/16] (factors as for E4M3)
    uint64_t wait_ns;                  // time limit of a pipeline wait (ns)
    int test_stall;                    // test hook (ta_test_stall_next_launches)
    cudaStream_t stream;
};

// Set the calling thread's message returned by ta_last_error (api.cpp).
void record_error(const std::string &msg);

// The test hook of ta_test_fail_next_launches (api.cpp): called by every
// launcher just before it would launch; cudaErrorLaunchFailure (and no
// launch) while injected failures are pending, else cudaSuccess.
cudaError_t injected_launch_failure();
// The test hook of ta_test_stall_next_launches (api.cpp): 1 while stalled
// launches are pending (the launch's producer then first waits on a barrier
// that nothing completes, so its time limit runs out), else 0.
int injected_stall();

// The argument checks of ta_decode_ex, on their own (api.cpp): TA_OK or the
// status (with its message recorded) that ta_decode_ex would return.
ta_status check_decode_params(const ta_decode_params *p);

// Whether the decode kernel merges a sequence's chunks itself (else a
// separate merge launch follows it).
inline bool decode_merges_itself(int n_split, int units)
{
    return n_split > 1 && n_split <= kFusedMergeMaxSplits && units <= kMaxFusedUnits;
}

// Keys the pi-Attention decode attends at most for caches of up to S keys:
// min(S, window + 1 + ceil(max(0, S - 1 - window) / period)).
inline int64_t pi_max_keys(int64_t S, int64_t window, int64_t period)
{
    const int64_t far = S - 1 - window > 0 ? S - 1 - window : 0;
    const int64_t n = (window + 1 < S ? window + 1 : S) + (far + period - 1) / period;
    return n < S ? n : S;
}

// A 3-D TMA tensor map (tmap.cpp): dims innermost first, strides in bytes
// of dims 1 and 2, box in elements; bf16 or fp32 elements; zero fill out of
// range.  false if the driver entry point or the encoding fails.
bool encode_tmap_3d(CUtensorMap *m, const void *base, bool bf16, const uint64_t dims[3], const uint64_t strides[2],
                    const uint32_t box[3], bool swizzle128);

// The same for one-byte elements (FP8 codes).
bool encode_tmap_3d_u8(CUtensorMap *m, const void *base, const uint64_t dims[3], const uint64_t strides[2],
                       const uint32_t box[3], bool swizzle128);

// Scheduler (sched.cpp).
ta_status plan_decode(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                      int sm_count, ta_decode_plan *plan, const char **why);
size_t combine_scratch_bytes(int R, int N, int D);
bool decode_shape_supported(int D, int G, ta_dtype in_dtype);
int decode_ctas_per_sm();

// Launchers (decode.cu, combine.cu, prefill.cu).  Return cudaGetLastError().
cudaError_t launch_decode(const DecodeLaunch &a);
// The tensor-core decode (decode_tc.cu): bf16 q/K/V in a contiguous cache,
// D = 128, G = 2 or 4; launch_decode hands such launches to it.
bool decode_tc_eligible(const DecodeLaunch &a);
cudaError_t launch_decode_tc(const DecodeLaunch &a);
// The tensor-core decode over an E4M3 cache (decode_fp8_tc.cu): contiguous
// cache, D = 128, G = 2 or 4.
bool decode_fp8_tc_eligible(const DecodeLaunch &a);
cudaError_t launch_decode_fp8_tc(const DecodeLaunch &a);
cudaError_t launch_combine(const float *m, const float *l, const float *o, int R, int N, int D, void *out,
                           ta_dtype out_dtype, float *lse, void *scratch, cudaStream_t stream);
// One causal prefill launch (prefill.cu): batched [B, H, S, D] layouts, or
// packed [T, heads, D] layouts when cu_seqlens is given (B sequences, S =
// the longest).
struct PrefillLaunch {
    const void *q, *k, *v;
    void *out;
    float *lse;
    int B, H, Hkv, S, D;
    float scale;
    const int32_t *cu_seqlens;
    int T;
    ta_dtype out_dtype;
    int32_t *status;
    uint64_t wait_ns;
    int test_stall;
    cudaStream_t stream;
};
cudaError_t launch_prefill(const PrefillLaunch &a);

}  // namespace ta
