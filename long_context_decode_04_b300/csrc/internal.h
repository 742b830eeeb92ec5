// internal.h -- declarations shared by the host-side files of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <cuda_runtime.h>

#include "../../include/ta.h"

namespace ta {

constexpr int kFanin = 64;            // partials merged by one warp per level
constexpr int kStatusBytes = 256;     // status word region at the workspace start

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
    float *part_m, *part_l, *part_o;   // [R, n_split], [R, n_split], [R, n_split, D]
    bool force_partials;               // write partials even when n_split == 1
    cudaStream_t stream;
};

// Set the calling thread's message returned by ta_last_error (api.cpp).
void record_error(const std::string &msg);

// The argument checks of ta_decode_ex, on their own (api.cpp): TA_OK or the
// status (with its message recorded) that ta_decode_ex would return.
ta_status check_decode_params(const ta_decode_params *p);

// Scheduler (sched.cpp).
ta_status plan_decode(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                      int sm_count, ta_decode_plan *plan, const char **why);
size_t combine_scratch_bytes(int R, int N, int D);
bool decode_shape_supported(int D, int G, ta_dtype in_dtype);
int decode_ctas_per_sm();

// Launchers (decode.cu, combine.cu, prefill.cu).  Return cudaGetLastError().
cudaError_t launch_decode(const DecodeLaunch &a);
cudaError_t launch_combine(const float *m, const float *l, const float *o, int R, int N, int D, void *out,
                           ta_dtype out_dtype, float *lse, void *scratch, cudaStream_t stream);
cudaError_t launch_prefill_causal(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                                  int H, int Hkv, int S, int D, float scale, int32_t *status,
                                  cudaStream_t stream);

}  // namespace ta
