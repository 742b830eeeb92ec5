// combine.cu -- log-sum-exp tree merge of split-KV partials.
//
// The Tree Attention explainer (aibr.jp/archives/143699, sections 1 and 3)
// reduces attention along the sequence axis as an associative tree of
// log-sum-exp merges.  On one GPU the tree is: one warp merges up to 64
// partials of a row; when a row has more, a first level of warps merges
// groups of 64 into intermediate partials and a further launch merges
// those, and so on.  For partials (m_i, l_i, o_i), natural-log units:
//   m* = max_i m_i,  l* = sum_i l_i e^(m_i - m*),  o* = sum_i o_i e^(m_i - m*)
// An intermediate level writes (m*, l*, o*); the last level writes
// out = o* / l* and lse = m* + ln l*.  An empty partial (m = -inf) has
// weight 0; a row with only empty partials gives out = 0, lse = -inf.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ta {
namespace {

constexpr int kWarpsPerBlock = 4;

__device__ __forceinline__ void store_val(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_val(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// One warp per (row r, group gi) merging partials [gi*group, min(N, (gi+1)*group)).
template <int D, typename OUT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) combine_kernel(
    const float *__restrict__ m, const float *__restrict__ l, const float *__restrict__ o, int R, int N, int group,
    int n_groups, OUT *__restrict__ out, float *__restrict__ lse, float *__restrict__ m2, float *__restrict__ l2,
    float *__restrict__ o2)
{
    constexpr int DPL = D / 32;  // dims per lane (2 or 4)
    constexpr unsigned kFull = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (wid >= (long long)R * n_groups)
        return;
    const int r = (int)(wid / n_groups);
    const int gi = (int)(wid - (long long)r * n_groups);
    const int i0 = gi * group;
    const int i1 = min(N, i0 + group);
    const float *mr = m + (size_t)r * N;
    const float *lr = l + (size_t)r * N;
    const float *orow = o + (size_t)r * N * D;

    float mx = -INFINITY;
    for (int i = i0 + lane; i < i1; i += 32)
        mx = fmaxf(mx, mr[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));

    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e)
        acc[e] = 0.f;
    float lsum = 0.f;
    if (mx != -INFINITY) {
        for (int base = i0; base < i1; base += 32) {
            const int i = base + lane;
            float w = 0.f;
            if (i < i1) {
                const float mi = mr[i];
                w = mi == -INFINITY ? 0.f : __expf(mi - mx);
                lsum = fmaf(w, lr[i], lsum);
            }
            const int cnt = min(32, i1 - base);
#pragma unroll 4
            for (int j = 0; j < cnt; ++j) {
                const float wj = __shfl_sync(kFull, w, j);
                const float *src = orow + (size_t)(base + j) * D + lane * DPL;
                if constexpr (DPL == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    acc[0] = fmaf(wj, v.x, acc[0]);
                    acc[1] = fmaf(wj, v.y, acc[1]);
                    acc[2] = fmaf(wj, v.z, acc[2]);
                    acc[3] = fmaf(wj, v.w, acc[3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[0] = fmaf(wj, v.x, acc[0]);
                    acc[1] = fmaf(wj, v.y, acc[1]);
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        lsum += __shfl_xor_sync(kFull, lsum, off);

    if (n_groups == 1) {
        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            store_val(out + (size_t)r * D + lane * DPL + e, acc[e] * inv);
        if (lane == 0 && lse)
            lse[r] = lsum > 0.f ? mx + logf(lsum) : -INFINITY;
    } else {
        const size_t pi = (size_t)r * n_groups + gi;
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            o2[pi * D + lane * DPL + e] = acc[e];
        if (lane == 0) {
            m2[pi] = mx;
            l2[pi] = lsum;
        }
    }
}

template <int D, typename OUT>
cudaError_t run_levels(const float *m, const float *l, const float *o, int R, int N, void *out, float *lse,
                       void *scratch, cudaStream_t stream)
{
    // scratch: two ping-pong (m, l, o) buffers sized for the first level.
    const long long n1 = (N + kFanin - 1) / kFanin;
    auto align = [](long long x) { return (x + 255) / 256 * 256; };
    const long long ml_bytes = align(4 * (long long)R * n1);
    const long long o_bytes = align(4 * (long long)R * n1 * D);
    const long long one = 2 * ml_bytes + o_bytes;
    char *base = static_cast<char *>(scratch);
    const float *sm = m, *sl = l, *so = o;
    int n = N;
    int buf = 0;
    for (;;) {
        const int n_groups = n <= kFanin ? 1 : (n + kFanin - 1) / kFanin;
        const int group = n_groups == 1 ? n : kFanin;
        const long long warps = (long long)R * n_groups;
        const unsigned blocks = (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
        float *dm = nullptr, *dl = nullptr, *dout = nullptr;
        if (n_groups > 1) {
            char *p = base + buf * one;
            dm = reinterpret_cast<float *>(p);
            dl = reinterpret_cast<float *>(p + ml_bytes);
            dout = reinterpret_cast<float *>(p + 2 * ml_bytes);
        }
        combine_kernel<D, OUT><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(
            sm, sl, so, R, n, group, n_groups, static_cast<OUT *>(out), lse, dm, dl, dout);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || n_groups == 1)
            return e;
        sm = dm;
        sl = dl;
        so = dout;
        n = n_groups;
        buf ^= 1;
    }
}

}  // namespace

cudaError_t launch_combine(const float *m, const float *l, const float *o, int R, int N, int D, void *out,
                           ta_dtype out_dtype, float *lse, void *scratch, cudaStream_t stream)
{
    if (cudaError_t inj = injected_launch_failure())
        return inj;
    if (D == 128)
        return out_dtype == TA_BF16 ? run_levels<128, __nv_bfloat16>(m, l, o, R, N, out, lse, scratch, stream)
                                    : run_levels<128, float>(m, l, o, R, N, out, lse, scratch, stream);
    if (D == 64)
        return out_dtype == TA_BF16 ? run_levels<64, __nv_bfloat16>(m, l, o, R, N, out, lse, scratch, stream)
                                    : run_levels<64, float>(m, l, o, R, N, out, lse, scratch, stream);
    return cudaErrorInvalidValue;
}

}  // namespace ta
