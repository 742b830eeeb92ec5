// api.cpp -- the C ABI: argument validation, the library workspace, and
// dispatch to the scheduler and the kernels.  Nothing here computes
// attention; every arithmetic step runs in the CUDA kernels.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace {

thread_local std::string g_error;
thread_local bool g_injected = false;     // the last launch failure came from the test hook
std::atomic<int> g_fail_launches{0};      // launches still to refuse (ta_test_fail_next_launches)
std::atomic<int> g_stall_launches{0};     // launches still to stall (ta_test_stall_next_launches)

ta_status fail(ta_status s, const std::string &msg)
{
    g_error = msg;
    return s;
}

ta_status cuda_fail(cudaError_t e, const char *where)
{
    if (g_injected) {
        g_injected = false;
        return fail(TA_ERR_CUDA, std::string(where) + ": launch not made (failure injected by ta_test_fail_next_launches)");
    }
    return fail(TA_ERR_CUDA, std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// ------------------------------------------------------------------ devices

struct DeviceState {
    int sm_count = 0;
    void *ws = nullptr;
    size_t ws_bytes = 0;
};

std::mutex g_mu;
std::vector<DeviceState> g_devices;

ta_status current_device(int *dev)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    return TA_OK;
}

DeviceState &state_for(int dev)
{
    if ((int)g_devices.size() <= dev)
        g_devices.resize(dev + 1);
    return g_devices[dev];
}

ta_status device_sm_count(int *sms)
{
    int dev;
    ta_status s = current_device(&dev);
    if (s != TA_OK)
        return s;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = state_for(dev);
    if (st.sm_count == 0) {
        int n = 0;
        cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
        st.sm_count = n;
    }
    *sms = st.sm_count;
    return TA_OK;
}

// The library's own per-device workspace, grown on demand.  Growth frees
// the old buffer (cudaFree synchronises the device) and zeroes the new one.
ta_status library_workspace(size_t need, void **ptr)
{
    int dev;
    ta_status s = current_device(&dev);
    if (s != TA_OK)
        return s;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = state_for(dev);
    need = align256(need < 256 ? 256 : need);
    if (st.ws_bytes < need) {
        if (st.ws) {
            cudaError_t e = cudaFree(st.ws);
            st.ws = nullptr;
            st.ws_bytes = 0;
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaFree(workspace)");
        }
        void *p = nullptr;
        cudaError_t e = cudaMalloc(&p, need);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(workspace)");
        e = cudaMemset(p, 0, need);
        if (e == cudaSuccess)
            e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(p);
            return cuda_fail(e, "cudaMemset(workspace)");
        }
        st.ws = p;
        st.ws_bytes = need;
    }
    *ptr = st.ws;
    return TA_OK;
}

ta_status validate_decode(const ta_decode_params *p)
{
    if (!p)
        return fail(TA_ERR_INVALID_ARG, "params pointer is NULL");
    if (!p->q || !p->k || !p->v || !p->out)
        return fail(TA_ERR_INVALID_ARG, "q, k, v and out must be non-NULL");
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->S < 1 || p->D < 1)
        return fail(TA_ERR_INVALID_ARG, "B, Hq, Hkv, S and D must all be >= 1");
    if (p->Hq % p->Hkv != 0)
        return fail(TA_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
    if (p->in_dtype != TA_F32 && p->in_dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARG, "in_dtype must be TA_F32 or TA_BF16");
    if (p->out_dtype != TA_F32 && p->out_dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARG, "out_dtype must be TA_F32 or TA_BF16");
    if (!std::isfinite(p->scale))
        return fail(TA_ERR_INVALID_ARG, "scale must be finite");
    if (p->chunk < 0 || p->n_split < 0)
        return fail(TA_ERR_INVALID_ARG, "chunk and n_split overrides must be >= 0");
    if (!aligned(p->q, 16) || !aligned(p->k, 16) || !aligned(p->v, 16) || !aligned(p->out, 16))
        return fail(TA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if ((p->lse && !aligned(p->lse, 4)) || (p->seqlens && !aligned(p->seqlens, 4)))
        return fail(TA_ERR_INVALID_ARG, "lse and seqlens must be 4-byte aligned");
    if (p->D != 64 && p->D != 128)
        return fail(TA_ERR_UNSUPPORTED, "decode supports head dim D = 64 or 128");
    if (p->in_dtype == TA_F32 && p->out_dtype != TA_F32)
        return fail(TA_ERR_UNSUPPORTED, "fp32 inputs need an fp32 output");
    if (!ta::decode_shape_supported(p->D, p->Hq / p->Hkv, p->in_dtype))
        return fail(TA_ERR_UNSUPPORTED, "query heads per KV head G = " + std::to_string(p->Hq / p->Hkv) +
                                            " is not supported for D = " + std::to_string(p->D) +
                                            " (G in {1,2,4} for D=128, {1,2,4,8} for D=64)");
    const double elems = (double)p->B * p->Hkv * p->S * p->D;
    if (elems > 9.0e18 / 4)
        return fail(TA_ERR_INVALID_ARG, "KV cache size overflows");
    return TA_OK;
}

}  // namespace

void ta::record_error(const std::string &msg) { g_error = msg; }

cudaError_t ta::injected_launch_failure()
{
    int n = g_fail_launches.load();
    while (n > 0) {
        if (g_fail_launches.compare_exchange_weak(n, n - 1)) {
            g_injected = true;
            return cudaErrorLaunchFailure;
        }
    }
    return cudaSuccess;
}

int ta::injected_stall()
{
    int n = g_stall_launches.load();
    while (n > 0)
        if (g_stall_launches.compare_exchange_weak(n, n - 1))
            return 1;
    return 0;
}

ta_status ta::check_decode_params(const ta_decode_params *p) { return validate_decode(p); }

extern "C" {

const char *ta_last_error(void) { return g_error.c_str(); }

int ta_test_fail_next_launches(int count) { return g_fail_launches.exchange(count > 0 ? count : 0); }

int ta_test_stall_next_launches(int count) { return g_stall_launches.exchange(count > 0 ? count : 0); }

ta_status ta_decode_plan_for(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                             int sm_count, ta_decode_plan *plan)
{
    if (sm_count == 0) {
        ta_status s = device_sm_count(&sm_count);
        if (s != TA_OK)
            return s;
    }
    const char *why = "";
    ta_status s = ta::plan_decode(B, Hq, Hkv, S, D, chunk, n_split, varlen, sm_count, plan, &why);
    if (s != TA_OK)
        return fail(s, why);
    return TA_OK;
}

size_t ta_decode_workspace_bytes(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen)
{
    ta_decode_plan plan;
    if (ta_decode_plan_for(B, Hq, Hkv, S, D, chunk, n_split, varlen, 0, &plan) != TA_OK)
        return 0;
    return plan.workspace_bytes;
}

}  // extern "C"

namespace {

// The decode of ta_decode_ex, reading K/V through a block table when one is
// given (block_table != nullptr; p->k, p->v are then the page pools).
ta_status decode_impl(const ta_decode_params *p, const int32_t *block_table, int page_size, int pages_per_seq,
                      int num_pages, int pi_window = 0, int pi_period = 0, bool kv_fp8 = false,
                      const float *k_scale = nullptr, const float *v_scale = nullptr, bool kv_nvfp4 = false,
                      const void *k_bs = nullptr, const void *v_bs = nullptr)
{
    ta_status s;
    ta_decode_plan plan;
    // the chunks cut the list of attended keys: all S of them, or the
    // pi-Attention set's at most pi_max_keys
    const int S_list = pi_period > 0 ? (int)ta::pi_max_keys(p->S, pi_window, pi_period) : p->S;
    s = ta_decode_plan_for(p->B, p->Hq, p->Hkv, S_list, p->D, p->chunk, p->n_split, p->seqlens != nullptr, 0,
                           &plan);
    if (s != TA_OK)
        return s;
    void *ws = p->workspace;
    if (ws) {
        if (!aligned(ws, 256))
            return fail(TA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        if (p->workspace_bytes < plan.workspace_bytes)
            return fail(TA_ERR_WORKSPACE, "workspace too small: need " + std::to_string(plan.workspace_bytes) +
                                              " bytes, got " + std::to_string(p->workspace_bytes));
    } else {
        s = library_workspace(plan.workspace_bytes, &ws);
        if (s != TA_OK)
            return s;
    }
    ta::DecodeLaunch a;
    a.force_partials = false;
    a.block_table = block_table;
    a.page_size = page_size;
    a.pages_per_seq = pages_per_seq;
    a.num_pages = num_pages;
    a.pi_window = pi_window;
    a.pi_period = pi_period;
    a.kv_fp8 = kv_fp8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.kv_nvfp4 = kv_nvfp4;
    a.k_bs = k_bs;
    a.v_bs = v_bs;
    a.wait_ns = ta::wait_limit_or_default(p->wait_limit_ns);
    a.test_stall = ta::injected_stall();
    a.q = p->q;
    a.k = p->k;
    a.v = p->v;
    a.out = p->out;
    a.lse = p->lse;
    a.B = p->B;
    a.Hq = p->Hq;
    a.Hkv = p->Hkv;
    a.S = p->S;
    a.D = p->D;
    a.scale = p->scale;
    a.seqlens = p->seqlens;
    a.in_dtype = p->in_dtype;
    a.out_dtype = p->out_dtype;
    a.plan = plan;
    a.stream = static_cast<cudaStream_t>(p->stream);
    char *base = static_cast<char *>(ws);
    a.status = reinterpret_cast<int32_t *>(base);
    const size_t R = (size_t)p->B * p->Hq, N = (size_t)plan.n_split;
    a.part_m = a.part_l = a.part_o = nullptr;
    a.counters = nullptr;
    char *scratch = nullptr;
    if (N > 1) {
        a.counters = reinterpret_cast<int32_t *>(base + ta::kStatusBytes);
        size_t off = ta::kCtrlBytes;
        a.part_m = reinterpret_cast<float *>(base + off);
        off += align256(4 * R * N);
        a.part_l = reinterpret_cast<float *>(base + off);
        off += align256(4 * R * N);
        a.part_o = reinterpret_cast<float *>(base + off);
        off += align256(4 * R * N * p->D);
        scratch = base + off;
    }
    cudaError_t e = ta::launch_decode(a);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode kernel launch");
    if (N > 1 && !ta::decode_merges_itself(plan.n_split, p->B * p->Hkv)) {
        e = ta::launch_combine(a.part_m, a.part_l, a.part_o, (int)R, (int)N, p->D, p->out, p->out_dtype, p->lse,
                               scratch, a.stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "combine kernel launch");
    }
    return TA_OK;
}

}  // namespace

extern "C" {

ta_status ta_decode_ex(const ta_decode_params *p)
{
    ta_status s = validate_decode(p);
    if (s != TA_OK)
        return s;
    return decode_impl(p, nullptr, 0, 0, 0);
}

ta_status ta_decode_fp8(const ta_decode_params *p, const float *k_scale, const float *v_scale)
{
    ta_status s = validate_decode(p);
    if (s != TA_OK)
        return s;
    if (p->in_dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARG, "fp8 decode takes bf16 queries (in_dtype = TA_BF16)");
    if (p->D != 128)
        return fail(TA_ERR_UNSUPPORTED, "fp8 decode supports head dim D = 128");
    if ((k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
        return fail(TA_ERR_INVALID_ARG, "k_scale and v_scale must be 4-byte aligned");
    return decode_impl(p, nullptr, 0, 0, 0, 0, 0, true, k_scale, v_scale);
}

ta_status ta_decode_nvfp4(const ta_decode_params *p, const void *k_block_scales, const void *v_block_scales,
                          const float *k_factor, const float *v_factor)
{
    ta_status s = validate_decode(p);
    if (s != TA_OK)
        return s;
    if (p->in_dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARG, "NVFP4 decode takes bf16 queries (in_dtype = TA_BF16)");
    if (!k_block_scales || !v_block_scales)
        return fail(TA_ERR_INVALID_ARG, "k_block_scales and v_block_scales must be non-NULL");
    if (!aligned(k_block_scales, 16) || !aligned(v_block_scales, 16))
        return fail(TA_ERR_INVALID_ARG, "k_block_scales and v_block_scales must be 16-byte aligned");
    if ((k_factor && !aligned(k_factor, 4)) || (v_factor && !aligned(v_factor, 4)))
        return fail(TA_ERR_INVALID_ARG, "k_factor and v_factor must be 4-byte aligned");
    const int G = p->Hq / p->Hkv;
    if (p->D != 128 || (G != 2 && G != 4))
        return fail(TA_ERR_UNSUPPORTED, "NVFP4 decode supports D = 128 with 2 or 4 query heads per KV head");
    if (p->S % 16 != 0)
        return fail(TA_ERR_UNSUPPORTED, "NVFP4 decode needs S (the cache's keys per sequence) a multiple of 16");
    ta_decode_plan plan;
    s = ta_decode_plan_for(p->B, p->Hq, p->Hkv, p->S, p->D, p->chunk, p->n_split, p->seqlens != nullptr, 0, &plan);
    if (s != TA_OK)
        return s;
    if (plan.n_split > 1 && plan.chunk % ta::kDecodeTileKeysTC != 0)
        return fail(TA_ERR_UNSUPPORTED, "NVFP4 decode needs chunks of whole 128-key tiles (chunk override a "
                                        "multiple of 128, or an n_split that gives such chunks)");
    return decode_impl(p, nullptr, 0, 0, 0, 0, 0, false, k_factor, v_factor, true, k_block_scales, v_block_scales);
}

ta_status ta_decode_pi(const ta_decode_params *p, int window, int period)
{
    ta_status s = validate_decode(p);
    if (s != TA_OK)
        return s;
    if (window < 0 || period < 1)
        return fail(TA_ERR_INVALID_ARG, "pi-Attention needs window >= 0 and period >= 1");
    return decode_impl(p, nullptr, 0, 0, 0, window, period);
}

size_t ta_decode_pi_workspace_bytes(int B, int Hq, int Hkv, int S, int D, int chunk, int n_split, int varlen,
                                    int window, int period)
{
    if (S < 1 || window < 0 || period < 1)
        return 0;
    return ta_decode_workspace_bytes(B, Hq, Hkv, (int)ta::pi_max_keys(S, window, period), D, chunk, n_split, varlen);
}

ta_status ta_decode_paged(const ta_paged_decode_params *pp)
{
    if (!pp)
        return fail(TA_ERR_INVALID_ARG, "params pointer is NULL");
    if (!pp->block_table || !pp->seqlens)
        return fail(TA_ERR_INVALID_ARG, "block_table and seqlens must be non-NULL");
    if (pp->page_size < 1 || pp->pages_per_seq < 1 || pp->num_pages < 1)
        return fail(TA_ERR_INVALID_ARG, "page_size, pages_per_seq and num_pages must all be >= 1");
    if ((int64_t)pp->page_size * pp->pages_per_seq > INT32_MAX)
        return fail(TA_ERR_INVALID_ARG, "page_size * pages_per_seq overflows");
    if (!aligned(pp->block_table, 4))
        return fail(TA_ERR_INVALID_ARG, "block_table must be 4-byte aligned");
    if ((double)pp->num_pages * pp->Hkv * pp->page_size * pp->D > 9.0e18 / 4)
        return fail(TA_ERR_INVALID_ARG, "page pool size overflows");
    ta_decode_params p;
    std::memset(&p, 0, sizeof p);
    p.q = pp->q;
    p.k = pp->k_pages;
    p.v = pp->v_pages;
    p.out = pp->out;
    p.lse = pp->lse;
    p.B = pp->B;
    p.Hq = pp->Hq;
    p.Hkv = pp->Hkv;
    p.S = pp->page_size * pp->pages_per_seq;
    p.D = pp->D;
    p.scale = pp->scale;
    p.seqlens = pp->seqlens;
    p.in_dtype = pp->in_dtype;
    p.out_dtype = pp->out_dtype;
    p.chunk = pp->chunk;
    p.n_split = pp->n_split;
    p.workspace = pp->workspace;
    p.workspace_bytes = pp->workspace_bytes;
    p.stream = pp->stream;
    p.wait_limit_ns = pp->wait_limit_ns;
    ta_status s = validate_decode(&p);
    if (s != TA_OK)
        return s;
    return decode_impl(&p, pp->block_table, pp->page_size, pp->pages_per_seq, pp->num_pages);
}

ta_status ta_decode_partials(const ta_decode_params *p, float *m, float *l, float *o)
{
    if (!p)
        return fail(TA_ERR_INVALID_ARG, "params pointer is NULL");
    ta_decode_params v = *p;
    v.out = o;  // validated as a 16-byte aligned output; the kernel writes partials only
    v.lse = nullptr;
    v.out_dtype = TA_F32;
    ta_status s = validate_decode(&v);
    if (s != TA_OK)
        return s;
    if (!m || !l || !o)
        return fail(TA_ERR_INVALID_ARG, "m, l and o must be non-NULL");
    if (!aligned(m, 4) || !aligned(l, 4))
        return fail(TA_ERR_INVALID_ARG, "m and l must be 4-byte aligned");
    ta_decode_plan plan;
    s = ta_decode_plan_for(p->B, p->Hq, p->Hkv, p->S, p->D, p->chunk, p->n_split, p->seqlens != nullptr, 0, &plan);
    if (s != TA_OK)
        return s;
    void *ws = p->workspace;
    if (ws) {
        if (!aligned(ws, 256) || p->workspace_bytes < (size_t)ta::kStatusBytes)
            return fail(TA_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= 256 bytes");
    } else {
        s = library_workspace(ta::kStatusBytes, &ws);
        if (s != TA_OK)
            return s;
    }
    ta::DecodeLaunch a;
    a.q = p->q;
    a.k = p->k;
    a.v = p->v;
    a.out = nullptr;
    a.lse = nullptr;
    a.B = p->B;
    a.Hq = p->Hq;
    a.Hkv = p->Hkv;
    a.S = p->S;
    a.D = p->D;
    a.scale = p->scale;
    a.seqlens = p->seqlens;
    a.in_dtype = p->in_dtype;
    a.out_dtype = TA_F32;
    a.plan = plan;
    a.plan.n_split = plan.n_split;
    a.force_partials = true;
    a.block_table = nullptr;
    a.page_size = a.pages_per_seq = a.num_pages = 0;
    a.pi_window = a.pi_period = 0;
    a.kv_fp8 = false;
    a.k_scale = a.v_scale = nullptr;
    a.kv_nvfp4 = false;
    a.k_bs = a.v_bs = nullptr;
    a.wait_ns = ta::wait_limit_or_default(p->wait_limit_ns);
    a.test_stall = ta::injected_stall();
    a.stream = static_cast<cudaStream_t>(p->stream);
    a.status = static_cast<int32_t *>(ws);
    a.counters = nullptr;
    a.part_m = m;
    a.part_l = l;
    a.part_o = o;
    cudaError_t e = ta::launch_decode(a);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode kernel launch");
    return TA_OK;
}

ta_status ta_decode(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq, int Hkv,
                    int S, int D, float scale, const int32_t *seqlens, void *stream)
{
    ta_decode_params p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.lse = lse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S = S;
    p.D = D;
    p.scale = scale;
    p.seqlens = seqlens;
    p.in_dtype = TA_BF16;
    p.out_dtype = TA_BF16;
    p.stream = stream;
    return ta_decode_ex(&p);
}

ta_status ta_decode_status(void *workspace, void *stream, int32_t *flags)
{
    if (!flags)
        return fail(TA_ERR_INVALID_ARG, "flags pointer is NULL");
    void *ws = workspace;
    size_t clear = ta::kStatusBytes;
    if (!ws) {
        ta_status s = library_workspace(256, &ws);
        if (s != TA_OK)
            return s;
        int dev = 0;
        cudaGetDevice(&dev);
        std::lock_guard<std::mutex> lock(g_mu);
        clear = std::min(state_for(dev).ws_bytes, (size_t)ta::kCtrlBytes);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    int32_t word = 0;
    e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(status)");
    // A launch that gave up can leave chunk counters behind: clear the
    // whole control region of the library's workspace then.
    e = cudaMemset(ws, 0, (word & TA_DEVERR_TIMEOUT) ? clear : ta::kStatusBytes);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemset(status)");
    *flags = word;
    return TA_OK;
}

size_t ta_combine_workspace_bytes(int R, int N, int D)
{
    if (R < 1 || N < 1 || D < 1)
        return 0;
    return ta::combine_scratch_bytes(R, N, D);
}

ta_status ta_combine(const float *m, const float *l, const float *o, int R, int N, int D, void *out,
                     ta_dtype out_dtype, float *lse, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!m || !l || !o || !out)
        return fail(TA_ERR_INVALID_ARG, "m, l, o and out must be non-NULL");
    if (R < 1 || N < 1 || D < 1)
        return fail(TA_ERR_INVALID_ARG, "R, N and D must all be >= 1");
    if (out_dtype != TA_F32 && out_dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARG, "out_dtype must be TA_F32 or TA_BF16");
    if (!aligned(o, 16) || !aligned(m, 4) || !aligned(l, 4) || !aligned(out, 16) || (lse && !aligned(lse, 4)))
        return fail(TA_ERR_INVALID_ARG, "o and out must be 16-byte aligned, m, l and lse 4-byte aligned");
    if (D != 64 && D != 128)
        return fail(TA_ERR_UNSUPPORTED, "combine supports D = 64 or 128");
    if ((double)R * N * D > 2.0e18)
        return fail(TA_ERR_INVALID_ARG, "partials size overflows");
    const size_t need = ta::combine_scratch_bytes(R, N, D);
    void *ws = workspace;
    if (need > 0) {
        if (ws) {
            if (!aligned(ws, 256))
                return fail(TA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
            if (workspace_bytes < need)
                return fail(TA_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes");
        } else {
            // the library workspace keeps its control region for decodes
            ta_status s = library_workspace(need + ta::kCtrlBytes, &ws);
            if (s != TA_OK)
                return s;
            ws = static_cast<char *>(ws) + ta::kCtrlBytes;
        }
    }
    cudaError_t e = ta::launch_combine(m, l, o, R, N, D, out, out_dtype, lse, ws, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "combine kernel launch");
    return TA_OK;
}

ta_status ta_prefill_causal_ex(const ta_prefill_params *p)
{
    if (!p)
        return fail(TA_ERR_INVALID_ARG, "params pointer is NULL");
    const bool packed = p->cu_seqlens != nullptr;
    if (!p->q || !p->k || !p->v || !p->out)
        return fail(TA_ERR_INVALID_ARG, "q, k, v and out must be non-NULL");
    if (p->B < 1 || p->H < 1 || p->Hkv < 1 || p->S < 1 || p->D < 1 || (packed && p->total_tokens < 1))
        return fail(TA_ERR_INVALID_ARG, packed ? "num_seqs, max_seqlen, total_tokens, H, Hkv and D must all be >= 1"
                                               : "B, H, Hkv, S and D must all be >= 1");
    if (p->H % p->Hkv != 0)
        return fail(TA_ERR_INVALID_ARG, "H must be a multiple of Hkv");
    if (!std::isfinite(p->scale))
        return fail(TA_ERR_INVALID_ARG, "scale must be finite");
    if (p->out_dtype != TA_F32 && p->out_dtype != TA_BF16)
        return fail(TA_ERR_INVALID_ARG, "out_dtype must be TA_F32 or TA_BF16");
    if (!aligned(p->q, 16) || !aligned(p->k, 16) || !aligned(p->v, 16) || !aligned(p->out, 16) ||
        (p->lse && !aligned(p->lse, 4)) || (packed && !aligned(p->cu_seqlens, 4)))
        return fail(TA_ERR_INVALID_ARG,
                    "q, k, v and out must be 16-byte aligned, lse and cu_seqlens 4-byte aligned");
    if (p->D != 128)
        return fail(TA_ERR_UNSUPPORTED, "prefill supports head dim D = 128");
    if (!(p->scale > 0.f))
        return fail(TA_ERR_UNSUPPORTED, "prefill supports scale > 0");
    if (!packed && (double)p->B * p->H * p->S * p->D > 9.0e18 / 4)
        return fail(TA_ERR_INVALID_ARG, "tensor size overflows");
    if (packed && ((double)p->total_tokens * p->H * p->D > 9.0e18 / 4 ||
                   (double)p->B * p->H * ((p->S + 255) / 256) > 2.0e9))
        return fail(TA_ERR_INVALID_ARG, "problem size overflows");
    if (!packed && (double)p->B * p->H * ((p->S + 255) / 256) > 2.0e9)
        return fail(TA_ERR_INVALID_ARG, "problem size overflows");
    void *ws = nullptr;
    ta_status s = library_workspace(256, &ws);
    if (s != TA_OK)
        return s;
    ta::PrefillLaunch a;
    a.q = p->q;
    a.k = p->k;
    a.v = p->v;
    a.out = p->out;
    a.lse = p->lse;
    a.B = p->B;
    a.H = p->H;
    a.Hkv = p->Hkv;
    a.S = p->S;
    a.D = p->D;
    a.scale = p->scale;
    a.cu_seqlens = p->cu_seqlens;
    a.T = packed ? p->total_tokens : 0;
    a.out_dtype = p->out_dtype;
    a.status = static_cast<int32_t *>(ws);
    a.wait_ns = ta::wait_limit_or_default(p->wait_limit_ns);
    a.test_stall = ta::injected_stall();
    a.stream = static_cast<cudaStream_t>(p->stream);
    cudaError_t e = ta::launch_prefill(a);
    if (e == cudaErrorNotSupported)
        return fail(TA_ERR_UNSUPPORTED, "causal prefill kernel is not available in this build");
    if (e != cudaSuccess)
        return cuda_fail(e, "prefill kernel launch");
    return TA_OK;
}

ta_status ta_prefill_causal(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                            int Hkv, int S, int D, float scale, void *stream)
{
    ta_prefill_params p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.S = S;
    p.D = D;
    p.scale = scale;
    p.out_dtype = TA_BF16;
    p.stream = stream;
    return ta_prefill_causal_ex(&p);
}

ta_status ta_prefill_causal_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                                   const int32_t *cu_seqlens, int num_seqs, int max_seqlen, int total_tokens, int H,
                                   int Hkv, int D, float scale, void *stream)
{
    if (!cu_seqlens)
        return fail(TA_ERR_INVALID_ARG, "q, k, v, out and cu_seqlens must be non-NULL");
    ta_prefill_params p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.lse = lse;
    p.B = num_seqs;
    p.H = H;
    p.Hkv = Hkv;
    p.S = max_seqlen;
    p.D = D;
    p.scale = scale;
    p.cu_seqlens = cu_seqlens;
    p.total_tokens = total_tokens;
    p.out_dtype = TA_BF16;
    p.stream = stream;
    return ta_prefill_causal_ex(&p);
}

}  // extern "C"
