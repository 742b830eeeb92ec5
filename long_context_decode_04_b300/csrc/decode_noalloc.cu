// decode_noalloc.cu -- split-KV decode whose scratch lives in a fixed,
// statically sized device array instead of memory the call allocates.
//
// Who needs this.  Some callers cannot let a library call cudaMalloc:
//   * programs whose device memory is owned by a pool allocator (a
//     framework's caching allocator, an inference server's arena) that has
//     already reserved almost all of the GPU, so a cudaMalloc from inside the
//     library fails, or succeeds only by fighting the pool for memory;
//   * latency-critical loops that cannot afford the device-wide
//     synchronisation that cudaMalloc / cudaFree can cause, stalling every
//     other stream on the GPU;
//   * deployments whose rules forbid dynamic device allocation after
//     start-up (fixed memory budgets decided at load time).
// ta_decode already avoids allocation when the caller hands it a workspace,
// but that still asks the caller to allocate one.  ta_decode_noalloc needs
// nothing from the caller except inputs and outputs: its scratch is the
// array below, which the CUDA runtime reserves when it loads this library's
// device code on a GPU and which stays reserved there until the process
// exits.
//
// Set-up: the array belongs to this file's device code, which the CUDA
// runtime loads on a device when it is first needed there (lazy module
// loading); the first cudaGetSymbolAddress on a device is that moment, and
// it is also when the array's 8 MiB are reserved.  So the first call on a
// device (or ta_decode_noalloc_setup) should come early: before a pool
// allocator takes the GPU's memory, and before any stream capture.  The
// address is cached per device for the life of the process; a
// cudaDeviceReset invalidates it, and nothing here notices.
//
// Device-side flags (a length outside [0, S], a timed-out wait) land in the
// scratch's status word; ta_decode_noalloc_status reads and clears it
// without allocating.
//
// What the scratch holds: the decode workspace (status word and work-queue
// counter in its first 256 bytes, the per-(sequence, KV head) chunk
// counters, then the per-chunk partials (m, l, o) and the merge's
// intermediates).  The status word and the counters are cleared on the
// call's stream at the start of every call; the rest is fully written before
// it is read.  All calls on a GPU share the one array, so calls that overlap on the
// GPU (different streams, or different host threads, with no ordering
// between them) race on it and give wrong results.
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(8) << 20;  // 8 MiB per GPU

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

ta_status fail(ta_status s, const std::string &msg)
{
    ta::record_error(msg);
    return s;
}

// The device address of the scratch array on the current device.  In host
// code `g_noalloc_scratch` names a host-side stand-in, not device memory, so
// the address must come from cudaGetSymbolAddress, asked once per device
// with that device current.
ta_status scratch_for_current_device(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(TA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TA_ERR_UNSUPPORTED, "device ordinal out of range for the allocation-free decode");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(TA_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return TA_OK;
}

}  // namespace

extern "C" {

ta_status ta_decode_noalloc_setup(void)
{
    void *scratch = nullptr;
    return scratch_for_current_device(&scratch);
}

ta_status ta_decode_noalloc_status(void *stream, int32_t *flags)
{
    if (!flags)
        return fail(TA_ERR_INVALID_ARG, "flags pointer is NULL");
    void *scratch = nullptr;
    ta_status s = scratch_for_current_device(&scratch);
    if (s != TA_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return fail(TA_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
    int32_t word = 0;
    e = cudaMemcpy(&word, scratch, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return fail(TA_ERR_CUDA, std::string("cudaMemcpy(status word): ") + cudaGetErrorString(e));
    // after a timeout the work-queue and chunk counters may be left behind
    e = cudaMemsetAsync(scratch, 0, (word & TA_DEVERR_TIMEOUT) ? ta::kCtrlBytes : ta::kStatusBytes, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return fail(TA_ERR_CUDA, std::string("cudaMemsetAsync(status word): ") + cudaGetErrorString(e));
    *flags = word;
    return TA_OK;
}

ta_status ta_decode_noalloc(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                            int Hkv, int S, int D, float scale, const int32_t *seqlens, void *stream)
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
    // Reject bad arguments before anything is enqueued.
    ta_status s = ta::check_decode_params(&p);
    if (s != TA_OK)
        return s;
    ta_decode_plan plan;
    s = ta_decode_plan_for(B, Hq, Hkv, S, D, 0, 0, seqlens != nullptr, 0, &plan);
    if (s != TA_OK)
        return s;
    if (plan.workspace_bytes > kNoallocScratchBytes)
        return fail(TA_ERR_WORKSPACE, "ta_decode_noalloc: this shape needs " + std::to_string(plan.workspace_bytes) +
                                          " bytes of scratch, more than its fixed " +
                                          std::to_string(kNoallocScratchBytes) +
                                          " bytes; use ta_decode or ta_decode_ex with a workspace");
    void *scratch = nullptr;
    s = scratch_for_current_device(&scratch);
    if (s != TA_OK)
        return s;
    // The status word, the work-queue counter and the per-unit chunk
    // counters must start at zero.
    const size_t zero_bytes = plan.n_split > 1 ? ta::kCtrlBytes : ta::kStatusBytes;
    cudaError_t e = cudaMemsetAsync(scratch, 0, zero_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(TA_ERR_CUDA, std::string("cudaMemsetAsync(status word): ") + cudaGetErrorString(e));
    p.workspace = scratch;
    p.workspace_bytes = kNoallocScratchBytes;
    return ta_decode_ex(&p);
}

}  // extern "C"
