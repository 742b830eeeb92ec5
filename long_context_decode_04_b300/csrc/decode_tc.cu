// decode_tc.cu -- split-KV exact decode for grouped-query attention with
// both contractions on the tensor cores (tcgen05, accumulators in TMEM).
//
// What is computed is the same as the CUDA-core decode (decode.cu): for
// each query head, scores s_j = scale * <q, k_j>, softmax weights and the
// weighted mean of the values (Attention glossary, jisaku.com/glossary/
// attention, "basic concepts and operating principle"), one partial
// (m, l, o) per KV chunk and the log-sum-exp merge of a sequence's
// partials (Tree Attention explainer, aibr.jp/archives/143699, sections 1
// and 3).  Chunks are whole 128-key tiles (the MMA's M); the partials'
// layout is the one every decode kernel writes.
//
// Why tensor cores in a bandwidth-bound step.  The G query heads of a KV
// head (grouped-query attention) share its keys, so per KV head the scores
// are the product [keys x D] . [D x G] and the output [D x keys] . [keys x G]:
// contractions of the streamed tile with a G-row matrix (G = 1, a
// matrix-vector product, stays on the CUDA cores).  On the CUDA cores they
// cost about 57 issued warp instructions per key row at G = 4, which keeps
// that kernel issue-bound under the HBM roofline.  Here each contraction is
// a handful of tcgen05.mma per tile and the remaining per-key work is a few
// instructions of softmax, so the issue slots no longer bound the kernel:
// how long a ring stage is held between its copy and its value product does.
//
// Per 128-key tile (M = 128 rows, one key row per TMEM lane):
//   S^T [128 keys x 16] = K [128 x D] . Q^T [D x 16]     (A = K, K-major;
//                                                        B = Q, heads padded to 16)
//   O_t^T [D x 32]      = V^T [D x 128] . P^T [128 x 32] (A = V, MN-major;
//                                                        B = P, K-major)
// P has one row per (softmax warp, head) in bf16 hi and lo parts (p = hi +
// lo to about 2^-17 relative), so one MMA per 16 keys sums both and the
// weights keep fp32-like precision against bf16 V; p = exp2(s - m) against
// its warp's reference m, raised lazily (only when a score passes it by
// more than 2^8).
//
// Kernel layout (one persistent CTA per SM, 8 warps):
//   * warp 0: producer.  Takes work items (sequence, KV head, chunk) from
//     the device-wide queue, loads the item's G query rows (TMA, 128-byte
//     swizzle) into one of two Q buffers and the chunk's K/V tiles into a
//     3-stage ring (TMA boxes of 128 rows x 64 dims; boxes of 8 rows at a
//     pi-Attention sequence's boundary between periodic and window keys).
//   * warp 1: allocates 128 TMEM columns (S double buffer, O double
//     buffer) and issues the score products; warp 2 issues the value
//     products.  Each blocks on the one barrier it needs next, so a tile's
//     value product never waits for the next tile's copy.
//   * warp 3 (fused mode): the ticket thread, which takes the merge tickets
//     the softmax warps ask for at their item ends.
//   * warps 4-7 (one warpgroup, TMEM lane quadrants 0-3): thread r owns key
//     row r of every tile for the softmax and output dimension r for the
//     accumulation.  Each warp runs its own online softmax over its 32 key
//     rows (running maximum, weights to the P rows of (warp, head)); per
//     tile a thread then adds the four warps' columns of the previous
//     tile's O_t to its registers, each rescaled by its warp's factor.  At
//     the end of an item the four warps' states are merged and the partial
//     (or the final output and lse) is written; in fused mode the ticket
//     and the merge follow.
//   * Every wait is bounded (kWaitLimitNs); on expiry the kernel records
//     TA_DEVERR_TIMEOUT, stops, lets its copies and MMAs land and frees its
//     TMEM.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "decode_tc_common.cuh"
#include "tcgen05.cuh"

namespace ta {
namespace {

constexpr int kD = 128;
constexpr int kTile = kDecodeTileKeysTC;  // 128 keys a tile
constexpr int kRows = 128;                // MMA rows: one key a row
constexpr int kN = 16;                  // MMA N: the group's heads, zero-padded
constexpr int kStages = 3;
constexpr int kHalf = kRows * 128;          // one 64-dim half of a staged K or V tile
constexpr int kTileBytes = 2 * kHalf;       // 32 KiB
constexpr int kStageBytes = 2 * kTileBytes; // K then V
constexpr int kQHalf = kN * 128;            // 16 rows x 128 bytes
constexpr int kQBytes = 2 * kQHalf;
constexpr int kON = 2 * kN;                 // value-product N: (warp, head) columns, hi then lo
constexpr int kPHalf = kON * 128;           // P rows x 64 keys of 128 bytes
constexpr int kPBytes = 2 * kPHalf;         // one P operand: 32 rows x 128 keys, bf16
constexpr int kQOff = kStages * kStageBytes;
constexpr int kPOff = kQOff + 2 * kQBytes;
constexpr int kMiscOff = kPOff + 2 * kPBytes;
constexpr uint32_t kTxBytes = 4u * kTile * 128u;  // K and V, two halves each
constexpr int kSoftWarp0 = 4;
constexpr int kSoftThreads = 128;
constexpr int kThreads = 256;
constexpr uint32_t kOCol = 2 * kN;   // S at TMEM columns 0 and 16, O at 32 and 64
constexpr uint32_t kTmemCols = 128;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kRescaleLog2 = 8.0f;
// partial outputs in flight per round of the fused merge (the register
// budget of 256 threads allows sixteen float4, that of 384 threads eight)
constexpr int kMergeBatch = 16;

enum : int { kFirst = 1, kLast = 2, kEnd = 4 };
constexpr int kModeFinal = tcd::kModeFinal, kModePartials = tcd::kModePartials, kModeFused = tcd::kModeFused;

struct TileDesc {
    int item;
    int j0;
    int n;
    int flags;
};

struct Misc {
    uint64_t full[kStages];      // K/V tile landed (TMA bytes) and its descriptor written
    uint64_t kv_empty[kStages];  // both products of the tile done (MMA commit)
    uint64_t s_full[2];          // S of a tile in TMEM (MMA commit)
    uint64_t p_full[2][4];       // a warp's P of a tile in shared memory (32 threads)
    uint64_t p_all[2];           // all four warps' P and factors (128 threads): a fast
                                 // warp cannot complete it alone, unlike its own p_full
    uint64_t o_full[2];          // O_t in TMEM (MMA commit)
    uint64_t o_empty[2];         // O_t added to the registers (128 threads)
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t grp_bar;            // softmax warpgroup rendezvous (end of item)
    uint64_t mma_done;
    TileDesc desc[kStages];
    float alpha[4][4][4];        // [tile % 4][warp][head] factor by which a warp's maximum rose
    tcd::ItemSmem isum;          // the item end's sums, maxima and ticket
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmem = (size_t)kMiscOff + sizeof(Misc) + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory per CTA");
static_assert(kTile <= kRows && kTile % 8 == 0, "tile rows");

struct TcParams {
    // q rows (box 64 x G); K/V tiles of 128 rows and groups of 8 rows;
    // pi-Attention periodic keys as rows (tiles of 128 and groups of 8)
    CUtensorMap qmap, kmap, vmap, k8map, v8map, kpimap, vpimap, kpi8map, vpi8map;
    const void *k, *v;
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
    // pi-Attention key set (pi_period > 0): the query at i = L - 1 attends
    // the window [max(0, i - pi_window), i] and the keys i - m * pi_period
    // (m >= 1) before it; the chunks cut the ascending list of those keys.
    int pi_window, pi_period;
    // Paged cache (block_table != nullptr): k, v are page pools [num_pages,
    // Hkv, page_size, D] seen as (D, page_size, num_pages * Hkv) with boxes
    // of pg_rows = min(page_size, 128) rows; page_size divides 128 or is a
    // multiple of it, so a 128-key tile is whole pages or part of one.
    const int32_t *block_table;
    int page_size, pages_per_seq, num_pages, pg_rows;
    CUtensorMap kpgmap, vpgmap;
};


template <int G, typename OUT>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Misc *ms = reinterpret_cast<Misc *>(smem + kMiscOff);
    volatile int *abort_flag = &ms->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Zero what no copy writes: the Q buffers (rows G..15 stay zero) and the
    // P buffers.  (Staged rows past a tile's keys are masked and their V
    // rows zeroed per tile by the softmax threads.)
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < (kMiscOff - kQOff) / 16; i += kThreads)
        *reinterpret_cast<uint4 *>(smem + kQOff + i * 16) = z4;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ms->full[s], 2);  // the producer arrives before and after its copies
            mbar_init(&ms->kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms->s_full[i], 1);
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
        // Lane 0 takes the decisions (work queue, ring waits, expected
        // bytes, descriptors); the 32 lanes share the copies of a tile.  A
        // tile is one TMA box of 128 rows when its keys are contiguous in
        // memory, else 16 groups of 8 rows: a box of 8 rows for a group whose
        // keys are contiguous (all periodic or all window keys), plain loads
        // and swizzled stores for the one group that straddles the two.  The full barrier
        // takes two arrivals from lane 0, with the expected TMA bytes before
        // the copies and once the plain stores are done.
        const bool leader = lane == 0;
        if (leader) {
            tc::prefetch_tensormap(&p.qmap);
            tc::prefetch_tensormap(p.block_table ? &p.kpgmap : &p.kmap);
            tc::prefetch_tensormap(p.block_table ? &p.vpgmap : &p.vmap);
        }
        const uint64_t policy = l2_policy_evict_first();
        const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(p.k);
        const __nv_bfloat16 *vg = static_cast<const __nv_bfloat16 *>(p.v);
        int stage = 0;
        uint32_t uses[kStages] = {0u, 0u, 0u};  // times each stage was armed
        uint32_t q_uses[2] = {0u, 0u};
        int ic = 0;  // items taken
        bool ok = true;
        if (p.test_stall) {
            // test hook: a wait that nothing ends (phase 0 of a barrier only
            // this warp arms), so the launch's time limit runs out
            int w = 1;
            if (leader)
                w = mbar_wait_bounded(&ms->full[0], 0, abort_flag, p.wait_ns);
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
                        w = mbar_wait_bounded(&ms->kv_empty[stage], (uses[stage] - 1) & 1, abort_flag, p.wait_ns);
                    if (w) {
                        ms->desc[stage] = TileDesc{item, 0, 0, kEnd};
                        mbar_arrive(&ms->full[stage]);
                        mbar_arrive(&ms->full[stage]);
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
            // the keys this sequence attends, as an ascending list of N
            // positions: n_skip periodic keys r0, r0 + pi, ... then the window
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
            // element offset of the K/V row of list position pos
            auto row_of = [&](int pos) -> size_t {
                const int key = pos < n_skip ? r0 + pos * p.pi_period : w0 + (pos - n_skip);
                return ((size_t)unit * p.S + key) * kD;
            };
            // the item's G query rows
            const int qb = ic & 1;
            int w = 1;
            if (leader) {
                if (q_uses[qb] > 0)
                    w = mbar_wait_bounded(&ms->q_empty[qb], (q_uses[qb] - 1) & 1, abort_flag, p.wait_ns);
                if (w) {
                    unsigned char *qd = smem + kQOff + qb * kQBytes;
                    mbar_arrive_expect_tx(&ms->q_full[qb], 2u * G * 128u);
                    tc::tma_load_3d(qd, &p.qmap, 0, 0, unit, &ms->q_full[qb]);
                    tc::tma_load_3d(qd + kQHalf, &p.qmap, 64, 0, unit, &ms->q_full[qb]);
                }
            }
            if (!__shfl_sync(kFull, w, 0))
                break;
            ++q_uses[qb];
            ++ic;
            int j0 = c0, flags = kFirst;
            for (;;) {
                const int n = max(0, min(kTile, c1 - j0));
                const bool last = j0 + n >= c1;
                if (last)
                    flags |= kLast;
                // whole-tile boxes: contiguous keys (y = ya of kmap), or 128
                // periodic keys (y = j0 of kpimap)
                const bool paged = p.block_table != nullptr;
                const bool whole = !paged && n > 0 && (p.pi_period == 0 || j0 >= n_skip);
                const bool whole_pi = !paged && n > 0 && p.pi_period > 0 && j0 + kTile <= n_skip;
                const int ya = p.pi_period > 0 ? w0 + (j0 - n_skip) : j0;
                const int ng = (whole || whole_pi || paged) ? 0 : (n + 7) >> 3;  // groups of 8 rows
                // paged cache: piece t (lane t) is rows [t * pg_rows, (t + 1) *
                // pg_rows) of the tile, all in one page (pg_rows = min(page
                // size, 128), and tiles start on page boundaries or inside
                // one page), one box of pg_rows rows from the page pool
                bool pg = false;
                int pg_y = 0, pg_z = 0;
                if (paged && lane * p.pg_rows < n) {
                    const int key = j0 + lane * p.pg_rows;
                    const int pid = p.block_table[(size_t)b * p.pages_per_seq + key / p.page_size];
                    if (pid >= 0 && pid < p.num_pages) {
                        pg = true;
                        pg_y = key % p.page_size;
                        pg_z = pid * p.Hkv + (unit - b * p.Hkv);
                    } else {
                        atomicOr(&p.status[0], TA_DEVERR_PAGE);  // not followed; output undefined
                    }
                }
                const unsigned pg_mask = __ballot_sync(kFull, pg);
                bool g8 = false;
                const CUtensorMap *gk = &p.k8map, *gv = &p.v8map;
                int gx = 0, gy = 0;
                if (lane < ng) {
                    const int pos = j0 + 8 * lane;
                    if (pos + 8 <= n_skip) {
                        g8 = true;
                        gk = &p.kpi8map;
                        gv = &p.vpi8map;
                        gx = r0 * kD;
                        gy = pos;
                    } else if (pos >= n_skip) {
                        g8 = true;
                        gy = w0 + (pos - n_skip);
                    }
                }
                const unsigned g8_mask = __ballot_sync(kFull, g8);
                const unsigned man_mask = __ballot_sync(kFull, lane < ng && !g8);
                const uint32_t bytes = (whole || whole_pi) ? kTxBytes
                                       : paged ? (uint32_t)__popc(pg_mask) * 4u * (uint32_t)p.pg_rows * 128u
                                               : (uint32_t)__popc(g8_mask) * 4096u;
                w = 1;
                if (leader) {
                    if (uses[stage] > 0)
                        w = mbar_wait_bounded(&ms->kv_empty[stage], (uses[stage] - 1) & 1, abort_flag, p.wait_ns);
                    if (w) {
                        ms->desc[stage] = TileDesc{item, j0, n, flags};
                        if (bytes)
                            mbar_arrive_expect_tx(&ms->full[stage], bytes);
                        else
                            mbar_arrive(&ms->full[stage]);
                    }
                }
                if (!__shfl_sync(kFull, w, 0)) {
                    ok = false;
                    break;
                }
                unsigned char *kd = smem + stage * kStageBytes;
                unsigned char *vd = kd + kTileBytes;
                uint64_t *fb = &ms->full[stage];
                if (leader && (whole || whole_pi)) {
                    // rows past S read as zero; rows in [n, 128) are zeroed by
                    // the softmax threads before the value product
                    const CUtensorMap *mk = whole ? &p.kmap : &p.kpimap;
                    const CUtensorMap *mv = whole ? &p.vmap : &p.vpimap;
                    const int x0 = whole ? 0 : r0 * kD, y = whole ? ya : j0;
                    tc::tma_load_3d_hint(kd, mk, x0, y, unit, fb, policy);
                    tc::tma_load_3d_hint(kd + kHalf, mk, x0 + 64, y, unit, fb, policy);
                    tc::tma_load_3d_hint(vd, mv, x0, y, unit, fb, policy);
                    tc::tma_load_3d_hint(vd + kHalf, mv, x0 + 64, y, unit, fb, policy);
                }
                if (pg) {
                    const int r = lane * p.pg_rows * 128;
                    tc::tma_load_3d_hint(kd + r, &p.kpgmap, 0, pg_y, pg_z, fb, policy);
                    tc::tma_load_3d_hint(kd + kHalf + r, &p.kpgmap, 64, pg_y, pg_z, fb, policy);
                    tc::tma_load_3d_hint(vd + r, &p.vpgmap, 0, pg_y, pg_z, fb, policy);
                    tc::tma_load_3d_hint(vd + kHalf + r, &p.vpgmap, 64, pg_y, pg_z, fb, policy);
                }
                if (g8) {
                    const int r = 8 * lane * 128;
                    tc::tma_load_3d_hint(kd + r, gk, gx, gy, unit, fb, policy);
                    tc::tma_load_3d_hint(kd + kHalf + r, gk, gx + 64, gy, unit, fb, policy);
                    tc::tma_load_3d_hint(vd + r, gv, gx, gy, unit, fb, policy);
                    tc::tma_load_3d_hint(vd + kHalf + r, gv, gx + 64, gy, unit, fb, policy);
                }
                // the other groups: lane = 4 * row + part, part = K or V x half
                for (unsigned mm = man_mask; mm; mm &= mm - 1) {
                    const int r = 8 * (__ffs(mm) - 1) + (lane >> 2);
                    const int part = lane & 3;
                    if (r < n) {
                        const __nv_bfloat16 *src = (part < 2 ? kg : vg) + row_of(j0 + r) + (part & 1) * 64;
                        uint4 x[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            x[c] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
                        unsigned char *dst = (part < 2 ? kd : vd) + (part & 1) * kHalf + r * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(dst + ((c ^ (r & 7)) << 4)) = x[c];
                    }
                }
                if (man_mask)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (leader)
                    mbar_arrive(fb);
                ++uses[stage];
                if (++stage == kStages)
                    stage = 0;
                if (last)
                    break;
                j0 += n;
                flags = 0;
            }
        }
        // Every copy issued lands before the CTA exits (immediate on the
        // normal path; bounded after an abort).
        __syncwarp();
        if (leader) {
            int drain_abort = 0;
            for (int s = 0; s < kStages; ++s)
                if (uses[s] > 0)
                    mbar_wait_bounded(&ms->full[s], (uses[s] - 1) & 1, &drain_abort);
            for (int i = 0; i < 2; ++i)
                if (q_uses[i] > 0)
                    mbar_wait_bounded(&ms->q_full[i], (q_uses[i] - 1) & 1, &drain_abort);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues the score products, warp 2 the value products, each
        // blocking on the one barrier it needs next, so that neither product
        // waits on the other's inputs.  Each thread's commits track its own
        // MMAs: the value product of a tile comes after its softmax, hence
        // after its score product, so its commit releases the stage.
        if (lane == 0) {
            const uint32_t sbase = smem_u32(smem);
            int t = 0, stage = 0;
            uint32_t sph = 0;
            if (warp == 1) {
                constexpr uint32_t kIdS = tc::idesc_bf16_f32_major(kRows, kN, false, false);
                int ic = 0;
                for (;;) {
                    if (!mbar_wait_bounded(&ms->full[stage], sph, abort_flag, p.wait_ns))
                        break;
                    const TileDesc d = ms->desc[stage];
                    // S and P buffers of this parity are free once the value
                    // product of tile t - 2 is done (its softmax read S, it read P)
                    if (t >= 2 && !mbar_wait_bounded(&ms->o_full[t & 1], ((t - 2) >> 1) & 1, abort_flag, p.wait_ns))
                        break;
                    if (d.flags & kEnd) {
                        mbar_arrive(&ms->s_full[t & 1]);  // tells the softmax warps to stop
                        break;
                    }
                    const int qb = ic & 1;
                    if ((d.flags & kFirst) && !mbar_wait_bounded(&ms->q_full[qb], (ic >> 1) & 1, abort_flag, p.wait_ns))
                        break;
                    tc::fence_after_sync();
                    // S_t^T = K Q^T over D in 8 steps of 16
                    const uint32_t s_tm = tmem + (t & 1) * kN;
                    const uint32_t kb = sbase + stage * kStageBytes;
                    const uint32_t qa = sbase + kQOff + qb * kQBytes;
                    // descriptors of the first K step; a later step adds its
                    // offset / 16 to the start-address field (no carry below
                    // 256 KiB), so no MMA rebuilds one
                    const uint64_t kdesc = tc::sw128_desc(kb, 16, 1024), qdesc = tc::sw128_desc(qa, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t ko = (kk >> 2) * kHalf + (kk & 3) * 32;
                        const uint32_t qo = (kk >> 2) * kQHalf + (kk & 3) * 32;
                        tc::mma_ss(s_tm, kdesc + (ko >> 4), qdesc + (qo >> 4), kIdS, kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&ms->s_full[t & 1]);
                    if (d.flags & kLast) {
                        tc::commit(&ms->q_empty[qb]);
                        ++ic;
                    }
                    ++t;
                    if (++stage == kStages) {
                        stage = 0;
                        sph ^= 1;
                    }
                }
            } else {
                constexpr uint32_t kIdPV = tc::idesc_bf16_f32_major(kRows, kON, true, false);
                for (;;) {
                    if (!mbar_wait_bounded(&ms->full[stage], sph, abort_flag, p.wait_ns))
                        break;
                    if (ms->desc[stage].flags & kEnd)
                        break;
                    if (!mbar_wait_bounded(&ms->o_empty[t & 1], ((t >> 1) & 1) ^ 1, abort_flag, p.wait_ns))
                        break;
                    // O_t^T = V^T P^T: A = V (MN-major: the two 64-dim halves
                    // 16 KiB apart, 8-key groups 1 KiB apart), B = P (K-major).
                    // Warp w's keys 32w .. 32w + 31 (K steps 2w, 2w + 1) go as
                    // soon as that warp has written its weights.
                    const uint32_t o_tm = tmem + kOCol + (t & 1) * kON;
                    const uint32_t vb = sbase + stage * kStageBytes + kTileBytes;
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
                    tc::commit(&ms->kv_empty[stage]);
                    ++t;
                    if (++stage == kStages) {
                        stage = 0;
                        sph ^= 1;
                    }
                }
            }
            // Every MMA this thread issued completes before the TMEM is freed.
            tc::commit(&ms->mma_done);
            int drain_abort = 0;
            mbar_wait_bounded(&ms->mma_done, 0, &drain_abort);
        }
        __syncwarp();
    } else if (warp >= kSoftWarp0) {
        // ------------------------------------------------------------ softmax + accumulation
        // Each warp w runs its own online softmax over its 32 key rows of
        // every tile (running maximum mw, weight sums), so no tile needs an
        // exchange between warps: its weights go to the P rows of (w, head),
        // and the value product keeps one column per (w, head), hi and lo.
        // Thread (w, lane) accumulates output dimension 32 w + lane of all
        // four warps' columns, each against that warp's maximum (the factors
        // come through shared memory); the four are merged at the item end.
        const int q4 = warp - kSoftWarp0;  // TMEM lane quadrant (warp % 4)
        const int row = q4 * 32 + lane;    // key row of a tile; output dimension
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        int stage = 0;
        uint32_t sph = 0, gph = 0;
        int t = 0;
        float mw[G], l_run[G], o[4][G];
        int unit = 0, split = 0, b = 0, kvh = 0;
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
        // o[w] = o[w] * alpha_w + O_x[w] for the four warps' columns of tile x
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
            bool w = mbar_wait_bounded(&ms->s_full[t & 1], (t >> 1) & 1, abort_flag, p.wait_ns);
            w = w && mbar_wait_bounded(&ms->full[stage], sph, abort_flag, p.wait_ns);  // descriptor and V visible
            if (!__all_sync(kFull, w))
                break;
            const TileDesc d = ms->desc[stage];
            if (d.flags & kEnd) {
                ended = true;
                break;
            }
            if (d.flags & kFirst) {
                unit = p.cm.unit_of(d.item);
                split = p.cm.split_of(d.item);
                b = unit / p.Hkv;
                kvh = unit - b * p.Hkv;
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
                s[g] = valid ? __uint_as_float(sr[g]) * p.qscale : -INFINITY;  // log2 units
                mx[g] = s[g];
            }
            // The warp's reference mw is raised only when a score exceeds it
            // by more than 2^8 (a warp vote), so the weights stay below 2^8;
            // then to the warp's maximum, with the factor alpha for the sums.
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
            // P^T: rows w*G + g (hi) and 16 + w*G + g (lo), column `row`
            // (key), 128-byte swizzle: the 16-byte chunk index within a
            // 128-byte row is xor-ed with row % 8
            unsigned char *pbase = smem + kPOff + (t & 1) * kPBytes;
            const int cb = (row & 63) * 2;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int rh = q4 * G + g, rl = kN + rh;
                const int base = (row >> 6) * kPHalf + (cb & 15);
                const __nv_bfloat16 hi = __float2bfloat16_rn(pw[g]);
                const __nv_bfloat16 lo = __float2bfloat16_rn(pw[g] - __bfloat162float(hi));
                *reinterpret_cast<__nv_bfloat16 *>(pbase + base + rh * 128 + ((((cb >> 4) ^ rh) & 7) << 4)) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(pbase + base + rl * 128 + ((((cb >> 4) ^ rl) & 7) << 4)) = lo;
            }
            // V rows of keys past the tile's end may hold anything (padding
            // past a sequence's length): zero them so that 0 * V stays 0
            if (d.n < kTile && row >= d.n && row < kTile) {
                unsigned char *vr = smem + stage * kStageBytes + kTileBytes + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    *reinterpret_cast<uint4 *>(vr + c * 16) = z4;
                    *reinterpret_cast<uint4 *>(vr + kHalf + c * 16) = z4;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc::fence_before_sync();
            mbar_arrive(&ms->p_full[t & 1][q4]);
            mbar_arrive(&ms->p_all[t & 1]);
            if (!(d.flags & kFirst) && !accumulate(t - 1))
                break;
            const int tt = t;
            ++t;
            if (++stage == kStages) {
                stage = 0;
                sph ^= 1;
            }
            if (!(d.flags & kLast))
                continue;
            if (!accumulate(tt))
                break;

            // ---- end of item: the partial, the result, and in fused mode the merge
            if (!tcd::finish_item<G, OUT, kMergeBatch>(io, &ms->isum, stage_area, q4, lane, unit, split, b, kvh, 1.f, mw, l_run,
                                          o, pt, group_sync))
                break;
        }
        if (ended)
            tcd::finish_pending<G, OUT, kMergeBatch>(io, &ms->isum, stage_area, q4, lane, pt, group_sync, smem,
                                                     (size_t)kStages * kStageBytes);
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

template <int G, typename OUT>
cudaError_t launch_typed(const DecodeLaunch &a, const TcParams &p)
{
    auto kern = decode_tc_kernel<G, OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess)
        return e;
    kern<<<a.plan.grid, kThreads, kSmem, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool decode_tc_eligible(const DecodeLaunch &a)
{
    const int G = a.Hq / a.Hkv;
    // a paged cache whose pages tile the 128-key tiles (page sizes 8, 16, 32,
    // 64 or multiples of 128: one TMA box per page piece, on the 128-byte
    // swizzle's 8-row grid); other page sizes go to the CUDA-core kernel
    // (and tiles that start on a multiple of 128 keys: chunks of whole tiles)
    const bool tiles_aligned = a.plan.n_split == 1 || a.plan.chunk % kTile == 0;
    const bool pages_ok = !a.block_table || (tiles_aligned && ((a.page_size % 128 == 0) ||
                          (a.page_size >= 8 && a.page_size <= 64 && 128 % a.page_size == 0)));
    return a.D == kD && (G == 2 || G == 4) && a.in_dtype == TA_BF16 && !a.kv_fp8 && !a.kv_nvfp4 && pages_ok;
}

cudaError_t launch_decode_tc(const DecodeLaunch &a)
{
    const int G = a.Hq / a.Hkv;
    TcParams p;
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
    p.k = a.k;
    p.v = a.v;
    p.pi_window = a.pi_window;
    p.pi_period = a.pi_period;
    // Tensor maps, boxes of 64 dims (128 bytes, the swizzle span):
    //   q [B, Hq, D] as (D, G, B*Hkv), box G rows;
    //   K, V [B, Hkv, S, D] as (D, S, B*Hkv), boxes of 128 and 8 rows;
    //   pi-Attention: each (sequence, KV head) as rows of pi_period keys,
    //     (pi*D, ceil(S/pi), B*Hkv): the box at x = r*D, y = m holds keys
    //     r + (m + t) * pi; it is only used where all its rows are keys of
    //     the periodic part, so below S of that (sequence, KV head).
    const uint64_t units = (uint64_t)a.B * a.Hkv;
    const uint64_t qd[3] = {(uint64_t)kD, (uint64_t)G, units};
    const uint64_t qs[2] = {(uint64_t)kD * 2, (uint64_t)G * kD * 2};
    const uint32_t qbox[3] = {64, (uint32_t)G, 1};
    const uint32_t boxt[3] = {64, (uint32_t)kTile, 1};
    const uint32_t box8[3] = {64, 8, 1};
    const uint64_t kd[3] = {(uint64_t)kD, (uint64_t)a.S, units};
    const uint64_t ks[2] = {(uint64_t)kD * 2, (uint64_t)a.S * kD * 2};
    bool ok = encode_tmap_3d(&p.qmap, a.q, true, qd, qs, qbox, true);
    // maps a launch does not use are copies of the q map (never read)
    p.kmap = p.vmap = p.k8map = p.v8map = p.qmap;
    p.kpimap = p.vpimap = p.kpi8map = p.vpi8map = p.qmap;
    p.kpgmap = p.vpgmap = p.qmap;
    p.block_table = a.block_table;
    p.page_size = a.page_size;
    p.pages_per_seq = a.pages_per_seq;
    p.num_pages = a.num_pages;
    p.pg_rows = a.page_size < kTile ? a.page_size : kTile;
    if (a.block_table) {
        // page pools [num_pages, Hkv, page_size, D] as (D, page_size, num_pages * Hkv)
        const uint64_t gd[3] = {(uint64_t)kD, (uint64_t)a.page_size, (uint64_t)a.num_pages * a.Hkv};
        const uint64_t gs[2] = {(uint64_t)kD * 2, (uint64_t)a.page_size * kD * 2};
        const uint32_t gbox[3] = {64, (uint32_t)p.pg_rows, 1};
        ok = ok && encode_tmap_3d(&p.kpgmap, a.k, true, gd, gs, gbox, true) &&
             encode_tmap_3d(&p.vpgmap, a.v, true, gd, gs, gbox, true);
    } else {
        ok = ok && encode_tmap_3d(&p.kmap, a.k, true, kd, ks, boxt, true) &&
             encode_tmap_3d(&p.vmap, a.v, true, kd, ks, boxt, true) &&
             encode_tmap_3d(&p.k8map, a.k, true, kd, ks, box8, true) &&
             encode_tmap_3d(&p.v8map, a.v, true, kd, ks, box8, true);
    }
    if (a.pi_period > 0) {
        const uint64_t per = (uint64_t)a.pi_period;
        const uint64_t pd[3] = {per * kD, ((uint64_t)a.S + per - 1) / per, units};
        const uint64_t ps[2] = {per * kD * 2, (uint64_t)a.S * kD * 2};
        ok = ok && encode_tmap_3d(&p.kpimap, a.k, true, pd, ps, boxt, true) &&
             encode_tmap_3d(&p.vpimap, a.v, true, pd, ps, boxt, true) &&
             encode_tmap_3d(&p.kpi8map, a.k, true, pd, ps, box8, true) &&
             encode_tmap_3d(&p.vpi8map, a.v, true, pd, ps, box8, true);
    }
    if (!ok)
        return cudaErrorInvalidValue;
    const bool bf16_out = a.out_dtype == TA_BF16;
    if (G == 2)
        return bf16_out ? launch_typed<2, __nv_bfloat16>(a, p) : launch_typed<2, float>(a, p);
    return bf16_out ? launch_typed<4, __nv_bfloat16>(a, p) : launch_typed<4, float>(a, p);
}

}  // namespace ta
