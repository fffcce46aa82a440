// K-attend: split-K flash-decode on the 5th-generation tensor cores, with the
// split merge inside the same kernel.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 技术细节 / 架构概览,
// per-layer box step 3 (indexed_cached_attention over window + selected rows)
// and "Memory Layout" (window KV [128, kv_dim] plus staging slots [gpu_chunks,
// kv_dim], one fp32 latent row per entry). Every head attends over the same
// rows (MQA over the latent, K = V = row):
//     o_h = sum_j softmax_j(<q_h, e_j> / sqrt(512)) e_j.
//
// Work: the rows of one (layer, sequence) -- the 128 window rows, then the
// layer's staged rows in selection order -- form tiles of 128 rows. A static
// plan built at context creation gives each CTA a list of segments (a range
// of tiles of one pair): one chunk of one pair when every pair's chunks fit
// one wave, otherwise a contiguous range of the whole call's tiles. Each row
// is read from HBM once per call.
//
// One CTA of 16 warps per SM. A CTA's row stream is bound by the bytes it
// keeps in flight, so every warp streams rows: warp w owns tile rows w + 16 j
// (j < 8), 1 KiB of contiguous bytes per load instruction (32-byte loads).
// A tile of fp16 staged rows has all eight of a warp's rows in flight; a tile
// holding fp32 window rows (2 KiB each) four, each row's registers taking the
// next row once stored: 128 KB in flight per CTA either way. Every row is
// stored once, as fp16, into one resident 128B-swizzled tile E [128 rows x
// 512 d] (8 d-blocks of 64). Rows past the segment's end are zero-filled, not
// loaded.
//   pass 1  S^T[r, h] = E[r, :] . Q[h, :]   (M = 128 rows, N = heads, K = 512),
//           E and Q K-major;
//   softmax every warp: warp w reads TMEM lanes 32 (w % 4) (its rows) and the
//           H/4 head columns of group w / 4; per-head tile max and sum by warp
//           reductions and a 4-warp exchange in shared memory; base-2 online
//           softmax with a lazily moved reference max (moved only when the tile
//           max exceeds it by 2^8); P written as fp16 [rows x heads];
//   pass 2  O^T[d, h] += E^T[d, r] P[r, h]   (M = 128 d, N = heads, K = rows),
//           the SAME smem tile read MN-major (a 128B-swizzled atom of 8 rows x
//           64 d serves both views), so no row is fetched twice.
// Both products are tcgen05 kind::f16 MMAs with fp32 accumulation in TMEM,
// issued by thread 0. fp16 keeps 11 significant bits, as tf32 does; 32-bit
// operands cannot be MN-major, which pass 2 needs. A latent or query value
// beyond fp16's finite range (65504) sets kErrRange; the results of that call
// are then not to be used. p <= 2^8 by construction, and bf16 queries of
// normal fp16 range convert exactly.
//
// With more than one tile in a segment, the next tile's rows are requested
// into L2 (one bulk prefetch per row) when a tile starts, so HBM keeps
// streaming while the tile's products and softmax run; its loads then find the
// rows in L2. Every wait is bounded; on a timeout the CTA records kErrTimeout,
// drains its MMAs, frees TMEM and returns.
//
// A pair spread over several segments: each segment writes its normalized
// output as fp16, (O / l) / sc with sc the power of two at or below the
// largest |row value| it read (so the values stay in fp16's normal range),
// with its statistics (m, l, sc), and raises the pair's arrival counter. When a CTA has run all its segments, it waits (bounded) for
// the counters of the split pairs it took part in and merges its share of each
// such pair's output, in split order:
//     o_h = sum_s w_s O_s[h] / l_s,   w_s = l_s 2^(m_s - M) / sum_s' l_s' 2^(m_s' - M),
// each stored partial multiplied back by its sc_s (folded into w_s).
// The CTAs of the grid wait on one another only there. A plan never has more
// CTAs than SMs and a CTA takes a whole SM, so every CTA of the grid becomes
// resident once the kernels ahead of it leave their SMs; the wait is bounded
// all the same. The plan depends only on the configuration, so identical rows
// give identical bits whatever slots hold them.
#include <cmath>
#include <cstddef>

#include "srh_internal.cuh"
#include "umma.cuh"

namespace srh {
namespace {

using namespace umma;

constexpr int kTileRows = kAttnTile;                // 128
static_assert(kWindow == kTileRows, "a pair's first tile is exactly its window rows");
constexpr int kThreads = 512;                       // 16 warps
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kTileRows / kWarps;    // 8 tile rows per warp
constexpr int kOffQ = 0;                            // 8 d-blocks x 8 KB: fp16 Q, K-major, row h
constexpr int kDBlockE = kTileRows * 128;           // 16 KB: one d-block of E
constexpr int kOffE = kOffQ + 8 * 8192;             // 8 d-blocks: fp16 E, row r
constexpr int kOffP = kOffE + 8 * kDBlockE;         // fp16 P [128 rows x 64 heads], heads contiguous
constexpr int kOffMisc = kOffP + kTileRows * 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                       // S^T: up to 64 columns
constexpr uint32_t kColO = 64;                      // O^T[mb]: 64 columns each
constexpr float kLazy = 8.0f;                       // reference max moves past 2^8 growth
constexpr int kMaxSplits = (kWindow + kMaxSelect + kTileRows - 1) / kTileRows;
constexpr int kMaxDuties = 4;                       // split pairs one CTA takes part in
constexpr int kMlStride = kAttnMlStride;            // floats per partial's statistics: m, l, scale
// A merge's inputs in the E area: each split's share of the partial (16 bytes
// per 8 values), then the splits' statistics.
constexpr int kMergeMlOff = 72 * 1024;
constexpr int kMergeWOff = 92 * 1024;                // the combined weights [split][head]
static_assert(64 * kKvDim * 2 + kMaxSplits * (16 + 127) <= kMergeMlOff, "merge shares overlap the statistics");
static_assert(kMergeMlOff + kMaxSplits * kMlStride * 4 <= kMergeWOff, "merge statistics overlap the weights");
static_assert(kMergeWOff + kMaxSplits * 64 * 4 <= 8 * kDBlockE, "merge inputs exceed the E area");
static_assert((kMlStride * 4) % 16 == 0, "partial statistics rows must be 16-byte multiples");

struct Misc {
    uint64_t s_full, o_full, drain, q_full, m_full;
    uint32_t tmem_base;
    int abort;
    int n_duties;
    int duty_merge[kMaxDuties];
    int duty_part[kMaxDuties];
    unsigned long long duty_target[kMaxDuties];
    // read and written as float4: 16-byte aligned
    alignas(16) float m_used[2][64];    // reference max per head (parity of the segment's tile)
    alignas(16) float l_run[2][64];     // running sum per head
    alignas(16) float red[4][64];       // per-quadrant tile maxima
    alignas(16) float red2[4][64];      // per-quadrant tile sums
    alignas(16) float alpha[64];        // this tile's rescale factor per head
    alignas(16) uint32_t wmax[kWarps];  // per-warp max |row value| (bits) of the segment
    alignas(16) float inv_l[64];        // 1 / l per head at a segment's end
};
static_assert(offsetof(Misc, m_used) % 16 == 0 && offsetof(Misc, red) % 16 == 0 && offsetof(Misc, inv_l) % 16 == 0 &&
                  offsetof(Misc, l_run) % 16 == 0 && offsetof(Misc, red2) % 16 == 0 && offsetof(Misc, alpha) % 16 == 0,
              "float4-accessed softmax state must be 16-byte aligned");
static_assert(kOffMisc % 16 == 0, "Misc must start 16-byte aligned");
constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc) + 1024;   // + base alignment slack
static_assert(kSmemBytes <= 232448, "attention shared memory exceeds 227 KB");

// f16-kind instruction descriptor: f16 A and B, f32 accumulate, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(int a_mn, int b_mn, int n) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

struct AttnArgs {
    const AttnSeg* segs;
    const int* cta_begin;   // CTA k runs segs[cta_begin[k] .. cta_begin[k + 1])
    const MergeItem* merges;
    unsigned long long* merge_cnt;   // arrivals per split pair (monotonic across calls)
    int B, G, S;
    const uint16_t* q;
    const float* window;
    const uint16_t* staging;   // fp16 staged rows
    const int32_t* phys;
    const int32_t* count_l;
    float* out;
    uint16_t* part_o;       // fp16 [slot][H][512]: (O / l) / sc of one segment
    float* part_ml;         // [slot][kMlStride]: m [H], l [H], sc
    uint32_t* err;
    float sl2;              // log2(e) / sqrt(kv_dim)
};

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Read-only streaming load of 32 bytes (no L1 allocation); p is 32-byte aligned.
__device__ __forceinline__ void ldg_stream8(const float* p, float4& lo, float4& hi) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
                 : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z), "=f"(hi.w)
                 : "l"(p));
}

// Bulk copy of bytes (a multiple of 16, both addresses 16-byte aligned) from
// global memory into shared memory, completing on bar's transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// 2^x by the hardware's approximate exponential (relative error about 2^-22,
// far below the fp16 rounding that every weight p gets next); subnormal
// results flush to zero. ex2(-inf) = 0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// The fp16 value in the low half of x times 2^-112, exactly: its sign, and its
// exponent and mantissa bits moved to the fp32 positions (an fp16 subnormal
// becomes an fp32 subnormal; no flush to zero is in force). Finite inputs only.
__device__ __forceinline__ float f16_bits_scaled(uint32_t x) {
    return __uint_as_float(((x & 0x8000u) << 16) | ((x & 0x7fffu) << 13));
}

__device__ __forceinline__ float f16_to_f32(uint32_t h) {
    float f;
    asm("{\n .reg .f16 t;\n mov.b16 t, %1;\n cvt.f32.f16 %0, t;\n}\n" : "=f"(f) : "h"((unsigned short)h));
    return f;
}

// Maximum over the 32 lanes of a warp (every lane receives it); -inf lanes
// take part like any other value.
__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(v));
    return r;
}

// Sum over the 32 lanes of a warp for N per-lane columns at once. The
// first log2(N) steps hand half of the columns to the partner lane; afterwards
// lane l holds column l / (32 / N), reduced over every lane.
template <int N>
__device__ __forceinline__ float sum_cols(float (&v)[N], int lane) {
#pragma unroll
    for (int s = 0; (1 << s) < N; ++s) {
        const int bit = 16 >> s;
        const int half = N >> (s + 1);
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, bit);
            v[i] = keep + recv;
        }
    }
#pragma unroll
    for (int bit = 16 / N; bit >= 1; bit >>= 1) {
        const float recv = __shfl_xor_sync(0xffffffffu, v[0], bit);
        v[0] += recv;
    }
    return v[0];
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1) attend_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int HPG = H / 4;                       // heads per softmax group (4 groups of 4 warps)
    constexpr int kQPer = H * 64 / kThreads;         // 16-byte query chunks per thread
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Misc& ms = *reinterpret_cast<Misc*>(sm + kOffMisc);
    volatile int* abort = &ms.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, grp = warp >> 2;      // TMEM lane quadrant; softmax / epilogue group

    // this CTA's segments of the static plan (written once, at creation)
    const int sb = a.cta_begin[blockIdx.x], se = a.cta_begin[blockIdx.x + 1];
    pdl_trigger();

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.o_full, 1);
        mbar_init(&ms.drain, 1);
        mbar_init(&ms.q_full, 1);
        mbar_init(&ms.m_full, 1);
        ms.abort = 0;
        ms.n_duties = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&ms.tmem_base, kTmemCols);
    float amax = 0.f;   // largest |value| converted to fp16 by this thread (range guard)
    float ramax = 0.f;  // largest |row value| of the current segment (scale of its partial)
    uint32_t rbits = 0; // ... of its fp16 staged rows: two maxima of |fp16| bit patterns

    // Wait for an mbarrier phase: thread 0 polls, every other thread waits at
    // the block barrier that follows (a waiting warp issues nothing). Returns
    // true, block-uniformly, if the CTA has failed.
    auto block_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (tid == 0 && !mbar_wait(bar, parity)) {
            atomicOr(a.err, kErrTimeout);
            ms.abort = 1;
        }
        const bool f = __syncthreads_or(*abort != 0);
        tc_fence_after();
        return f;
    };
    // Queries of pair lbq: bf16 [H][512], copied as they are into the E area
    // (free between segments) by one bulk copy per 16 KiB, then converted to
    // fp16 K-major in the Q area: d-block d / 64 at (d / 64) * 8192, row h.
    uint32_t q_uses = 0;                             // phases of q_full
    auto fetch_q = [&](int lbq) {                    // thread 0
        const unsigned char* qg = reinterpret_cast<const unsigned char*>(a.q + (size_t)lbq * H * kKvDim);
        constexpr uint32_t kBytes = H * kKvDim * 2, kPiece = 16384;
        mbar_arrive_expect_tx(&ms.q_full, kBytes);
#pragma unroll 1
        for (uint32_t o = 0; o < kBytes; o += kPiece)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                    smem_u32(sm + kOffE + o)),
                "l"(qg + o), "r"(kPiece), "r"(smem_u32(&ms.q_full))
                : "memory");
    };
    // after q_full's phase and a block barrier: every thread converts its chunks
    auto convert_q = [&]() {
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int i = tid + k * kThreads, h = i >> 6, c8 = i & 63;
            const uint4 v = *reinterpret_cast<const uint4*>(sm + kOffE + (size_t)i * 16);
            const float f[8] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u),
                                __uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                                __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u)};
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
            const uint4 w = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                                       pack_f16x2(f[6], f[7]));
            *reinterpret_cast<uint4*>(sm + kOffQ + (c8 >> 3) * 8192 + sw128(h, c8 & 7)) = w;
        }
    };
    // Half h2 (d 256 h2 .. +255) of a tile row: this lane's 8 values d = 8 lane
    // + 256 h2 .. + 7, as fp16 into E row r: d-block (lane >> 3) + 4 h2, 16-byte
    // chunk lane & 7.
    auto store_half = [&](const float4& lo, const float4& hi, int r, int h2) {
        const float t = fmaxf(fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(lo.z), fabsf(lo.w))),
                              fmaxf(fmaxf(fabsf(hi.x), fabsf(hi.y)), fmaxf(fabsf(hi.z), fabsf(hi.w))));
        amax = fmaxf(amax, t);
        ramax = fmaxf(ramax, t);
        *reinterpret_cast<uint4*>(sm + kOffE + ((lane >> 3) + 4 * h2) * kDBlockE + sw128(r, lane & 7)) =
            make_uint4(pack_f16x2(lo.x, lo.y), pack_f16x2(lo.z, lo.w), pack_f16x2(hi.x, hi.y), pack_f16x2(hi.z, hi.w));
    };
    auto zero_half = [&](int r, int h2) {
        *reinterpret_cast<uint4*>(sm + kOffE + ((lane >> 3) + 4 * h2) * kDBlockE + sw128(r, lane & 7)) =
            make_uint4(0u, 0u, 0u, 0u);
    };

    // Rows [row0, row1) of segment sg: the count comes from the resolve kernel.
    auto seg_rows = [&](const AttnSeg& sg, int& row0, int& row1) {
        int cnt = a.count_l[sg.lb];
        if (cnt < 0 || cnt > a.S) {
            if (tid == 0) atomicOr(a.err, kErrBounds);
            cnt = cnt < 0 ? 0 : a.S;
        }
        row0 = sg.r0;
        row1 = min(kWindow + cnt, sg.r1);
    };
    // Ask L2 for the rows of the tile at tr0 of pair lb (threads 0-127, one
    // 2 KiB bulk prefetch each): no registers or shared memory, so HBM streams
    // the whole tile while its loads and the products of the tile before run.
    auto prefetch_tile = [&](size_t lb, int tr0, int row1) {
        const int row = tr0 + tid;
        if (tid >= kTileRows || row >= row1) return;
        const void* p;
        uint32_t bytes;
        if (row < kWindow) {
            p = a.window + (lb * kWindow + row) * kKvDim;
            bytes = kKvDim * 4;
        } else {
            const int slot = a.phys[lb * a.S + row - kWindow] - kWindow;
            if (slot < 0 || slot >= a.G) return;            // reported by the loads
            p = a.staging + (lb * (size_t)a.G + slot) * kKvDim;
            bytes = kKvDim * 2;
        }
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
    };

    // the barriers, the abort flag and the TMEM address are set; every thread sees them from here on
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // The first segment's queries are this call's own input: their copy is
    // issued before the dependency wait.
    int q_lb = -1;
    if (sb < se) {
        if (tid == 0) fetch_q(a.segs[sb].lb);
        q_lb = a.segs[sb].lb;
    }

    // Slots, counts and staged rows come from earlier kernels, and the partial
    // buffers and arrival counts are shared with the previous call: all of them
    // are touched only after the dependency wait. A CTA whose first segment
    // starts with the window tile runs that tile (rows, queries, both products)
    // before the wait, while the earlier kernels still run.
    bool dep_ready = false;
    auto dep_wait = [&]() {
        if (!dep_ready) {
            pdl_wait();
            dep_ready = true;
        }
    };
    bool q_pending = sb < se;   // a queries' copy into the E area is issued and not yet converted

    constexpr uint32_t id1 = idesc_f16(0, 0, H);   // pass 1: K-major E and Q
    constexpr uint32_t id2 = idesc_f16(1, 1, H);   // pass 2: MN-major E^T and P
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint32_t gt = 0;            // tiles this CTA has run (mbarrier phases of s_full / o_full)
    bool failed = false;        // block-uniform: a wait gave up (the abort flag, OR-ed at a barrier)

    int si = sb;
    for (; si < se; ++si) {
        const AttnSeg sg = a.segs[si];
        const size_t lb = (size_t)sg.lb;
        // a first tile of window rows only (always present) of the CTA's first
        // segment runs before the wait; the segment's other rows are known after it
        const bool early = !dep_ready && sg.r0 < kWindow && sg.r1 > sg.r0 && (sg.r0 == 0 || sg.r1 <= kWindow);
        int row0 = sg.r0, row1 = min(sg.r1, kWindow), n_tiles = 1;
        // A split pair's arrival count before this CTA's own arrival (read after
        // the dependency wait: every earlier call's arrivals are in). The pair is
        // complete when it reaches the next multiple of its split count.
        unsigned long long seen = 0;
        const int32_t* ph = a.phys + lb * a.S;
        // Sources of this warp's rows w + 16 i (lane i < 8) of the tile at tr0:
        // -1 - row for a window row, else the row's phys entry (window + slot).
        // Bounded by the plan's rows, not by the count: the first tile's entries
        // are loaded together with the count (an entry past the count is never
        // used: every row load, store and slot check is bounded by row1).
        auto fetch_src = [&](int tr0) -> int {
            const int row = tr0 + warp + kWarps * (lane & 7);
            if (lane >= kRowsPerWarp || row >= sg.r1) return -1;
            return row < kWindow ? -1 - row : ph[row - kWindow];
        };
        int src0 = INT_MIN;           // the first tile's sources, when taken beside the count
        auto seg_after_wait = [&]() {
            seg_rows(sg, row0, row1);
            n_tiles = row1 > row0 ? (row1 - row0 + kTileRows - 1) / kTileRows : 0;
            if (sg.slot >= 0 && tid == 0) seen = ld_relaxed_u64(&a.merge_cnt[sg.merge]);
        };
        if (!early) {
            dep_wait();
            src0 = fetch_src(row0);   // issued before the count is used (no loads for window rows)
            seg_after_wait();
        }
        if (si > sb && n_tiles > 0 && sg.lb != q_lb) {
            // the previous segment drained its MMAs before its epilogue: Q and E are
            // free; a copy that an earlier segment without rows left unused lands first
            if (q_pending && block_wait(&ms.q_full, q_uses & 1)) {
                failed = true;
                break;
            }
            if (q_pending) ++q_uses;
            if (tid == 0) fetch_q(sg.lb);
            q_lb = sg.lb;
            q_pending = true;
        }
        if (tid < 64) {
            ms.m_used[0][tid] = -INFINITY;
            ms.l_run[0][tid] = 0.f;
        }
        ramax = 0.f;
        rbits = 0u;

        auto staged_ptr = [&](int src) -> const uint16_t* {
            int slot = src - kWindow;
            if (slot < 0 || slot >= a.G) {
                atomicOr(a.err, kErrBounds);
                slot = 0;
            }
            return a.staging + (lb * (size_t)a.G + slot) * kKvDim;
        };
        // window row w + 16 j (j < 8) of the tile at tr0 (fp32): the whole row,
        // 1 KiB of contiguous bytes per load instruction
        auto load_row = [&](float4 (&v)[4], int tr0, int j, int src) {
            const int s = __shfl_sync(0xffffffffu, src, j);
            if (tr0 + warp + kWarps * j < row1) {
                const float* p = a.window + (lb * kWindow + (-1 - s)) * kKvDim + 8 * lane;
                ldg_stream8(p, v[0], v[1]);
                ldg_stream8(p + 256, v[2], v[3]);
            }
        };
        // staged row w + 16 j (fp16, 1 KiB): this lane's 16 values d = 16 lane ..
        auto load_row_h = [&](float4& lo, float4& hi, int tr0, int j, int src) {
            const int s = __shfl_sync(0xffffffffu, src, j);
            if (tr0 + warp + kWarps * j < row1)
                ldg_stream8(reinterpret_cast<const float*>(staged_ptr(s) + 16 * lane), lo, hi);
        };
        // as they are into E row r: d-block lane / 4, 16-byte chunks 2 (lane % 4) and + 1
        auto store_row_h = [&](const float4& lo, const float4& hi, int tr0, int j) {
            const int r = warp + kWarps * j;
            unsigned char* e = sm + kOffE + (lane >> 2) * kDBlockE;
            const int c = 2 * (lane & 3);
            uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
            if (tr0 + r < row1) {
                w0 = make_uint4(__float_as_uint(lo.x), __float_as_uint(lo.y), __float_as_uint(lo.z), __float_as_uint(lo.w));
                w1 = make_uint4(__float_as_uint(hi.x), __float_as_uint(hi.y), __float_as_uint(hi.z), __float_as_uint(hi.w));
                const uint32_t m = __vmaxu2(__vmaxu2(__vmaxu2(w0.x & 0x7fff7fffu, w0.y & 0x7fff7fffu),
                                                     __vmaxu2(w0.z & 0x7fff7fffu, w0.w & 0x7fff7fffu)),
                                            __vmaxu2(__vmaxu2(w1.x & 0x7fff7fffu, w1.y & 0x7fff7fffu),
                                                     __vmaxu2(w1.z & 0x7fff7fffu, w1.w & 0x7fff7fffu)));
                rbits = __vmaxu2(rbits, m);
            }
            *reinterpret_cast<uint4*>(e + sw128(r, c)) = w0;
            *reinterpret_cast<uint4*>(e + sw128(r, c + 1)) = w1;
        };
        auto store_row = [&](const float4 (&v)[4], int tr0, int j) {
            const int r = warp + kWarps * j;
            if (tr0 + r < row1) {
                store_half(v[0], v[1], r, 0);
                store_half(v[2], v[3], r, 1);
            } else {
                zero_half(r, 0);
                zero_half(r, 1);
            }
        };
        // row w + 16 j of a tile that holds window rows: fp32 or fp16 by its place
        auto load_any = [&](float4 (&v)[4], int tr0, int j, int src) {
            if (tr0 + warp + kWarps * j < kWindow) load_row(v, tr0, j, src);
            else load_row_h(v[0], v[1], tr0, j, src);
        };
        auto store_any = [&](const float4 (&v)[4], int tr0, int j) {
            if (tr0 + warp + kWarps * j < kWindow) store_row(v, tr0, j);
            else store_row_h(v[0], v[1], tr0, j);
        };
        auto issue_pass1 = [&](int x0) {   // d-blocks x0 .. x0 + 3 (thread 0)
            const uint32_t e0 = smem_u32(sm + kOffE), q0 = smem_u32(sm + kOffQ);
#pragma unroll 1
            for (int x = x0; x < x0 + 4; ++x)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16kind(ms.tmem_base + kColS, desc_sw128(e0 + x * kDBlockE + kk * 32, 16, 1024),
                                desc_sw128(q0 + x * 8192 + kk * 32, 16, 1024), id1, (x | kk) != 0);
        };

        for (int tile = 0; tile < n_tiles; ++tile) {
            const int tr0 = row0 + tile * kTileRows;
            const int par = tile & 1;
            if (tile + 1 < n_tiles) prefetch_tile(lb, tr0 + kTileRows, row1);
            // ------------------------------------------------------------ E (all warps)
            int src;                                  // this tile's row sources (lanes 0-7)
            if (src0 != INT_MIN) {
                src = src0;
                src0 = INT_MIN;
            } else {
                src = fetch_src(tr0);
            }
            const bool mixed = tr0 < kWindow;         // window rows (fp32) in the tile
            float4 v[4][4];
            if (mixed) {
                // four rows in flight per warp (128 KB per CTA); each row's registers
                // take the next row's loads as soon as they are stored, so the
                // stream does not drain between the tile's two halves
#pragma unroll
                for (int i = 0; i < 4; ++i) load_any(v[i], tr0, i, src);
            } else {
                // staged rows, fp16: all eight of this warp's rows in flight at once
#pragma unroll
                for (int j = 0; j < 8; ++j) load_row_h(v[j >> 1][2 * (j & 1)], v[j >> 1][2 * (j & 1) + 1], tr0, j, src);
            }
            if (q_pending) {
                // the queries' copy has landed in the E area: convert it while the rows arrive
                if (block_wait(&ms.q_full, q_uses & 1)) {
                    failed = true;
                    break;
                }
                ++q_uses;
                convert_q();
                __syncthreads();   // every thread is done reading the E area
                q_pending = false;
            }
            // the previous tile's pass 2 reads E: wait for it before overwriting
            if (tile > 0 && block_wait(&ms.o_full, (gt - 1) & 1)) {
                failed = true;
                break;
            }
            if (mixed) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    store_any(v[i], tr0, i);
                    load_any(v[i], tr0, 4 + i, src);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) store_any(v[i], tr0, 4 + i);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) store_row_h(v[j >> 1][2 * (j & 1)], v[j >> 1][2 * (j & 1) + 1], tr0, j);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // ------------------------------------------------------------ pass 1 (thread 0)
            if (tid == 0) {
                issue_pass1(0);
                issue_pass1(4);
                mma_commit(&ms.s_full);
            }
            const uint32_t tmem = ms.tmem_base;

            // ------------------------------------------------------------ softmax (all warps)
            const int r = quad * 32 + lane;               // tile row = TMEM lane
            if (block_wait(&ms.s_full, gt & 1)) {
                failed = true;
                break;
            }
            const uint32_t ts = tmem + lane_base + kColS + HPG * grp;
            const bool valid = tr0 + r < row1;
            float sv[HPG];
            tmem_ld<HPG>(ts, sv);                            // stale after an abort, then unused
            tmem_ld_wait();
            tmem_regs_ready_n(sv);
#pragma unroll
            for (int i = 0; i < HPG; ++i) sv[i] = valid ? sv[i] * a.sl2 : -INFINITY;
            {
                // each head's maximum over this warp's 32 rows: one warp reduction per column
                float mx[HPG];
#pragma unroll
                for (int i = 0; i < HPG; ++i) mx[i] = warp_max(sv[i]);
                if (lane == 0) {
#pragma unroll
                    for (int c = 0; c < HPG / 4; ++c)
                        *reinterpret_cast<float4*>(&ms.red[quad][HPG * grp + 4 * c]) =
                            make_float4(mx[4 * c], mx[4 * c + 1], mx[4 * c + 2], mx[4 * c + 3]);
                }
            }
            named_sync(1 + grp, 128);
            // lane i < HPG: head HPG * grp + i's tile maximum over the four quadrants
            // and its reference max (every warp of the group computes the same)
            float mn = 0.f, al = 1.f;   // reference max, rescale of the running sums
            bool mv = false;
            if (lane < HPG) {
                const int h = HPG * grp + lane;
                const float mt = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
                const float mu = ms.m_used[par][h];
                mv = mt > mu + kLazy || (mu == -INFINITY && mt > -INFINITY);
                mn = mv ? mt : mu;
                al = mv ? ex2_approx(mu - mt) : 1.f;   // 0 when mu = -inf
                if (quad == 0) {
                    ms.alpha[h] = al;
                    ms.m_used[par ^ 1][h] = mn;
                }
            }
            const bool moved = __any_sync(0xffffffffu, mv);
#pragma unroll
            for (int i = 0; i < HPG; ++i)
                sv[i] = ex2_approx(sv[i] - __shfl_sync(0xffffffffu, mn, i));   // 0 for a row past the end
            // P row r, heads HPG * grp ..: fp16, MN-major (heads contiguous), swizzled
            {
                if constexpr (HPG >= 8) {
#pragma unroll
                    for (int c = 0; c < HPG / 8; ++c)
                        *reinterpret_cast<uint4*>(sm + kOffP + sw128(r, (HPG * grp) / 8 + c)) =
                            make_uint4(pack_f16x2(sv[8 * c + 0], sv[8 * c + 1]), pack_f16x2(sv[8 * c + 2], sv[8 * c + 3]),
                                       pack_f16x2(sv[8 * c + 4], sv[8 * c + 5]), pack_f16x2(sv[8 * c + 6], sv[8 * c + 7]));
                } else {
                    *reinterpret_cast<uint2*>(sm + kOffP + sw128(r, (HPG * grp) >> 3) + 2 * ((HPG * grp) & 7)) =
                        make_uint2(pack_f16x2(sv[0], sv[1]), pack_f16x2(sv[2], sv[3]));
                }
            }
            {
                const float sum = sum_cols<HPG>(sv, lane);   // sv is consumed
                if ((lane & (32 / HPG - 1)) == 0) ms.red2[quad][HPG * grp + lane / (32 / HPG)] = sum;
            }
            // the previous tile's pass 2 completed before E was overwritten, so
            // O is free here: O^T[d, h] *= alpha[h] for this group's heads
            if (moved && tile > 0) {
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb) {
                    float o[HPG];
                    const uint32_t ta = tmem + lane_base + kColO + 64 * mb + HPG * grp;
                    tmem_ld<HPG>(ta, o);
                    tmem_ld_wait();
                    tmem_regs_ready_n(o);
#pragma unroll
                    for (int i = 0; i < HPG; ++i) o[i] *= __shfl_sync(0xffffffffu, al, i);
                    tmem_st<HPG>(ta, o);
                }
                tmem_st_wait();
            }
            fence_async_smem();
            tc_fence_before();
            failed = __syncthreads_or(*abort != 0);
            if (tid == 0 && !failed) {
                // ------------------------------------------------------------ pass 2 (thread 0)
                tc_fence_after();
                const uint32_t e0 = smem_u32(sm + kOffE), p0 = smem_u32(sm + kOffP);
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16kind(tmem + kColO + 64 * mb, desc_sw128(e0 + 2 * mb * kDBlockE + kk * 2048, kDBlockE, 1024),
                                    desc_sw128(p0 + kk * 2048, 8192, 1024), id2, (tile > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&ms.o_full);
            }
            if (quad == 0 && lane < HPG && !failed) {
                // this tile's running sums (the barrier above ordered every quadrant's sums);
                // read at the next tile's update or in the epilogue, after further barriers
                const int h = HPG * grp + lane;
                const float l = ms.l_run[par][h] * ms.alpha[h] +
                                ((ms.red2[0][h] + ms.red2[1][h]) + (ms.red2[2][h] + ms.red2[3][h]));
                ms.l_run[par ^ 1][h] = l;
                ms.inv_l[h] = __fdividef(1.f, l);   // used after the segment's last tile; l >= 1
            }
            ++gt;
            if (early && tile == 0) {
                // the window tile's products are issued: the selection's rows next
                dep_wait();
                seg_after_wait();   // n_tiles >= 1: the window tile is in range
            }
            if (failed) break;
        }
        if (failed) break;

        // ---------------------------------------------------------------- epilogue: all warps
        // warp w reads TMEM lanes 32 (w % 4).. of d-block w / 4, all heads in
        // chunks of 16 columns
        const int fpar = n_tiles & 1;
        const bool single = sg.slot < 0;
        const int mb = grp;
        {
            // the staged rows' largest |value|; one that is not finite fp16 is out of range
            const uint32_t hb = max(rbits & 0xffffu, rbits >> 16);
            if (hb >= 0x7c00u) amax = INFINITY;
            else ramax = fmaxf(ramax, f16_to_f32(hb));
        }
        if (!single) {
            // the partial is stored as (O / l) / sc, sc = 2^floor(log2 max |row value|),
            // so that it stays in fp16's normal range whatever the rows' magnitude
            const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(ramax));   // ramax >= 0
            if (lane == 0) ms.wmax[warp] = wm;
        }
        if (n_tiles > 0 && block_wait(&ms.o_full, (gt - 1) & 1)) {
            failed = true;
            break;
        }
        float inv_sc = 1.f, sc = 1.f;
        if (!single) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) m = max(m, ms.wmax[w]);
            const uint32_t e = m & 0x7f800000u;          // 2^floor(log2 m) for a normal m
            if (e != 0u && e != 0x7f800000u) {
                sc = __uint_as_float(e);
                inv_sc = __uint_as_float(0x7f000000u - e);   // 1 / sc, exact
            }
        }
        if (n_tiles > 0) {
            const int d = mb * 128 + quad * 32 + lane;
            // 32 heads' columns per round of TMEM loads (16 when H = 16)
            constexpr int kEpi = H >= 32 ? 32 : 16;
#pragma unroll 1
            for (int h0 = 0; h0 < H; h0 += kEpi) {
                float o[kEpi];
                tmem_ld<kEpi>(ms.tmem_base + lane_base + kColO + 64 * mb + h0, o);
                tmem_ld_wait();
                tmem_regs_ready_n(o);
#pragma unroll
                for (int c = 0; c < kEpi / 4; ++c) {
                    const float4 il = reinterpret_cast<const float4*>(&ms.inv_l[h0])[c];
                    o[4 * c + 0] *= il.x * inv_sc;
                    o[4 * c + 1] *= il.y * inv_sc;
                    o[4 * c + 2] *= il.z * inv_sc;
                    o[4 * c + 3] *= il.w * inv_sc;
                }
                if (single) {
                    float* dst = a.out + (lb * H + h0) * kKvDim + d;
#pragma unroll
                    for (int i = 0; i < kEpi; ++i) dst[(size_t)i * kKvDim] = o[i];
                } else {
                    // lanes 2k and 2k + 1 hold d and d + 1: the even lane stores both
                    // values of head i, the odd lane both of head i + 1 (4-byte stores)
                    const bool odd = lane & 1;
                    uint32_t* dst = reinterpret_cast<uint32_t*>(a.part_o + ((size_t)sg.slot * H + h0) * kKvDim +
                                                                (d & ~1));
#pragma unroll
                    for (int i = 0; i < kEpi; i += 2) {
                        const float other = __shfl_xor_sync(0xffffffffu, odd ? o[i] : o[i + 1], 1);
                        const uint32_t w = odd ? pack_f16x2(other, o[i + 1]) : pack_f16x2(o[i], other);
                        __stcg(&dst[(size_t)(i + (odd ? 1 : 0)) * (kKvDim / 2)], w);
                    }
                }
            }
        }
        if (!single && tid <= H) {
            float* pml = a.part_ml + (size_t)sg.slot * kMlStride;
            if (tid < H) {
                __stcg(&pml[tid], ms.m_used[fpar][tid]);
                __stcg(&pml[H + tid], n_tiles > 0 ? ms.l_run[fpar][tid] : 0.f);
            } else {
                __stcg(&pml[2 * H], sc);
            }
        }
        // the next segment overwrites O, S, E, P, Q and the softmax state: every
        // thread is done with this one's TMEM reads and shared values first
        tc_fence_before();
        failed = __syncthreads_or(*abort != 0);
        tc_fence_after();
        if (failed) break;
        if (!single && tid == 0) {
            // this segment's partial is written (every thread's stores precede the
            // barrier; the release makes them visible GPU-wide with the count):
            // count it, and note the share of the pair this CTA merges at the end
            const MergeItem mi = a.merges[sg.merge];
            asm volatile("red.release.gpu.global.add.u64 [%0], 1;\n" ::"l"(&a.merge_cnt[sg.merge]) : "memory");
            const int k = ms.n_duties;
            if (k < kMaxDuties) {
                ms.duty_merge[k] = sg.merge;
                ms.duty_part[k] = sg.part;
                ms.duty_target[k] = (seen / (unsigned long long)mi.ns + 1ull) * (unsigned long long)mi.ns;
                ms.n_duties = k + 1;
            } else {
                atomicOr(a.err, kErrBounds);
            }
        }
    }   // segments

    dep_wait();   // a CTA without segments, or one that stopped early
    if (q_pending) {
        // a queries' copy still lands in the E area: wait for it before leaving
        if (tid == 0 && !mbar_wait(&ms.q_full, q_uses & 1)) atomicOr(a.err, kErrTimeout);
        __syncthreads();
    }
    if (failed) {
        // the split pairs of the segments not finished: a zero-weight partial
        // each, counted, so that the other CTAs of those pairs do not wait
        for (int sj = si; sj < se; ++sj) {
            const AttnSeg sg = a.segs[sj];
            if (sg.slot < 0) continue;
            if (tid < H) __stcg(&a.part_ml[(size_t)sg.slot * kMlStride + H + tid], 0.f);
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                atomicAdd(&a.merge_cnt[sg.merge], 1ull);
            }
        }
    }

    // ---------------------------------------------------------------- range guard
    if (__any_sync(0xffffffffu, !(amax <= 65504.f)) && lane == 0) atomicOr(a.err, kErrRange);

    // ---------------------------------------------------------------- merges
    __syncthreads();
    const int n_duties = failed ? 0 : ms.n_duties;
    uint32_t m_uses = 0;   // phases of m_full
    for (int k = 0; k < n_duties; ++k) {
        const MergeItem mi = a.merges[ms.duty_merge[k]];
        const int ns = min(mi.ns, kMaxSplits);
        // this CTA's share: 8-value chunks [c0, c1) of the pair's H x 512
        // outputs, contiguous in every split's partial and in the output
        constexpr int kChunks = H * kKvDim / 8;
        const int j = ms.duty_part[k];
        const int c0 = j * kChunks / ns, c1 = (j + 1) * kChunks / ns;
        const uint32_t share = (uint32_t)(c1 - c0) * 16u;
        const uint32_t stride = (share + 127u) & ~127u;   // bytes per split in shared memory
        if (tid == 0) {
            const unsigned long long* c = &a.merge_cnt[ms.duty_merge[k]];
            const unsigned long long target = ms.duty_target[k];
            bool ok = ld_acquire_u64(c) >= target;
            if (!ok) {
                const uint64_t t0 = global_ns();
                while (!(ok = ld_acquire_u64(c) >= target)) {
                    __nanosleep(32);
                    if (global_ns() - t0 > kWaitLimitNs) break;
                }
            }
            if (ok) {
                // every split's share of the partial and the splits' statistics,
                // by bulk copies into the E area (free: no MMA reads it any more)
                asm volatile("fence.proxy.async.global;\n" ::: "memory");
                fence_async_smem();
                const uint32_t ml_bytes = (uint32_t)ns * kMlStride * 4u;
                mbar_arrive_expect_tx(&ms.m_full, (uint32_t)ns * share + ml_bytes);
                for (int sp = 0; sp < ns; ++sp)
                    bulk_g2s(sm + kOffE + sp * stride,
                             a.part_o + ((size_t)(mi.first + sp) * H * kKvDim + (size_t)c0 * 8), share, &ms.m_full);
                bulk_g2s(sm + kOffE + kMergeMlOff, a.part_ml + (size_t)mi.first * kMlStride, ml_bytes, &ms.m_full);
            } else {
                atomicOr(a.err, kErrTimeout);
                ms.abort = 1;
            }
        }
        if (__syncthreads_or(*abort != 0)) break;
        if (block_wait(&ms.m_full, m_uses & 1)) break;
        ++m_uses;
        // each head's weights over the splits, once:
        //   w_s = l_s 2^(m_s - M) sc_s / sum_s' l_s' 2^(m_s' - M),  M = max m_s over splits with rows
        const float* mls = reinterpret_cast<const float*>(sm + kOffE + kMergeMlOff);
        float* wts = reinterpret_cast<float*>(sm + kOffE + kMergeWOff);
        // eight lanes per head, each taking splits j, j + 8, ...: maximum and
        // sum over the splits by shuffles within the eight lanes
        {
            const int h = tid >> 3, j = tid & 7;
            const bool hv = h < H;
            float M = -INFINITY;
            for (int sp = j; hv && sp < ns; sp += 8)
                if (mls[sp * kMlStride + H + h] > 0.f) M = fmaxf(M, mls[sp * kMlStride + h]);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float L = 0.f;
            for (int sp = j; hv && sp < ns; sp += 8) {
                const float l = mls[sp * kMlStride + H + h];
                const float wl = l > 0.f ? l * ex2_approx(mls[sp * kMlStride + h] - M) : 0.f;
                wts[sp * 64 + h] = wl;
                L += wl;
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            // 2^112 undoes the exponent offset of the fp16 bits read as fp32 below
            const float inv = L > 0.f ? 0x1p112f / L : 0.f;
            for (int sp = j; hv && sp < ns; sp += 8) wts[sp * 64 + h] *= mls[sp * kMlStride + 2 * H] * inv;
        }
        __syncthreads();
        // every thread combines its chunks over the splits, in split order; a
        // split without rows (weight 0) is skipped: its partial was not written
        for (int c = c0 + tid; c < c1; c += kThreads) {
            const int h = c >> 6;
            const unsigned char* pv = sm + kOffE + (size_t)(c - c0) * 16;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 4
            for (int sp = 0; sp < ns; ++sp) {
                const float w = wts[sp * 64 + h];
                if (w != 0.f) {
                    const uint4 v = *reinterpret_cast<const uint4*>(pv + (size_t)sp * stride);
                    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] = fmaf(w, f16_bits_scaled(x[e]), acc[2 * e]);
                        acc[2 * e + 1] = fmaf(w, f16_bits_scaled(x[e] >> 16), acc[2 * e + 1]);
                    }
                }
            }
            float4* dst = reinterpret_cast<float4*>(a.out + (size_t)mi.lb * H * kKvDim + (size_t)c * 8);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        __syncthreads();   // the E area is read before the next merge's copies land
    }

    // ---------------------------------------------------------------- teardown
    if (tid == 0 && gt > 0) {
        // completes once every MMA issued above has completed
        mma_commit(&ms.drain);
        if (!mbar_wait(&ms.drain, 0)) atomicOr(a.err, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(ms.tmem_base, kTmemCols);
    }
}

template <int H>
cudaError_t launch_h(const AttnArgs& args, int n_ctas, cudaStream_t st, bool chained) {
    return launch_k(attend_kernel<H>, dim3(n_ctas), dim3(kThreads), kSmemBytes, st, chained, args);
}

}  // namespace

int attend_max_splits() { return kMaxSplits; }
int attend_max_duties() { return kMaxDuties; }

cudaError_t set_attend_attrs() {
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attend_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attend_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    return e;
}

cudaError_t launch_attend(const AttnSeg* segs, const int* cta_begin, int n_ctas, const MergeItem* merges,
                          unsigned long long* merge_cnt, int n_heads, int B, int G, int S, const uint16_t* q,
                          const float* window, const uint16_t* staging, const int32_t* phys, const int32_t* count_l,
                          float* out, uint16_t* part_o, float* part_ml, uint32_t* err, cudaStream_t st,
                          bool chained) {
    if (n_ctas <= 0) return cudaSuccess;
    AttnArgs args{segs, cta_begin, merges, merge_cnt, B, G, S, q, window, staging, phys, count_l,
                  out, part_o, part_ml, err, (float)(1.4426950408889634 / std::sqrt((double)kKvDim))};
    switch (n_heads) {
        case 16: return launch_h<16>(args, n_ctas, st, chained);
        case 32: return launch_h<32>(args, n_ctas, st, chained);
        case 64: return launch_h<64>(args, n_ctas, st, chained);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace srh
