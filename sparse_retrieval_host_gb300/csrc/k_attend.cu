// K-attend + K-merge: split-K flash-decode on the 5th-generation tensor cores.
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
// one wave, otherwise a contiguous range of the whole call's tiles. A CTA runs
// its segments for all heads, tile by tile. Each row is read from HBM once per
// step; a tile's rows are requested into L2 with bulk prefetches before the
// loads below:
//   load    all 8 warps stream the tile's fp32 rows (warp w: rows 16w..16w+15,
//           whole 2 KiB rows, 512 contiguous bytes per load instruction) into
//           registers, convert to fp16 and store them into one resident
//           128B-swizzled tile E [128 rows x 512 d] (8 d-blocks of 64);
//   pass 1  S^T[r, h] = E[r, :] . Q[h, :]   (M = 128 rows, N = heads, K = 512),
//           E and Q K-major;
//   softmax (warps 0-3, one TMEM lane = one row): base-2 online softmax with a
//           lazily moved reference max per head (moved only when the tile max
//           exceeds it by 2^8), warp butterfly transpose-reductions for the
//           per-head max and sum; P written as fp16 [rows x heads];
//   pass 2  O^T[d, h] += E^T[d, r] P[r, h]   (M = 128 d, N = heads, K = rows),
//           the SAME smem tile read MN-major (a 128B-swizzled atom of 8 rows x
//           64 d serves both views), so no row is fetched twice.
// Both products are tcgen05 kind::f16 MMAs with fp32 accumulation in TMEM,
// issued by thread 0. fp16 keeps 11 significant bits, as tf32 does; 32-bit
// operands cannot be MN-major, which pass 2 needs. The latents are O(1),
// p <= 2^8 by construction, and bf16 queries of normal fp16 range convert
// exactly.
//
// With more than one tile in a segment, warps 4-7 issue the loads of the next
// tile while warps 0-3 run the softmax; every warp waits for the previous
// tile's pass 2 before it overwrites E. Every wait is bounded; on a timeout
// the CTA records kErrTimeout, drains its MMAs, frees TMEM and returns.
//
// A pair spread over several segments writes (m, l, O) partials per segment;
// a second kernel merges them in row order. The plan depends only on the
// configuration, so identical rows give identical bits whatever slots hold
// them.
#include <cmath>

#include "srh_internal.cuh"
#include "umma.cuh"

namespace srh {
namespace {

using namespace umma;

constexpr int kTileRows = kAttnTile;                // 128
constexpr int kThreads = 256;                       // 8 warps
constexpr int kSoftThreads = 128;                   // warps 0-3: softmax, TMEM lanes 0-127
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

struct Misc {
    uint64_t s_full, o_full, drain;
    uint32_t tmem_base;
    int abort;
    int rescale;
    int epi_ok;
    float m_used[64];
    float l_run[64];
    float alpha[64];        // per-tile rescale factors; 1 / l after the last tile
    float red[4][64];
};
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
    int B, G, S;
    const uint16_t* q;
    const float* window;
    const float* staging;
    const int32_t* phys;
    const int32_t* count_l;
    float* out;
    float* part_o;
    float* part_ml;
    uint32_t* err;
    float sl2;   // log2(e) / sqrt(kv_dim)
};

// Bounded wait that also gives up when another thread has aborted the CTA.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              uint32_t* err) {
    const int r = mbar_wait_abort(bar, parity, abort);
    if (r < 0) atomicOr(err, kErrTimeout);
    return r > 0;
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so a
// failed wait in any of them makes all of them leave together.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n"
        " setp.ne.u32 pi, %1, 0;\n"
        " bar.red.or.pred po, %2, %3, pi;\n"
        " selp.u32 %0, 1, 0, po;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Read-only streaming load of 16 bytes (no L1 allocation).
__device__ __forceinline__ float4 ldg_stream(const float4* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// Max / sum over the 32 lanes of a warp for 32 per-lane values at once: after
// the call, lane l holds the reduction of column l. Each step hands half of
// the columns to the partner lane, so 31 shuffles do all 32 reductions.
template <bool kMax>
__device__ __forceinline__ float butterfly32(float (&v)[32], int lane) {
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int bit = 16 >> step;
        const int half = 16 >> step;
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, bit);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const __grid_constant__ AttnArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Misc& ms = *reinterpret_cast<Misc*>(sm + kOffMisc);
    volatile int* abort = &ms.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // this CTA's segments of the static plan (written once, at creation)
    const int sb = a.cta_begin[blockIdx.x], se = a.cta_begin[blockIdx.x + 1];
    pdl_trigger();

    // ---------------------------------------------------------------- set-up
    // Everything up to the dependency wait reads only this call's inputs (the
    // queries), so with chained launches it overlaps the kernels that resolve
    // and gather the staged rows.
    if (tid == 0) {
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.o_full, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        ms.rescale = 0;
        ms.epi_ok = 0;
        fence_mbar_init();
    }
    if (tid < 64) {
        ms.m_used[tid] = -INFINITY;
        ms.l_run[tid] = 0.f;
        ms.alpha[tid] = 1.f;
    }
    if (warp == 0) tmem_alloc(&ms.tmem_base, kTmemCols);
    // queries of (layer, sequence) lb: bf16 [H][512] -> fp16 K-major; d-block d / 64
    // at (d / 64) * 8192, row h
    constexpr int kQPer = H * 64 / kThreads;             // 16-byte chunks per thread
    auto load_q = [&](int lbq, uint4 (&qv)[kQPer]) {
        const uint16_t* qg = a.q + (size_t)lbq * H * kKvDim;
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int i = tid + k * kThreads;
            qv[k] = *reinterpret_cast<const uint4*>(qg + (i >> 6) * kKvDim + (i & 63) * 8);
        }
    };
    auto store_q = [&](const uint4 (&qv)[kQPer]) {
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int i = tid + k * kThreads, h = i >> 6, c8 = i & 63;
            const uint4 v = qv[k];
            uint4 w;
            w.x = pack_f16x2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
            w.y = pack_f16x2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
            w.z = pack_f16x2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
            w.w = pack_f16x2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
            *reinterpret_cast<uint4*>(sm + kOffQ + (c8 >> 3) * 8192 + sw128(h, c8 & 7)) = w;
        }
    };
    auto convert_q = [&](int lbq) {
        uint4 qv[kQPer];
        load_q(lbq, qv);
        store_q(qv);
    };
    int q_lb = sb < se ? a.segs[sb].lb : 0;
    // The window rows are this call's own input: the first segment's (when it
    // starts at tile 0) are requested from HBM before the dependency wait.
    if (sb < se && a.segs[sb].tile0 == 0 && tid < kWindow)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(a.window + ((size_t)q_lb * kWindow + tid) * kKvDim),
                     "r"(kKvDim * 4) : "memory");
    // The first pair's queries are loaded after the dependency wait (below);
    // L2 is asked for them now.
    constexpr int kQChunk = 16384;
    if (sb < se && tid < H * kKvDim * 2 / kQChunk)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(
                         reinterpret_cast<const unsigned char*>(a.q + (size_t)q_lb * H * kKvDim) + tid * kQChunk),
                     "r"(kQChunk) : "memory");
    // the barriers, the abort flag, the softmax state and the TMEM address are
    // set: every thread sees them from here on
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ... as fp16 into E: d-block (lane >> 4) + 2 j, 16-byte chunk (lane & 15) >> 1, half lane & 1.
    auto store4 = [&](const float4 (&v)[4][4], int rbase) {
        unsigned char* e = sm + kOffE + (lane >> 4) * kDBlockE + 8 * (lane & 1);
        const int chunk = (lane & 15) >> 1;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint2*>(e + 2 * j * kDBlockE + sw128(rbase + i, chunk)) =
                    make_uint2(pack_f16x2(v[i][j].x, v[i][j].y), pack_f16x2(v[i][j].z, v[i][j].w));
    };

    constexpr uint32_t id1 = idesc_f16(0, 0, H);   // pass 1: K-major E and Q
    constexpr uint32_t id2 = idesc_f16(1, 1, H);   // pass 2: MN-major E^T and P
    const int rw = 16 * warp;                       // this warp's first tile row
    bool ok = true;

    pdl_wait();   // slots, counts and staged rows come from earlier kernels

    // The first segment's row count and first-tile slots, then its queries:
    // all in flight together (one round trip for a CTA that starts once the
    // earlier kernels are done, as most do: an attention CTA needs a whole SM).
    int pre_cnt = 0, pre_ph0 = -1;
    if (sb < se) {
        const AttnSeg s0 = a.segs[sb];
        const int rr = s0.tile0 * kTileRows + tid - kWindow;
        if (tid < kTileRows && rr >= 0 && rr < a.S) pre_ph0 = a.phys[(size_t)s0.lb * a.S + rr];
        pre_cnt = a.count_l[s0.lb];
        convert_q(q_lb);   // read by pass 1 after the tile loop's barrier
    }

    uint32_t gt0 = 0;     // tiles this CTA ran before the current segment (mbarrier phases)
    uint32_t n_drain = 0; // drains this CTA ran (phases of ms.drain)
    for (int si = sb; si < se && !*abort; ++si) {
    const AttnSeg sg = a.segs[si];
    const size_t lb = (size_t)sg.lb;
    if (si > sb) {
        // a new segment: the previous one drained its MMAs and wrote its
        // epilogue; reset the running softmax and, for a new pair, load its queries
        if (sg.lb != q_lb) {
            convert_q(sg.lb);
            q_lb = sg.lb;
        }
        if (tid < 64) {
            ms.m_used[tid] = -INFINITY;
            ms.l_run[tid] = 0.f;
            ms.alpha[tid] = 1.f;
        }
        if (tid == 0) ms.rescale = 0;
        __syncthreads();
    }
    const int32_t* ph = a.phys + lb * a.S;
    // the slot of this thread's row of the first tile, loaded beside the count
    // (a slot past the count is never used); the first segment's were loaded
    // after the dependency wait, beside its queries
    int ph0 = pre_ph0, cnt = pre_cnt;
    if (si > sb) {
        ph0 = -1;
        const int rr = sg.tile0 * kTileRows + tid - kWindow;
        if (tid < kTileRows && rr >= 0 && rr < a.S) ph0 = ph[rr];
        cnt = a.count_l[lb];
    }
    if (cnt < 0 || cnt > a.S) {
        if (tid == 0) atomicOr(a.err, kErrBounds);
        cnt = cnt < 0 ? 0 : a.S;
    }
    const int R = kWindow + cnt;
    const int row0 = sg.tile0 * kTileRows;
    const int row1 = min(R, sg.tile1 * kTileRows);
    const int n_tiles = row1 > row0 ? (row1 - row0 + kTileRows - 1) / kTileRows : 0;

    // Source of tile row tr: window rows first, then the staged rows in list
    // order; rows past the split end repeat its last row (finite data that the
    // softmax masks).
    auto row_src = [&](int tr0, int tr) -> const float4* {
        const int row = min(tr0 + tr, row1 - 1);
        if (row < kWindow) return reinterpret_cast<const float4*>(a.window + (lb * kWindow + row) * kKvDim);
        int slot = ph[row - kWindow] - kWindow;
        if (slot < 0 || slot >= a.G) {
            atomicOr(a.err, kErrBounds);
            slot = 0;
        }
        return reinterpret_cast<const float4*>(a.staging + (lb * (size_t)a.G + slot) * kKvDim);
    };
    // Ask L2 for the rows of the tile at tr0: one 2 KiB bulk prefetch per row,
    // issued by threads 0-127. It holds no registers or shared memory, so the
    // whole tile is requested from HBM at once and the loads below find it in L2.
    // `first`: the segment's first tile, whose slots are already in ph0.
    auto prefetch_tile = [&](int tr0, bool first) {
        const int row = tr0 + tid;
        if (tid >= kTileRows || row >= row1) return;
        if (si == sb && row < kWindow) return;             // requested before the wait
        const float* p;
        if (row < kWindow) {
            p = a.window + (lb * kWindow + row) * kKvDim;
        } else {
            const int slot = (first ? ph0 : ph[row - kWindow]) - kWindow;
            if (slot < 0 || slot >= a.G) return;            // reported by the loads
            p = a.staging + (lb * (size_t)a.G + slot) * kKvDim;
        }
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(kKvDim * 4) : "memory");
    };
    // Four rows of this warp: lane holds float4 lane + 32 j of each (d = 4 (lane + 32 j)).
    auto load4 = [&](float4 (&v)[4][4], int tr0, int rbase) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4* src = row_src(tr0, rbase + i);
#pragma unroll
            for (int j = 0; j < 4; ++j) v[i][j] = ldg_stream(src + lane + 32 * j);
        }
    };

    if (n_tiles > 0) prefetch_tile(row0, true);
    for (int tile = 0; tile < n_tiles; ++tile) {
        // ------------------------------------------------------------ load E (all warps)
        const int tr0 = row0 + tile * kTileRows;
        if (tile + 1 < n_tiles) prefetch_tile(tr0 + kTileRows, false);   // the next tile's rows, during this one
        float4 b0[4][4], b1[4][4];
        if (ok) {
            load4(b0, tr0, rw);
            load4(b1, tr0, rw + 4);
            // the previous tile's pass 2 reads E: wait for it before overwriting
            if (tile > 0 && !wait_or_abort(&ms.o_full, (gt0 + tile - 1) & 1, abort, a.err)) ok = false;
        }
        if (ok) {
            store4(b0, rw);
            load4(b0, tr0, rw + 8);
            store4(b1, rw + 4);
            load4(b1, tr0, rw + 12);
            store4(b0, rw + 8);
            store4(b1, rw + 12);
        }
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t tmem = ms.tmem_base;

        // ------------------------------------------------------------ pass 1 (thread 0)
        if (tid == 0) {
            const uint32_t e0 = smem_u32(sm + kOffE), q0 = smem_u32(sm + kOffQ);
#pragma unroll 1
            for (int x = 0; x < 8; ++x)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16kind(tmem + kColS, desc_sw128(e0 + x * kDBlockE + kk * 32, 16, 1024),
                                desc_sw128(q0 + x * 8192 + kk * 32, 16, 1024), id1, (x | kk) != 0);
            mma_commit(&ms.s_full);
        }
        if (tid >= kSoftThreads) continue;   // warps 4-7: on to the next tile's loads

        // ------------------------------------------------------------ softmax (warps 0-3)
        const int r = tid;                                // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const bool got = wait_or_abort(&ms.s_full, (gt0 + tile) & 1, abort, a.err);
        if (named_sync_or(1, kSoftThreads, !got)) {
            ok = false;
            *abort = 1;
            continue;                                     // leaves at the next block barrier
        }
        tc_fence_after();
        float v[64];
#pragma unroll
        for (int c = 0; c < H; c += 16) {
            float t16[16];
            tmem_ld16(tmem + lane_base + kColS + c, t16);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[c + i] = t16[i];
        }
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < H; c += 16) tmem_regs_ready(v + c);
        const bool valid = tr0 + r < row1;
#pragma unroll
        for (int h = 0; h < 64; ++h) v[h] = (h < H && valid) ? v[h] * a.sl2 : -INFINITY;
        // per-head tile max over the 128 rows: warp butterflies, then the 4 warps
#pragma unroll
        for (int hh = 0; hh < H; hh += 32) {
            float red[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) red[i] = hh + i < H ? v[hh + i] : -INFINITY;
            ms.red[warp][hh + lane] = butterfly32<true>(red, lane);
        }
        named_sync(1, kSoftThreads);
        if (tid < H) {
            const int h = tid;
            const float mt = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
            const float mu = ms.m_used[h];
            float al = 1.f;
            if (mt > mu + kLazy || (mu == -INFINITY && mt > -INFINITY)) {
                al = exp2f(mu - mt);                      // 0 when mu = -inf
                ms.m_used[h] = mt;
                ms.l_run[h] *= al;
                if (tile > 0 && al != 1.f) ms.rescale = 1;
            }
            ms.alpha[h] = al;
        }
        named_sync(1, kSoftThreads);
#pragma unroll
        for (int h = 0; h < 64; ++h) v[h] = (h < H) ? exp2f(v[h] - ms.m_used[h]) : 0.f;
#pragma unroll
        for (int hh = 0; hh < H; hh += 32) {
            float red[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) red[i] = v[hh + i];
            ms.red[warp][hh + lane] = butterfly32<false>(red, lane);
        }
        named_sync(1, kSoftThreads);
        if (tid < H) ms.l_run[tid] += (ms.red[0][tid] + ms.red[1][tid]) + (ms.red[2][tid] + ms.red[3][tid]);
        // pass 2 of the previous tile completed before E was overwritten, so O
        // and P are free here
        if (ms.rescale) {
            // O^T[d, h] *= alpha[h]: this thread owns TMEM lane r of each d-block
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
                for (int c = 0; c < H; c += 16) {
                    float t16[16];
                    const uint32_t ta = tmem + lane_base + kColO + 64 * mb + c;
                    tmem_ld16(ta, t16);
                    tmem_ld_wait();
                    tmem_regs_ready(t16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) t16[i] *= ms.alpha[c + i];
                    tmem_st16(ta, t16);
                }
            }
            tmem_st_wait();
        }
        // P row r: 64 fp16 heads = 128 B, MN-major (heads contiguous), swizzled
        unsigned char* prow = sm + kOffP;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 w;
            w.x = pack_f16x2(v[8 * c + 0], v[8 * c + 1]);
            w.y = pack_f16x2(v[8 * c + 2], v[8 * c + 3]);
            w.z = pack_f16x2(v[8 * c + 4], v[8 * c + 5]);
            w.w = pack_f16x2(v[8 * c + 6], v[8 * c + 7]);
            *reinterpret_cast<uint4*>(prow + sw128(r, c)) = w;
        }
        fence_async_smem();
        tc_fence_before();
        named_sync(1, kSoftThreads);
        if (tid == 0) {
            // ------------------------------------------------------------ pass 2 (thread 0)
            ms.rescale = 0;
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
    }

    // ---------------------------------------------------------------- drain
    if (tid == 0 && n_tiles > 0) {
        // completes once every MMA issued above has completed
        mma_commit(&ms.drain);
        if (!mbar_wait(&ms.drain, n_drain & 1)) {
            atomicOr(a.err, kErrTimeout);
            ok = false;
        }
    }
    if (n_tiles > 0) ++n_drain;
    gt0 += (uint32_t)n_tiles;
    tc_fence_before();
    const bool failed = __syncthreads_or(!ok);
    tc_fence_after();
    if (tid < H) ms.alpha[tid] = 1.f / ms.l_run[tid];
    if (tid == 0) ms.epi_ok = failed ? 0 : 1;
    __syncthreads();

    // ---------------------------------------------------------------- epilogue: all 8 warps
    const bool single = sg.slot < 0;
    float* dst = single ? a.out + lb * H * kKvDim : a.part_o + (size_t)sg.slot * H * kKvDim;
    if (n_tiles > 0 && ms.epi_ok) {
        const uint32_t tmem = ms.tmem_base;
        // warp w reads TMEM lanes 32 (w & 3).. of d-blocks 2 (w >> 2) and 2 (w >> 2) + 1
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
        for (int mm = 0; mm < 2; ++mm) {
            const int mb = 2 * (warp >> 2) + mm;
            const int d = mb * 128 + (warp & 3) * 32 + lane;
            // all H columns of this d-block in one TMEM round trip
            float t[H];
#pragma unroll
            for (int c = 0; c < H; c += 16) tmem_ld16(tmem + lane_base + kColO + 64 * mb + c, *reinterpret_cast<float(*)[16]>(t + c));
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < H; c += 16) tmem_regs_ready(t + c);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                if (single) dst[h * kKvDim + d] = t[h] * ms.alpha[h];
                else __stcg(&dst[h * kKvDim + d], t[h]);
            }
        }
    } else if (!single) {
        for (int i = tid; i < H * kKvDim; i += kThreads) __stcg(&dst[i], 0.f);
    }
    if (!single && tid < H) {
        float* pml = a.part_ml + (size_t)sg.slot * 2 * H;
        __stcg(&pml[tid], ms.m_used[tid]);
        __stcg(&pml[H + tid], n_tiles > 0 && ms.epi_ok ? ms.l_run[tid] : 0.f);
    }
    // the next segment overwrites O, S, E, P and the softmax state: every
    // thread is done with this one's TMEM reads and shared values first
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!ms.epi_ok && n_tiles > 0) *abort = 1;
    }   // segments

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(ms.tmem_base, kTmemCols);
    }
}

// Merge the split partials of one (layer, sequence), one head per CTA (thread
// i owns float4 i of the head's 512 values):
//     o_h = sum_s w_s O_s[h] / sum_s w_s l_s,   w_s = 2^(m_s - max_s m_s),
// over the splits with l_s > 0, in split order. A split with l_s = 0 (no rows,
// or a failed CTA) wrote zeros and gets weight 0. Every thread loads the
// splits' statistics itself, together with its values of the first splits, so
// the merge costs one round of loads and no barrier.
// L2 loads of data an earlier kernel wrote: volatile with a memory clobber, so
// the compiler keeps them after pdl_wait().
__device__ __forceinline__ float ld_dep(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];\n" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_dep4(const float4* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

template <int H>
__global__ void __launch_bounds__(kKvDim / 4) merge_kernel(const MergeItem* __restrict__ merges, int merge0,
                                                           const float* part_o, const float* part_ml,
                                                           float* __restrict__ out) {
    constexpr int kFirst = 5;   // splits loaded in the first round (a 640-row pair has 5)
    const MergeItem mi = merges[merge0 + blockIdx.x];   // the plan: written once, at creation
    const int h = blockIdx.y;
    const int ns = min(mi.ns, kMaxSplits);
    const int t = threadIdx.x;
    const float* ml = part_ml + (size_t)mi.first * 2 * H;
    const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)mi.first * H + h) * kKvDim) + t;
    const size_t split_stride = (size_t)H * kKvDim / 4;   // float4s between consecutive splits
    pdl_wait();   // the partials come from the attention kernel
    float4 v[kFirst];
    float mv[kFirst], lv[kFirst];
#pragma unroll
    for (int j = 0; j < kFirst; ++j) {
        if (j < ns) {
            v[j] = ld_dep4(src + (size_t)j * split_stride);
            mv[j] = ld_dep(&ml[(size_t)j * 2 * H + h]);
            lv[j] = ld_dep(&ml[(size_t)j * 2 * H + H + h]);
        }
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kFirst; ++j)
        if (j < ns && lv[j] > 0.f) M = fmaxf(M, mv[j]);
    for (int s = kFirst; s < ns; ++s) {
        const float ls = ld_dep(&ml[(size_t)s * 2 * H + H + h]);
        if (ls > 0.f) M = fmaxf(M, ld_dep(&ml[(size_t)s * 2 * H + h]));
    }
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kFirst; ++j) {
        if (j < ns) {
            mv[j] = lv[j] > 0.f ? exp2f(mv[j] - M) : 0.f;   // the weight w_j
            L += mv[j] * lv[j];
        }
    }
    for (int s = kFirst; s < ns; ++s) {
        const float ls = ld_dep(&ml[(size_t)s * 2 * H + H + h]);
        const float w = ls > 0.f ? exp2f(ld_dep(&ml[(size_t)s * 2 * H + h]) - M) : 0.f;
        L += w * ls;
    }
    const float inv = 1.f / L;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kFirst; ++j) {
        if (j < ns) {
            const float w = mv[j] * inv;
            acc.x += w * v[j].x;
            acc.y += w * v[j].y;
            acc.z += w * v[j].z;
            acc.w += w * v[j].w;
        }
    }
    for (int s = kFirst; s < ns; ++s) {
        const float ls = ld_dep(&ml[(size_t)s * 2 * H + H + h]);
        const float w = (ls > 0.f ? exp2f(ld_dep(&ml[(size_t)s * 2 * H + h]) - M) : 0.f) * inv;
        const float4 x = ld_dep4(src + (size_t)s * split_stride);
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
    }
    reinterpret_cast<float4*>(out + ((size_t)mi.lb * H + h) * kKvDim)[t] = acc;
}

template <int H>
cudaError_t launch_h(const AttnArgs& args, int n_ctas, const MergeItem* merges, int n_merges,
                     cudaStream_t st, bool chained) {
    cudaError_t e = launch_k(attend_tc_kernel<H>, dim3(n_ctas), dim3(kThreads), kSmemBytes, st, chained, args);
    if (e != cudaSuccess || n_merges <= 0) return e;
    // the merge follows its own attention kernel: always chained
    return launch_k(merge_kernel<H>, dim3((unsigned)n_merges, H), dim3(kKvDim / 4), 0, st, true, merges, 0,
                    (const float*)args.part_o, (const float*)args.part_ml, args.out);
}

}  // namespace

int attend_max_splits() { return kMaxSplits; }

cudaError_t set_attend_attrs() {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attend_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attend_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    return e;
}

cudaError_t launch_attend(const AttnSeg* segs, const int* cta_begin, int n_ctas, const MergeItem* merges,
                          int n_merges, int n_heads, int B, int G, int S, const uint16_t* q, const float* window,
                          const float* staging, const int32_t* phys, const int32_t* count_l, float* out,
                          float* part_o, float* part_ml, uint32_t* err, cudaStream_t st, bool chained) {
    if (n_ctas <= 0) return cudaSuccess;
    AttnArgs args{segs, cta_begin, B, G, S, q, window, staging, phys, count_l,
                  out, part_o, part_ml, err, (float)(1.4426950408889634 / std::sqrt((double)kKvDim))};
    switch (n_heads) {
        case 16: return launch_h<16>(args, n_ctas, merges, n_merges, st, chained);
        case 32: return launch_h<32>(args, n_ctas, merges, n_merges, st, chained);
        case 64: return launch_h<64>(args, n_ctas, merges, n_merges, st, chained);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace srh
