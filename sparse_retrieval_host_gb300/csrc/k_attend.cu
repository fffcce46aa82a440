// K-attend + K-combine: split-K flash-decode on the 5th-generation tensor cores.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 技术细节 / 架构概览,
// per-layer box step 3 (indexed_cached_attention over window + selected rows)
// and "Memory Layout" (window KV [128, kv_dim] plus staging slots [gpu_chunks,
// kv_dim], one fp32 latent row per entry). Every head attends over the same
// rows (MQA over the latent, K = V = row):
//     o_h = sum_j softmax_j(<q_h, e_j> / sqrt(512)) e_j.
//
// Work: the rows of one (layer, sequence) -- the 128 window rows, then the
// layer's staged rows in selection order -- are cut into fixed splits of
// `split_rows` (a multiple of 128); one CTA runs one split for all heads, in
// tiles of 128 rows. Per tile:
//   pass 1  S^T[r, h] = E[r, :] . Q[h, :]   (M = 128 rows, N = heads, K = 512)
//           over 8 pieces [128 rows x 64 d];
//   softmax (4 warps, one TMEM lane = one row): base-2 online softmax with a
//           lazily moved reference max per head (moved only when the tile max
//           exceeds it by 2^8), warp butterfly transpose-reductions for the
//           per-head max and sum; P written as fp16 [rows x heads];
//   pass 2  O^T[d, h] += E^T[d, r] P[r, h]   (M = 128 d, N = heads, K = rows)
//           over 8 pieces [64 rows x 128 d]; the tile's rows are read a second
//           time, from L2.
// Both products run as tcgen05 kind::f16 MMAs with fp32 accumulation in TMEM.
// The fp32 rows are gathered by bulk copies into a landing ring, then
// converted to fp16 into a 128B-swizzled operand ring (K-major for pass 1,
// MN-major for pass 2: 32-bit operands must be K-major, and pass 2 contracts
// over rows). fp16 keeps 11 significant bits, as tf32 does; the latents are
// O(1), p <= 2^8 by construction, and bf16 queries of normal fp16 range
// convert exactly.
//
// Roles: warps 4-7 only issue the gathers: one 256-byte bulk copy (TMA) per
// thread and piece, counted on the piece's mbarrier as transaction bytes, so
// they never wait on their own copies. Warps 0-3 convert landed pieces, run the softmax (TMEM lanes
// 0-127) and write the output with warps 4-7; they issue no copies, so the
// proxy fence that publishes each converted piece to the tensor core stays
// cheap. Warp 0 allocates TMEM and its lane 0 issues the MMAs, each piece as
// soon as all four converter warps have published it. Every wait is bounded;
// on a timeout the CTA records kErrTimeout, drains its copies and MMAs, frees
// TMEM and returns.
//
// A split writes (m, l, O) partials; the last CTA of a (layer, sequence) to
// finish (an atomic ticket, no waiting) merges them in split order. The split
// layout depends only on the row count, so identical rows give identical bits
// whatever slots hold them.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "srh_internal.cuh"
#include "umma.cuh"

namespace srh {
namespace {

using namespace umma;

constexpr int kTileRows = kAttnTile;    // 128
constexpr int kSoftWarps = 4;
constexpr int kLoadWarps = 4;
constexpr int kThreads = (kSoftWarps + kLoadWarps) * 32;   // 256: two warps per SM sub-partition
constexpr int kLoads = 16;                                  // landing loads per tile (8 per pass)
constexpr int kNLand = 3;                                   // fp32 landing slots
constexpr int kNOp = 3;                                     // fp16 operand slots (shared with the MMA)
constexpr int kLand = 32768;                                // [128 rows x 64 d] or [64 rows x 128 d] fp32
constexpr int kOp = 16384;                                  // the same piece in fp16
constexpr int kOffQ = 0;                                    // 8 K-blocks [64 heads x 64 d] fp16
constexpr int kOffLand = kOffQ + 8 * 8192;
constexpr int kOffOp = kOffLand + kNLand * kLand;
constexpr int kOffP = kOffOp + kNOp * kOp;                  // fp16 [128 rows x 64 heads]
constexpr int kOffMisc = kOffP + kTileRows * 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                               // S^T: 64 columns
constexpr uint32_t kColO = 64;                              // O^T[mb]: 64 columns each
constexpr float kLazy = 8.0f;                               // reference max moves past 2^8 growth
constexpr int kMaxSplits = (kWindow + kMaxSelect + kTileRows - 1) / kTileRows;

struct Misc {
    uint64_t lfull[kNLand];
    uint64_t lempty[kNLand];
    uint64_t opfull[kNOp];
    uint64_t opempty[kNOp];
    uint64_t s_full, p_full, o_full, drain;
    uint32_t tmem_base;
    uint32_t ticket;
    int abort;
    int rescale;
    int epi_ok;
    float m_used[64];
    float l_run[64];
    float alpha[64];        // per-tile rescale factors; 1 / l after the last tile
    float red[kSoftWarps][64];
};
constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc) + 1024;   // + base alignment slack
static_assert(kSmemBytes <= 232448, "attention shared memory exceeds 227 KB");

// f16-kind instruction descriptor: f16 A and B, f32 accumulate, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(int a_mn, int b_mn, int n) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

// Gather maps: window [L*B*128 rows][512] and staging [L*B*G rows][512] fp32,
// each with a 64- and a 128-column box one row high.
struct AttnMaps {
    CUtensorMap win64, win128, stg64, stg128;
};

struct AttnArgs {
    const AttnItem* items;
    int item0;
    int split_rows;
    int B, G, S;
    const uint16_t* q;
    const float* window;
    const float* staging;
    const int32_t* phys;
    const int32_t* count_l;
    float* out;
    float* part_o;
    float* part_ml;
    unsigned* counters;
    uint32_t* err;
    float sl2;   // log2(e) / sqrt(kv_dim)
};

// Bounded wait that also gives up when another role has aborted the CTA.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              uint32_t* err) {
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && *abort) return false;
    }
    *abort = 1;
    atomicOr(err, kErrTimeout);
    return false;
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
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const __grid_constant__ AttnArgs a,
                                                                 const __grid_constant__ AttnMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Misc& ms = *reinterpret_cast<Misc*>(sm + kOffMisc);
    volatile int* abort = &ms.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int item_idx = a.item0 + blockIdx.x;
    const AttnItem it = a.items[item_idx];
    const size_t lb = (size_t)it.layer * a.B + it.seq;
    int cnt = a.count_l[lb];
    if (cnt < 0 || cnt > a.S) {
        if (tid == 0) atomicOr(a.err, kErrBounds);
        cnt = cnt < 0 ? 0 : a.S;
    }
    const int R = kWindow + cnt;
    const int row0 = it.split * a.split_rows;
    const int row1 = min(R, row0 + a.split_rows);
    const int n_tiles = row1 > row0 ? (row1 - row0 + kTileRows - 1) / kTileRows : 0;
    const int32_t* ph = a.phys + lb * a.S;

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int s = 0; s < kNLand; ++s) {
            mbar_init(&ms.lfull[s], 1);
            mbar_init(&ms.lempty[s], kSoftWarps * 32);
        }
        for (int s = 0; s < kNOp; ++s) {
            mbar_init(&ms.opfull[s], kSoftWarps * 32);
            mbar_init(&ms.opempty[s], 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.p_full, kSoftWarps * 32);
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
    if (warp == 0 && n_tiles > 0) tmem_alloc(&ms.tmem_base, kTmemCols);
    if (n_tiles > 0) {
        // queries: bf16 [H][512] -> fp16 K-major; K-block d / 64 at (d / 64) * 8192, row h.
        // All loads first, then the conversions.
        constexpr int kPer = H * 64 / kThreads;          // 16-byte chunks per thread
        const uint16_t* qg = a.q + lb * H * kKvDim;
        uint4 qv[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + k * kThreads;
            qv[k] = *reinterpret_cast<const uint4*>(qg + (i >> 6) * kKvDim + (i & 63) * 8);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + k * kThreads, h = i >> 6, c8 = i & 63;
            const uint4 v = qv[k];
            uint4 w;
            w.x = pack_f16x2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
            w.y = pack_f16x2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
            w.z = pack_f16x2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
            w.w = pack_f16x2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
            *reinterpret_cast<uint4*>(sm + kOffQ + (c8 >> 3) * 8192 + sw128(h, c8 & 7)) = w;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;

    if (n_tiles > 0 && warp == kSoftWarps) {
        // ------------------------------------------------------------ loader warp
        // Load g (g = 16 * tile + x) lands in landing slot g % 3. x < 8: pass-1
        // piece of d-block x, [128 rows x 64 d], as 32 gathers of 4 rows; x >= 8:
        // pass-2 piece y = x - 8, [64 rows x 128 d] of rows 64 (y >> 2).. and
        // columns 128 (y & 3).., as 16 gathers. Lane j owns tile rows 4j..4j+3.
        // Tile 0 is the window; later tiles are staged rows. Rows past the
        // split end repeat its last row (finite data the softmax masks).
        bool ok = true;
        int g = 0;
        const uint64_t lb_rows_win = lb * kWindow;
        const uint64_t lb_rows_stg = lb * (uint64_t)a.G;
        for (int tile = 0; tile < n_tiles && ok; ++tile) {
            const int tr0 = row0 + tile * kTileRows;
            int rq[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int row = min(tr0 + 4 * lane + k, row1 - 1);   // row1 > tr0 for every tile
                if (row < kWindow) {
                    rq[k] = (int)(lb_rows_win + row);
                } else {
                    int slot = ph[row - kWindow] - kWindow;
                    if (slot < 0 || slot >= a.G) {
                        atomicOr(a.err, kErrBounds);
                        slot = 0;
                    }
                    rq[k] = (int)(lb_rows_stg + slot);
                }
            }
            const bool in_win = tr0 < kWindow;          // tile 0: window rows only (tiles are 128 = W)
            const void* m64 = in_win ? (const void*)&maps.win64 : (const void*)&maps.stg64;
            const void* m128 = in_win ? (const void*)&maps.win128 : (const void*)&maps.stg128;
            for (int x = 0; x < kLoads; ++x) {
                const int ls = g % kNLand;
                if (!wait_or_abort(&ms.lempty[ls], ((g / kNLand) & 1) ^ 1, abort, a.err)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(&ms.lfull[ls], kLand);
                __syncwarp();
                const uint32_t land = smem_u32(sm + kOffLand + ls * kLand);
                if (x < 8) {
                    tma_gather4(land + lane * 1024, m64, 64 * x, rq[0], rq[1], rq[2], rq[3], &ms.lfull[ls]);
                } else {
                    const int y = x - 8, src = 16 * (y >> 2) + (lane & 15);
                    const int q0 = __shfl_sync(0xffffffffu, rq[0], src), q1 = __shfl_sync(0xffffffffu, rq[1], src);
                    const int q2 = __shfl_sync(0xffffffffu, rq[2], src), q3 = __shfl_sync(0xffffffffu, rq[3], src);
                    if (lane < 16) tma_gather4(land + lane * 2048, m128, 128 * (y & 3), q0, q1, q2, q3, &ms.lfull[ls]);
                }
                ++g;
            }
        }
        // after an abort, wait (bounded) for the copies of the last pieces issued
        if (!ok && lane == 0)
            for (int k = g > kNLand ? g - kNLand : 0; k < g; ++k)
                mbar_wait(&ms.lfull[k % kNLand], (k / kNLand) & 1, 1u << 20);
        __syncwarp();
    } else if (n_tiles > 0 && warp > kSoftWarps) {
        // warps 5-7 join for the output
    } else if (n_tiles > 0) {
        // ------------------------------------------------------------ converters + MMA issue
        constexpr uint32_t id1 = idesc_f16(0, 0, H);   // pass 1: K-major E and Q
        constexpr uint32_t id2 = idesc_f16(1, 1, H);   // pass 2: MN-major E^T and P
        bool cv_ok = true;
        int g = 0;                                       // pieces converted (all four warps in step)
        // convert landed piece g into operand slot g % 3 (this thread's 16 units)
        auto convert = [&]() {
            const int x = g & 15, ls = g % kNLand, s = g % kNOp;
            if (!wait_or_abort(&ms.lfull[ls], (g / kNLand) & 1, abort, a.err) ||
                !wait_or_abort(&ms.opempty[s], ((g / kNOp) & 1) ^ 1, abort, a.err)) {
                cv_ok = false;
                return;
            }
            const unsigned char* land = sm + kOffLand + ls * kLand;
            unsigned char* op = sm + kOffOp + s * kOp;
            const int u = tid;                           // unit owner index, 0..127
            if (x < 8) {
                // K-major [128 rows x 64 d] fp16: row r, 16-byte chunk d4 >> 1, half d4 & 1
                const int d4 = u & 15;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 f = *reinterpret_cast<const float4*>(land + 16 * u + 2048 * i);
                    const int r = (u >> 4) + 8 * i;
                    *reinterpret_cast<uint2*>(op + sw128(r, d4 >> 1) + 8 * (d4 & 1)) =
                        make_uint2(pack_f16x2(f.x, f.y), pack_f16x2(f.z, f.w));
                }
            } else {
                // MN-major [64 rows x 128 d] fp16: atom d4 >> 4 (64 d) at 8 KB, row r, chunk (d4 & 15) >> 1
                const int d4 = u & 31;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 f = *reinterpret_cast<const float4*>(land + 16 * u + 2048 * i);
                    const int r = (u >> 5) + 4 * i;
                    *reinterpret_cast<uint2*>(op + (d4 >> 4) * 8192 + sw128(r, (d4 & 15) >> 1) + 8 * (d4 & 1)) =
                        make_uint2(pack_f16x2(f.x, f.y), pack_f16x2(f.z, f.w));
                }
            }
            mbar_arrive(&ms.lempty[ls]);
            fence_async_smem();
            mbar_arrive(&ms.opfull[s]);
        };
        // lane 0 of warp 0: MMAs of piece g once all four warps have published it
        auto mma_piece = [&](int tile) {
            const int x = g & 15, s = g % kNOp;
            if (!wait_or_abort(&ms.opfull[s], (g / kNOp) & 1, abort, a.err)) {
                cv_ok = false;
                return;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(sm + kOffOp + s * kOp);
            if (x < 8) {
                const uint32_t sb = smem_u32(sm + kOffQ + x * 8192);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16kind(tmem + kColS, desc_sw128(sa + kk * 32, 16, 1024), desc_sw128(sb + kk * 32, 16, 1024),
                                id1, (x | kk) != 0);
            } else {
                const int y = x - 8, rb = y >> 2, mb = y & 3;
                const uint32_t sb = smem_u32(sm + kOffP + (64 * rb) * 128);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16kind(tmem + kColO + 64 * mb, desc_sw128(sa + kk * 2048, 8192, 1024),
                                desc_sw128(sb + kk * 2048, 8192, 1024), id2,
                                (tile > 0 || rb > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&ms.opempty[s]);
            if (x == 7) mma_commit(&ms.s_full);
            if (x == 15) mma_commit(&ms.o_full);
        };
        // the eight pieces of one pass: convert, then (warp 0) issue
        auto run_pass = [&](int tile) {
            for (int k = 0; k < 8; ++k) {
                if (cv_ok) convert();
                if (warp == 0) {
                    __syncwarp();
                    if (lane == 0 && cv_ok) mma_piece(tile);
                    __syncwarp();
                }
                ++g;
            }
        };

        // ------------------------------------------------------------ softmax
        const int r = tid;                                // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        bool ok = true;
        for (int tile = 0; tile < n_tiles && ok; ++tile) {
            run_pass(tile);                              // pass 1
            const bool got = cv_ok && wait_or_abort(&ms.s_full, tile & 1, abort, a.err);
            if (named_sync_or(1, kSoftWarps * 32, !got)) { ok = false; break; }
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
            const bool valid = row0 + tile * kTileRows + r < row1;
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
            named_sync(1, kSoftWarps * 32);
            if (tid < H) {
                const int h = tid;
                const float mt = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
                const float mu = ms.m_used[h];
                float al = 1.f;
                if (mt > mu + kLazy || (mu == -INFINITY && mt > -INFINITY)) {
                    al = exp2f(mu - mt);                  // 0 when mu = -inf
                    ms.m_used[h] = mt;
                    ms.l_run[h] *= al;
                    if (tile > 0 && al != 1.f) ms.rescale = 1;
                }
                ms.alpha[h] = al;
            }
            named_sync(1, kSoftWarps * 32);
#pragma unroll
            for (int h = 0; h < 64; ++h) v[h] = (h < H) ? exp2f(v[h] - ms.m_used[h]) : 0.f;
#pragma unroll
            for (int hh = 0; hh < H; hh += 32) {
                float red[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) red[i] = v[hh + i];
                ms.red[warp][hh + lane] = butterfly32<false>(red, lane);
            }
            // the previous tile's pass 2 still reads P and writes O: wait for it
            const bool prev = tile == 0 || wait_or_abort(&ms.o_full, (tile - 1) & 1, abort, a.err);
            if (named_sync_or(1, kSoftWarps * 32, !prev)) { ok = false; break; }
            if (tid < H)
                ms.l_run[tid] += (ms.red[0][tid] + ms.red[1][tid]) + (ms.red[2][tid] + ms.red[3][tid]);
            if (ms.rescale) {
                // O^T[d, h] *= alpha[h]: this thread owns TMEM lane r of each d-block
                tc_fence_after();
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
                    for (int c = 0; c < H; c += 16) {
                        float t16[16];
                        const uint32_t ta = tmem + lane_base + kColO + 64 * mb + c;
                        tmem_ld16(ta, t16);
                        tmem_ld_wait();
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
            named_sync(1, kSoftWarps * 32);
            if (tid == 0) ms.rescale = 0;
            mbar_arrive(&ms.p_full);
            if (warp == 0) {
                // the pass-2 MMAs read P: every softmax thread must have written it
                if (lane == 0 && !wait_or_abort(&ms.p_full, tile & 1, abort, a.err)) cv_ok = false;
                __syncwarp();
                tc_fence_after();
            }
            run_pass(tile);                              // pass 2
        }
        if (warp == 0) {
            // drain: completes once every MMA issued above has completed
            if (lane == 0) {
                mma_commit(&ms.drain);
                if (!mbar_wait(&ms.drain, 0, 1u << 26)) atomicOr(a.err, kErrTimeout);
            }
            __syncwarp();
        }
        const bool got = ok && wait_or_abort(&ms.o_full, (n_tiles - 1) & 1, abort, a.err);
        ok = !named_sync_or(1, kSoftWarps * 32, !got);    // the same verdict in all 128 threads
        if (tid < H) ms.alpha[tid] = 1.f / ms.l_run[tid];
        if (tid == 0) ms.epi_ok = ok ? 1 : 0;
    }

    // ---------------------------------------------------------------- epilogue: all 8 warps
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool single = it.n_splits == 1;
    float* dst = single ? a.out + lb * H * kKvDim : a.part_o + (size_t)item_idx * H * kKvDim;
    if (n_tiles > 0 && ms.epi_ok) {
        // warp w reads TMEM lanes 32 (w & 3).. of d-blocks 2 (w >> 2) and 2 (w >> 2) + 1
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
        for (int mm = 0; mm < 2; ++mm) {
            const int mb = 2 * (warp >> 2) + mm;
            const int d = mb * 128 + (warp & 3) * 32 + lane;
#pragma unroll
            for (int c = 0; c < H; c += 16) {
                float t16[16];
                tmem_ld16(tmem + lane_base + kColO + 64 * mb + c, t16);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int h = c + i;
                    if (single) dst[h * kKvDim + d] = t16[i] * ms.alpha[h];
                    else __stcg(&dst[h * kKvDim + d], t16[i]);
                }
            }
        }
    } else if (!single) {
        for (int i = tid; i < H * kKvDim; i += kThreads) __stcg(&dst[i], 0.f);
    }
    if (!single && tid < H) {
        float* pml = a.part_ml + (size_t)item_idx * 2 * H;
        __stcg(&pml[tid], ms.m_used[tid]);
        __stcg(&pml[H + tid], n_tiles > 0 && ms.epi_ok ? ms.l_run[tid] : 0.f);
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && n_tiles > 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (it.n_splits == 1) return;

    // ---------------------------------------------------------------- last CTA merges the splits
    __threadfence();
    __syncthreads();
    if (tid == 0) ms.ticket = atomicAdd(&a.counters[lb], 1u);
    __syncthreads();
    if (ms.ticket != (unsigned)(it.n_splits - 1)) return;
    __threadfence();
    const int ns = it.n_splits;
    const int base = item_idx - it.split;
    float* wts = reinterpret_cast<float*>(sm + kOffLand);   // [ns][H]
    for (int h = tid; h < H; h += kThreads) {
        float M = -INFINITY;
        for (int s = 0; s < ns; ++s) {
            const float* ml = a.part_ml + (size_t)(base + s) * 2 * H;
            if (__ldcg(&ml[H + h]) > 0.f) M = fmaxf(M, __ldcg(&ml[h]));
        }
        float L = 0.f;
        for (int s = 0; s < ns; ++s) {
            const float* ml = a.part_ml + (size_t)(base + s) * 2 * H;
            const float ls = __ldcg(&ml[H + h]);
            const float w = ls > 0.f ? exp2f(__ldcg(&ml[h]) - M) : 0.f;
            wts[s * H + h] = w;
            L += w * ls;
        }
        const float inv = 1.f / L;
        for (int s = 0; s < ns; ++s) wts[s * H + h] *= inv;
    }
    __syncthreads();
    float* o = a.out + lb * H * kKvDim;
    for (int i = tid; i < H * kKvDim / 4; i += kThreads) {
        const int h = (i * 4) / kKvDim;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < ns; ++s) {
            const float w = wts[s * H + h];
            if (w == 0.f) continue;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part_o + (size_t)(base + s) * H * kKvDim) + i);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        reinterpret_cast<float4*>(o)[i] = acc;
    }
    if (tid == 0) a.counters[lb] = 0u;
}

template <int H>
cudaError_t launch_h(const AttnArgs& args, const AttnMaps& maps, int n_items, cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    attend_tc_kernel<H><<<n_items, kThreads, kSmemBytes, st>>>(args, maps);
    return cudaGetLastError();
}

}  // namespace

int attend_max_splits() { return kMaxSplits; }

// 2-D fp32 map over [rows][512] with a box of `box` columns x 1 row, no swizzle.
static cudaError_t encode_rows_map(CUtensorMap* m, const float* base, unsigned long long rows, unsigned box) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        cudaDriverEntryPointQueryResult qr;
        cudaError_t e = cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", (void**)&enc, cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !enc) return cudaErrorNotSupported;
    }
    cuuint64_t dims[2] = {(cuuint64_t)kKvDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kKvDim * sizeof(float)};
    cuuint32_t boxd[2] = {box, 1};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, boxd,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_attend(const AttnItem* items, int item0, int n_items, int split_rows,
                          int n_heads, int L, int B, int G, int S, const uint16_t* q, const float* window,
                          const float* staging, const int32_t* phys, const int32_t* count_l,
                          float* out, float* part_o, float* part_ml, unsigned* counters,
                          uint32_t* err, cudaStream_t st) {
    if (n_items <= 0) return cudaSuccess;
    if (split_rows % kTileRows != 0) return cudaErrorInvalidValue;
    AttnMaps maps;
    const unsigned long long win_rows = (unsigned long long)L * B * kWindow;
    const unsigned long long stg_rows = (unsigned long long)L * B * G;
    cudaError_t e = encode_rows_map(&maps.win64, window, win_rows, 64);
    if (e == cudaSuccess) e = encode_rows_map(&maps.win128, window, win_rows, 128);
    if (e == cudaSuccess) e = encode_rows_map(&maps.stg64, staging, stg_rows, 64);
    if (e == cudaSuccess) e = encode_rows_map(&maps.stg128, staging, stg_rows, 128);
    if (e != cudaSuccess) return e;
    AttnArgs args{items, item0, split_rows, B, G, S, q, window, staging, phys, count_l,
                  out, part_o, part_ml, counters, err,
                  (float)(1.4426950408889634 / std::sqrt((double)kKvDim))};
    switch (n_heads) {
        case 16: return launch_h<16>(args, maps, n_items, st);
        case 32: return launch_h<32>(args, maps, n_items, st);
        case 64: return launch_h<64>(args, maps, n_items, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace srh
