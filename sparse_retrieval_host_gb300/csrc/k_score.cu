// K-score: memory-indexer scoring + ensemble for every compressed chunk, with
// mma.sync: the path for per-indexer key sets (indexer i scores its own key
// set i; three key streams) and for one key set below kTcMinChunks chunks per
// call. Longer single-set streams run on the tensor-core kernel of
// k_score_tc.cu.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 技术细节 / 架构概览,
// scoring box steps 1-3, and the FlashMemory-DeepSeek-V4 summary, sections
// "LSA 让模型预判 KV chunk" and "Memory Indexer 放哪里":
//   s_{i,h}(c) = <Q[i,h,:], K[c,:]>, s_i(c) = scale * max_h s_{i,h}(c) + b_i,
//   s(c) = max_i s_i(c) (OR-mode) or mean_i s_i(c).
//
// The keys are streamed once (256 B per chunk) with 16-byte non-allocating
// loads; the 24 x 128 query block stays in registers as mma B fragments. Each
// warp scores 16 chunks per step with bf16 m16n8k16 MMAs (fp32 accumulation):
// one n-tile of 8 columns is exactly one indexer's 8 heads, so the head max is
// a 4-lane shuffle. The epilogue writes the fp32 score and bumps a 4096-bin
// histogram of its order-preserving key (top 12 bits) that the selector uses
// to skip its first radix pass; a pass that follows a threshold selection
// builds no histogram and instead appends the chunks above that threshold to
// the selection's candidate list (warp-aggregated).
//
// The reduction dimension is permuted inside every 32-wide block of d so each
// lane reads 16 contiguous bytes of a key row; A and B use the same
// permutation, so the dot products are unchanged.
#include "srh_internal.cuh"

namespace srh {
namespace {

constexpr int kScoreWarps = 8;

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

struct KeyTile {
    uint4 r0[4];   // row g,   d blocks j = 0..3 (16 B each at 32j + 8t)
    uint4 r1[4];   // row g+8
};

__device__ __forceinline__ void load_tile(KeyTile& kt, const uint16_t* keys_b, long long c0, int n,
                                          int g, int t) {
    const long long ra = c0 + g, rb = c0 + g + 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        kt.r0[j] = make_uint4(0, 0, 0, 0);
        kt.r1[j] = make_uint4(0, 0, 0, 0);
    }
    if (ra < n) {
        const uint16_t* p = keys_b + ra * kIdxDim + 8 * t;
#pragma unroll
        for (int j = 0; j < 4; ++j) kt.r0[j] = ld_stream(p + 32 * j);
    }
    if (rb < n) {
        const uint16_t* p = keys_b + rb * kIdxDim + 8 * t;
#pragma unroll
        for (int j = 0; j < 4; ++j) kt.r1[j] = ld_stream(p + 32 * j);
    }
}

// kSets = 1: one key set shared by the three indexers; kSets = 3: indexer i
// scores against its own key set i (key sets `set_stride` elements apart).
template <int kSets>
__global__ void __launch_bounds__(kScoreWarps * 32, kSets == 1 ? 2 : 1)
score_kernel(const uint16_t* __restrict__ keys, long long set_stride, int n, const uint16_t* __restrict__ q,
             float scale, float b0, float b1, float b2, int ensemble, float* __restrict__ scores,
             uint32_t* __restrict__ hist, const CandSink sink) {
    __shared__ uint32_t h_s[kHistBins];
    pdl_trigger();
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    if (hist)
        for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h_s[i] = 0;

    // B fragments: bq[i][k-step][2]; indexer i = n-tile i, head = g.
    uint32_t bq[kIdx][8][2];
    const uint16_t* qb = q + (size_t)b * kIdx * kIdxHeads * kIdxDim;
#pragma unroll
    for (int i = 0; i < kIdx; ++i) {
        const uint16_t* row = qb + (i * kIdxHeads + g) * kIdxDim + 8 * t;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + 32 * j);
            bq[i][2 * j][0] = v.x;
            bq[i][2 * j][1] = v.y;
            bq[i][2 * j + 1][0] = v.z;
            bq[i][2 * j + 1][1] = v.w;
        }
    }
    __syncthreads();

    const uint16_t* keys_b = keys + (size_t)b * n * kIdxDim;
    float* scores_b = scores + (size_t)b * n;
    const long long n_tiles = (n + 15) / 16;
    const long long stride = (long long)gridDim.x * kScoreWarps;
    long long tile = (long long)blockIdx.x * kScoreWarps + warp;
    const float bias[3] = {b0, b1, b2};

    // one unit = (tile, key set); the next unit's keys load while this one's MMAs run
    KeyTile cur, nxt;
    if (tile < n_tiles) load_tile(cur, keys_b, tile * 16, n, g, t);
    for (; tile < n_tiles; tile += stride) {
        const long long next = tile + stride;
        float acc[kIdx][4];
#pragma unroll
        for (int i = 0; i < kIdx; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int u = 0; u < kSets; ++u) {
            if (u + 1 < kSets) load_tile(nxt, keys_b + (u + 1) * set_stride, tile * 16, n, g, t);
            else if (next < n_tiles) load_tile(nxt, keys_b, next * 16, n, g, t);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int i = 0; i < kIdx; ++i) {
                    if (kSets != 1 && i != u) continue;   // per-set keys: indexer u only
                    mma_bf16(acc[i], cur.r0[j].x, cur.r1[j].x, cur.r0[j].y, cur.r1[j].y,
                             bq[i][2 * j][0], bq[i][2 * j][1]);
                    mma_bf16(acc[i], cur.r0[j].z, cur.r1[j].z, cur.r0[j].w, cur.r1[j].w,
                             bq[i][2 * j + 1][0], bq[i][2 * j + 1][1]);
                }
            }
            if (u + 1 < kSets) cur = nxt;
        }
        // max over the 8 heads of each indexer: 2 in-thread, 4 lanes of the quad
        float sa[kIdx], sb[kIdx];
#pragma unroll
        for (int i = 0; i < kIdx; ++i) {
            float ma = fmaxf(acc[i][0], acc[i][1]);
            float mb = fmaxf(acc[i][2], acc[i][3]);
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            sa[i] = fmaf(scale, ma, bias[i]);
            sb[i] = fmaf(scale, mb, bias[i]);
        }
        float ea, eb;
        if (ensemble == SRH_ENSEMBLE_MAX) {
            ea = fmaxf(fmaxf(sa[0], sa[1]), sa[2]);
            eb = fmaxf(fmaxf(sb[0], sb[1]), sb[2]);
        } else {
            ea = (sa[0] + sa[1] + sa[2]) / 3.0f;
            eb = (sb[0] + sb[1] + sb[2]) / 3.0f;
        }
        // lane t = 0 writes chunk c0 + g, lane t = 1 chunk c0 + g + 8
        const long long c = tile * 16 + g + (t == 1 ? 8 : 0);
        const float e = t == 0 ? ea : eb;
        const bool wr = t < 2 && c < n;
        const uint32_t key = ordered_key(e);
        if (wr) {
            scores_b[c] = e;
            if (hist) atomicAdd(&h_s[key >> 20], 1u);
        }
        if (sink.cand) append_candidate(sink, b, wr && key > sink.key, key, (uint32_t)c);
        cur = nxt;
    }
    if (!hist) return;
    __syncthreads();
    uint32_t* hb = hist + (size_t)b * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
        if (h_s[i]) atomicAdd(&hb[i], h_s[i]);
}

__global__ void hist_kernel(const float* __restrict__ scores, int n, uint32_t* __restrict__ hist) {
    __shared__ uint32_t h_s[kHistBins];
    pdl_trigger();
    const int b = blockIdx.y;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h_s[i] = 0;
    __syncthreads();
    const float* sb = scores + (size_t)b * n;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        atomicAdd(&h_s[ordered_key(sb[i]) >> 20], 1u);
    __syncthreads();
    uint32_t* hb = hist + (size_t)b * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
        if (h_s[i]) atomicAdd(&hb[i], h_s[i]);
}

}  // namespace

cudaError_t launch_score(const uint16_t* keys, int n, int B, const uint16_t* q, float scale,
                         const float* bias3, int ensemble, float* scores, uint32_t* hist, uint32_t* err,
                         int sm_count, cudaStream_t st, int key_sets, bool clear_hist, CandSink sink,
                         bool clear_cand) {
    if (clear_hist && hist) {
        const cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(uint32_t) * kHistBins * B, st);
        if (e != cudaSuccess) return e;
    }
    if (clear_cand && sink.cand) {
        const cudaError_t e = cudaMemsetAsync(sink.cnt, 0, sizeof(int) * B, st);
        if (e != cudaSuccess) return e;
    }
    // One key set over many tiles: the tensor-core stream (k_score_tc.cu). Its
    // fixed cost (TMEM, barriers, tensor maps) is about 1.5 us more per call than
    // this kernel's, which its higher streaming rate repays only on long streams:
    // measured 16.8 against 15.0 us at 2^18 chunks, 47 against 60 us at 2^20.
    if (key_sets == 1 && (long long)B * n >= kTcMinChunks)
        return launch_score_tc(keys, n, B, q, scale, bias3, ensemble, scores, hist, err, sm_count, st, sink);
    const long long tiles = (n + 15) / 16;
    long long bx = (tiles + kScoreWarps - 1) / kScoreWarps;
    const long long cap = (2LL * sm_count + B - 1) / B;
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    dim3 grid((unsigned)bx, (unsigned)B);
    const long long set_stride = (long long)B * n * kIdxDim;
    if (key_sets == 3)
        score_kernel<3><<<grid, kScoreWarps * 32, 0, st>>>(keys, set_stride, n, q, scale, bias3[0], bias3[1],
                                                           bias3[2], ensemble, scores, hist, sink);
    else
        score_kernel<1><<<grid, kScoreWarps * 32, 0, st>>>(keys, 0, n, q, scale, bias3[0], bias3[1], bias3[2],
                                                           ensemble, scores, hist, sink);
    return cudaGetLastError();
}

cudaError_t launch_hist(const float* scores, int n, int B, uint32_t* hist, cudaStream_t st, bool clear_hist) {
    if (clear_hist) {
        const cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(uint32_t) * kHistBins * B, st);
        if (e != cudaSuccess) return e;
    }
    long long bx = (n + 4095) / 4096;
    if (bx > 64) bx = 64;
    if (bx < 1) bx = 1;
    hist_kernel<<<dim3((unsigned)bx, (unsigned)B), 256, 0, st>>>(scores, n, hist);
    return cudaGetLastError();
}

}  // namespace srh
