// K-score with fp8 indexer keys.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 限制与未来工作:
// the indexer keys are the per-step stream of the scoring pass, and quantizing
// them to fp8/int8 (with a scorer kernel that reads them) is the planned cut.
// Keys are stored as e4m3 codes with one fp32 scale per chunk:
//     kscale_c = amax_c / 448,   K8[c][d] = e4m3(K[c][d] / kscale_c)
// rounded to nearest (ties to even) and saturated, computed with IEEE fp32
// division. Scoring reads 128 B of codes + 4 B of scale per chunk instead of
// 256 B of bf16:
//     s_i(c) = scale * kscale_c * max_h <Q[i,h,:], e4m3(K8[c,:])> + b_i.
// e4m3 values are exact in fp16, and so are bf16 queries of normal fp16 range,
// so the MMAs run on fp16 operands (m16n8k16, fp32 accumulate) with the codes
// widened in registers; kscale_c > 0 commutes with the head max.
//
// Reduction order: within each 64-wide block of d, lane t of a quad reads the
// 16 contiguous codes d = 64 jb + 16 t .. + 15 of its row; k-step s of the block
// takes codes 4s .. 4s+3 of every lane (slots 2t, 2t+1 <- 4s, 4s+1 and slots
// 2t+8, 2t+9 <- 4s+2, 4s+3). The query fragments use the same map, so the dot
// products are unchanged.
#include "srh_internal.cuh"

namespace srh {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 codes (low byte first) -> f16x2 (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    const unsigned short v = (unsigned short)two;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------- quantizer
// One warp per chunk: lane l holds d = 4l .. 4l+3.
__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ keys, long long total,
                                                       uint8_t* __restrict__ codes, float* __restrict__ kscale) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long c = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < total; c += warps) {
        const uint2 raw = *reinterpret_cast<const uint2*>(keys + c * kIdxDim + 4 * lane);
        float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(amax, 448.0f);
        uint32_t word = 0;
        if (s > 0.f) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(__fdiv_rn(x[j], s), __NV_SATFINITE, __NV_E4M3);
                word |= (uint32_t)q << (8 * j);
            }
        }
        *reinterpret_cast<uint32_t*>(codes + c * kIdxDim + 4 * lane) = word;
        if (lane == 0) kscale[c] = s;
    }
}

// ---------------------------------------------------------------- scorer
struct Tile8 {
    uint4 r0[2];   // row g:   codes 64 jb + 16 t .. + 15, jb = 0, 1
    uint4 r1[2];   // row g+8
    float s0, s1;  // kscale of the two rows
};

__device__ __forceinline__ void load_tile8(Tile8& kt, const uint8_t* codes_b, const float* ks_b, long long c0,
                                           int n, int g, int t) {
    const long long ra = c0 + g, rb = c0 + g + 8;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        kt.r0[j] = make_uint4(0, 0, 0, 0);
        kt.r1[j] = make_uint4(0, 0, 0, 0);
    }
    kt.s0 = kt.s1 = 0.f;
    if (ra < n) {
        const uint8_t* p = codes_b + ra * kIdxDim + 16 * t;
        kt.r0[0] = ld_stream(p);
        kt.r0[1] = ld_stream(p + 64);
        kt.s0 = __ldg(ks_b + ra);
    }
    if (rb < n) {
        const uint8_t* p = codes_b + rb * kIdxDim + 16 * t;
        kt.r1[0] = ld_stream(p);
        kt.r1[1] = ld_stream(p + 64);
        kt.s1 = __ldg(ks_b + rb);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int s) {
    return s == 0 ? v.x : (s == 1 ? v.y : (s == 2 ? v.z : v.w));
}

__global__ void __launch_bounds__(kWarps * 32, 2)
score_fp8_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ kscale, int n,
                 const uint16_t* __restrict__ q, float scale, float b0, float b1, float b2, int ensemble,
                 float* __restrict__ scores, uint32_t* __restrict__ hist) {
    __shared__ uint32_t h_s[kHistBins];
    pdl_trigger();
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h_s[i] = 0;

    // query fragments, fp16: bq[i][4 jb + s] = {d 4s, 4s+1 | d 4s+2, 4s+3} of
    // the 16 values at 64 jb + 16 t of head g of indexer i
    uint32_t bq[kIdx][8][2];
    const uint16_t* qb = q + (size_t)b * kIdx * kIdxHeads * kIdxDim;
#pragma unroll
    for (int i = 0; i < kIdx; ++i) {
        const uint16_t* row = qb + (i * kIdxHeads + g) * kIdxDim + 16 * t;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
            const uint4 lo = *reinterpret_cast<const uint4*>(row + 64 * jb);
            const uint4 hi = *reinterpret_cast<const uint4*>(row + 64 * jb + 8);
            const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t p0 = w[2 * s], p1 = w[2 * s + 1];   // bf16 pairs (4s, 4s+1), (4s+2, 4s+3)
                bq[i][4 * jb + s][0] = pack_f16x2(__uint_as_float(p0 << 16), __uint_as_float(p0 & 0xffff0000u));
                bq[i][4 * jb + s][1] = pack_f16x2(__uint_as_float(p1 << 16), __uint_as_float(p1 & 0xffff0000u));
            }
        }
    }
    __syncthreads();

    const uint8_t* codes_b = codes + (size_t)b * n * kIdxDim;
    const float* ks_b = kscale + (size_t)b * n;
    float* scores_b = scores + (size_t)b * n;
    const long long n_tiles = (n + 15) / 16;
    const long long stride = (long long)gridDim.x * kWarps;
    long long tile = (long long)blockIdx.x * kWarps + warp;
    const float bias[3] = {b0, b1, b2};

    Tile8 cur, nxt;
    if (tile < n_tiles) load_tile8(cur, codes_b, ks_b, tile * 16, n, g, t);
    for (; tile < n_tiles; tile += stride) {
        const long long next = tile + stride;
        if (next < n_tiles) load_tile8(nxt, codes_b, ks_b, next * 16, n, g, t);
        float acc[kIdx][4];
#pragma unroll
        for (int i = 0; i < kIdx; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t w0 = word_of(cur.r0[jb], s), w1 = word_of(cur.r1[jb], s);
                const uint32_t a0 = e4m3x2_to_f16x2(w0), a2 = e4m3x2_to_f16x2(w0 >> 16);
                const uint32_t a1 = e4m3x2_to_f16x2(w1), a3 = e4m3x2_to_f16x2(w1 >> 16);
#pragma unroll
                for (int i = 0; i < kIdx; ++i)
                    mma_f16(acc[i], a0, a1, a2, a3, bq[i][4 * jb + s][0], bq[i][4 * jb + s][1]);
            }
        }
        // max over the 8 heads (2 in-thread, 4 lanes of the quad), then the chunk scale
        float sa[kIdx], sb[kIdx];
#pragma unroll
        for (int i = 0; i < kIdx; ++i) {
            float ma = fmaxf(acc[i][0], acc[i][1]);
            float mb = fmaxf(acc[i][2], acc[i][3]);
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            sa[i] = fmaf(scale, ma * cur.s0, bias[i]);
            sb[i] = fmaf(scale, mb * cur.s1, bias[i]);
        }
        float ea, eb;
        if (ensemble == SRH_ENSEMBLE_MAX) {
            ea = fmaxf(fmaxf(sa[0], sa[1]), sa[2]);
            eb = fmaxf(fmaxf(sb[0], sb[1]), sb[2]);
        } else {
            ea = (sa[0] + sa[1] + sa[2]) / 3.0f;
            eb = (sb[0] + sb[1] + sb[2]) / 3.0f;
        }
        const long long c0 = tile * 16;
        if (t == 0 && c0 + g < n) {
            scores_b[c0 + g] = ea;
            atomicAdd(&h_s[ordered_key(ea) >> 20], 1u);
        } else if (t == 1 && c0 + g + 8 < n) {
            scores_b[c0 + g + 8] = eb;
            atomicAdd(&h_s[ordered_key(eb) >> 20], 1u);
        }
        cur = nxt;
    }
    __syncthreads();
    uint32_t* hb = hist + (size_t)b * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
        if (h_s[i]) atomicAdd(&hb[i], h_s[i]);
}

}  // namespace

cudaError_t launch_quantize_keys(const uint16_t* keys, long long total, uint8_t* codes, float* kscale,
                                 int sm_count, cudaStream_t st) {
    if (total <= 0) return cudaSuccess;
    long long bx = (total + 7) / 8;
    if (bx > 16LL * sm_count) bx = 16LL * sm_count;
    quantize_kernel<<<(unsigned)bx, 256, 0, st>>>(keys, total, codes, kscale);
    return cudaGetLastError();
}

cudaError_t launch_score_fp8(const uint8_t* codes, const float* kscale, int n, int B, const uint16_t* q, float scale,
                             const float* bias3, int ensemble, float* scores, uint32_t* hist, int sm_count,
                             cudaStream_t st, bool clear_hist) {
    if (clear_hist) {
        const cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(uint32_t) * kHistBins * B, st);
        if (e != cudaSuccess) return e;
    }
    const long long tiles = (n + 15) / 16;
    long long bx = (tiles + kWarps - 1) / kWarps;
    const long long cap = (2LL * sm_count + B - 1) / B;
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    score_fp8_kernel<<<dim3((unsigned)bx, (unsigned)B), kWarps * 32, 0, st>>>(
        codes, kscale, n, q, scale, bias3[0], bias3[1], bias3[2], ensemble, scores, hist);
    return cudaGetLastError();
}

}  // namespace srh
