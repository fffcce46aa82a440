// K-select: top-k and sigmoid-threshold selection with a fixed tie-break.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 技术细节 / 架构概览,
// scoring box step 3 (global top-k, index_topk = 512), and the
// FlashMemory-DeepSeek-V4 summary, section "LSA 让模型预判 KV chunk" (entries
// whose sigmoid score exceeds a threshold are recalled; the count varies).
//
// Every chunk gets a unique 64-bit composite key
//     (ordered_key(s) << 32) | ~c
// so "larger composite" means (score descending, index ascending) and ties
// cannot exist. One CTA per sequence runs a radix select on the composite:
// the first 12-bit digit histogram comes from the scoring pass; further
// 12-bit digits are histogrammed only while the class holding the k-th key
// has more than kCandCap members. Then one pass collects the keys above the
// class and the class members into shared memory, a bitonic sort picks the
// needed class members, and a last bitonic sort orders the output.
//
// Threshold mode (s > ln(tau/(1-tau)), strict) collects the passing chunks in
// one pass; if more than `clamp` pass, the best `clamp` of them are exactly the
// global top-`clamp`, so it falls through to the top-k path with k = clamp.
#include "srh_internal.cuh"

namespace srh {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kCandCap = 8192;
constexpr int kDigit = 12;

__device__ __forceinline__ unsigned long long composite(uint32_t key, uint32_t idx) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~idx);
}

// Inclusive block scan of one int per thread (blockDim.x == kSelThreads).
__device__ int block_inclusive_scan(int v, int* warp_buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_buf[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_buf[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        warp_buf[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? warp_buf[warp - 1] : 0);
    __syncthreads();
    return r;
}

// Descending bitonic sort of a[0..m) in shared memory (pads to a power of two
// with zeros, which sort last). All threads of the block must call it.
__device__ void bitonic_sort_desc(unsigned long long* a, int m) {
    int m2 = 1;
    while (m2 < m) m2 <<= 1;
    for (int i = m + threadIdx.x; i < m2; i += blockDim.x) a[i] = 0ull;
    __syncthreads();
    for (int size = 2; size <= m2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (m2 >> 1); i += blockDim.x) {
                const int lo = 2 * stride * (i / stride) + (i % stride);
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const unsigned long long x = a[lo], y = a[hi];
                if ((x < y) == up) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// Descending bitonic sort of one element per thread over the first m2 threads
// (m2 a power of two <= blockDim.x); returns the element now at position tid.
// Strides below a warp use shuffles, larger ones go through `xchg` in shared
// memory. Threads past m2 sort their own padding. All threads must call it.
__device__ unsigned long long reg_bitonic_desc(unsigned long long v, int m2, unsigned long long* xchg) {
    const int tid = threadIdx.x;
    for (int size = 2; size <= m2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            unsigned long long o;
            if (stride >= 32) {
                xchg[tid] = v;
                __syncthreads();
                o = xchg[tid ^ stride];
                __syncthreads();
            } else {
                o = __shfl_xor_sync(0xffffffffu, v, stride);
            }
            const bool up = (tid & size) == 0;
            const bool lower = (tid & stride) == 0;
            v = (lower == up) ? (v > o ? v : o) : (v < o ? v : o);
        }
    }
    return v;
}

__device__ __forceinline__ int pow2_at_least(int m) {
    int m2 = 32;
    while (m2 < m) m2 <<= 1;
    return m2;
}

struct SelShared {
    uint32_t hist[kHistBins];
    int warp_buf[32];
    int n_out;
    int n_cand;
    int found_digit;
    int found_above;
};

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float* __restrict__ scores, int n, int mode, int k, float thresh, int clamp,
              int S, const uint32_t* __restrict__ hist_in, int32_t* __restrict__ sel,
              int32_t* __restrict__ count) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw + sizeof(SelShared));
    unsigned long long* outk = cand + kCandCap;

    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const float* sc = scores + (size_t)b * n;
    int32_t* sel_b = sel + (size_t)b * S;

    if (tid == 0) {
        sh.n_out = 0;
        sh.n_cand = 0;
    }
    __syncthreads();

    int K;
    if (mode == SRH_SELECT_THRESH) {
        const uint32_t kt = ordered_key(thresh);
        for (int i = tid; i < n; i += kSelThreads) {
            const uint32_t key = ordered_key(sc[i]);
            if (key > kt) {
                const int pos = atomicAdd(&sh.n_cand, 1);
                if (pos < kCandCap) cand[pos] = composite(key, (uint32_t)i);
            }
        }
        __syncthreads();
        const int total = sh.n_cand;
        if (total <= clamp) {
            if (total <= kSelThreads) {
                unsigned long long v = tid < total ? cand[tid] : 0ull;
                __syncthreads();
                v = reg_bitonic_desc(v, pow2_at_least(total), outk);
                if (tid < total) sel_b[tid] = (int32_t)(~(uint32_t)v);
            } else {
                bitonic_sort_desc(cand, total);
                for (int i = tid; i < total; i += kSelThreads) sel_b[i] = (int32_t)(~(uint32_t)cand[i]);
            }
            if (tid == 0) count[b] = total;
            return;
        }
        K = clamp;
        __syncthreads();
        if (tid == 0) sh.n_cand = 0;
        __syncthreads();
    } else {
        K = k < n ? k : n;
    }
    if (K <= 0) {
        if (tid == 0) count[b] = 0;
        return;
    }

    // ---- radix select of the K-th largest composite key
    unsigned long long prefix = 0ull;
    int pbits = 0;
    int remaining = K;
    bool use_hist_in = hist_in != nullptr;
    for (;;) {
        const int D = (64 - pbits) < kDigit ? (64 - pbits) : kDigit;
        const int shift = 64 - pbits - D;
        const unsigned long long mask = (1ull << D) - 1ull;
        if (tid == 0) sh.found_digit = -1;
        if (pbits == 0 && use_hist_in) {
            for (int i = tid; i < kHistBins; i += kSelThreads) sh.hist[i] = hist_in[(size_t)b * kHistBins + i];
        } else {
            for (int i = tid; i < kHistBins; i += kSelThreads) sh.hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kSelThreads) {
                const unsigned long long c = composite(ordered_key(sc[i]), (uint32_t)i);
                if (pbits == 0 || (c >> (64 - pbits)) == (prefix >> (64 - pbits)))
                    atomicAdd(&sh.hist[(c >> shift) & mask], 1u);
            }
        }
        __syncthreads();
        // thread tid owns bins 4095-4*tid .. 4092-4*tid (descending)
        int local = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) local += (int)sh.hist[kHistBins - 1 - 4 * tid - j];
        const int incl = block_inclusive_scan(local, sh.warp_buf);
        int cum = incl - local;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int bin = kHistBins - 1 - 4 * tid - j;
            const int c = (int)sh.hist[bin];
            if (c > 0 && cum < remaining && remaining <= cum + c) {
                sh.found_digit = bin;
                sh.found_above = cum;
            }
            cum += c;
        }
        __syncthreads();
        const int digit = sh.found_digit;
        if (digit < 0) {
            // the histogram handed in does not describe these scores: rebuild it
            if (pbits == 0 && use_hist_in) {
                use_hist_in = false;
                __syncthreads();
                continue;
            }
            if (tid == 0) count[b] = 0;   // unreachable for consistent inputs
            return;
        }
        const int cls = (int)sh.hist[digit];
        remaining -= sh.found_above;
        prefix |= ((unsigned long long)digit) << shift;
        pbits += D;
        __syncthreads();
        if (cls <= kCandCap || pbits >= 64) break;
    }

    // ---- collect: keys above the class go out directly, class members to cand
    for (int i = tid; i < n; i += kSelThreads) {
        const unsigned long long c = composite(ordered_key(sc[i]), (uint32_t)i);
        const unsigned long long top = c >> (64 - pbits), pre = prefix >> (64 - pbits);
        if (top > pre) {
            const int pos = atomicAdd(&sh.n_out, 1);
            if (pos < K) outk[pos] = c;
        } else if (top == pre) {
            const int pos = atomicAdd(&sh.n_cand, 1);
            if (pos < kCandCap) cand[pos] = c;
        }
    }
    __syncthreads();
    // consistent inputs give n_above == K - remaining; the clamps keep a stale
    // histogram from writing outside the arrays
    const int n_above = sh.n_out < K ? sh.n_out : K;
    const int n_cls = sh.n_cand < kCandCap ? sh.n_cand : kCandCap;
    if (n_above + n_cls <= kSelThreads) {
        // one register sort of everything at or above the class; keep the first K
        unsigned long long v = tid < n_above ? outk[tid] : (tid < n_above + n_cls ? cand[tid - n_above] : 0ull);
        __syncthreads();
        v = reg_bitonic_desc(v, pow2_at_least(n_above + n_cls), outk);
        if (tid < K) sel_b[tid] = (int32_t)(~(uint32_t)v);
        if (tid == 0) count[b] = K;
        return;
    }
    bitonic_sort_desc(cand, n_cls);
    for (int i = tid; i < remaining && n_above + i < K; i += kSelThreads) outk[n_above + i] = cand[i];
    __syncthreads();
    bitonic_sort_desc(outk, K);
    for (int i = tid; i < K; i += kSelThreads) sel_b[i] = (int32_t)(~(uint32_t)outk[i]);
    if (tid == 0) count[b] = K;
}

}  // namespace

cudaError_t launch_select(const float* scores, int n, int B, int mode, int k, float thresh,
                          int clamp, int S, const uint32_t* hist, int32_t* sel, int32_t* count,
                          cudaStream_t st) {
    const size_t smem = sizeof(SelShared) + sizeof(unsigned long long) * (kCandCap + kMaxSelect);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    select_kernel<<<B, kSelThreads, smem, st>>>(scores, n, mode, k, thresh, clamp, S, hist, sel, count);
    return cudaGetLastError();
}

}  // namespace srh
