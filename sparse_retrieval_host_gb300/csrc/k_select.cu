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
//
// Two accelerations, both exact:
//   * for large n, the per-sequence CTA works on a candidate list instead of
//     all n scores: the chunks that can be selected (first digit at or above
//     the cut-off digit of the k-th key, or above the threshold). A multi-CTA
//     collect pass appends them; in threshold mode the scoring pass after a
//     threshold selection has already appended the chunks above that same
//     threshold, and the collect pass is skipped. If the list overflows its
//     capacity, the CTA scans all n scores as before;
//   * when the first digit already isolates the selection, the output is
//     placed without a sort. The keys at or above the cut-off digit are
//     counted into 4096 fine buckets: a shift of the 32-bit score key over the
//     digits from the cut-off to the highest one present, so bucket order is
//     key order and a bucket holds a few keys. A prefix sum gives each bucket's
//     first output position; the keys are scattered into their buckets, and a
//     key's position is its bucket's start plus the number of larger keys in
//     its bucket.
// Histograms are owned four bins per thread, highest digit first (thread t:
// digits 4095-4t .. 4092-4t), read and written with one 16-byte access.
#include "srh_internal.cuh"

namespace srh {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kCandCap = 8192;
constexpr int kDigit = 12;
constexpr int kArr = kCandCap + kMaxSelect;             // cand + outk, contiguous in shared memory
constexpr unsigned kBucketWork = 256u * kSelThreads;   // bound on sum of squared bucket sizes
constexpr int kPre = 8;                                 // keys per thread held in registers
constexpr int kCollectThreads = 256;
constexpr int kCollectPer = 16;                         // scores per collect thread

__device__ __forceinline__ unsigned long long composite(uint32_t key, uint32_t idx) {
    return candidate_key(key, idx);
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

// Inclusive block scan of one int per thread with a single barrier
// (blockDim.x == kSelThreads, 32 warps): each warp adds up the totals of the
// warps before it itself. `total` receives the block's sum. Two calls on the
// same warp_buf must be separated by another barrier.
__device__ __forceinline__ int block_scan_1bar(int v, int* warp_buf, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_buf[warp] = v;
    __syncthreads();
    const int w = warp_buf[lane];
    total = __reduce_add_sync(0xffffffffu, w);
    return v + __reduce_add_sync(0xffffffffu, lane < warp ? w : 0);
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

// 16-byte aligned size: the 64-bit key arrays follow it in shared memory
struct alignas(16) SelShared {
    uint32_t hist[kHistBins];   // digit histogram of the rounds not handed in
    uint32_t fcnt[kHistBins];   // fine-bucket sizes
    int fpos[kHistBins];        // fine-bucket starts; after the scatter, ends
    int warp_buf[32];
    int n_out;
    int n_cand;
    int found_digit;
    int found_above;
    int found_cls;
    int top_digit;              // highest non-empty first digit
    unsigned sq;                // sum of squared fine-bucket sizes (saturating)
};
static_assert(sizeof(SelShared) % 16 == 0, "key arrays after SelShared need 8-byte alignment");
static_assert(offsetof(SelShared, fcnt) % 16 == 0 && offsetof(SelShared, fpos) % 16 == 0,
              "histograms are accessed 16 bytes at a time");

// The keys the selection runs over: all n scores of the sequence, or a
// candidate list of composites made by collect_kernel.
struct Src {
    const float* sc;
    const unsigned long long* cl;
    int n;
    __device__ __forceinline__ unsigned long long get(int j) const {
        return cl ? cl[j] : composite(ordered_key(sc[j]), (uint32_t)j);
    }
};

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float* scores, int n, int mode, int k, float thresh, int clamp,
              int S, uint32_t* hist_in, const unsigned long long* cand_in,
              int* cand_cnt, int cand_cap, int32_t* __restrict__ sel,
              int32_t* __restrict__ count) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelShared& sh = *reinterpret_cast<SelShared*>(smem_raw);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw + sizeof(SelShared));
    unsigned long long* outk = cand + kCandCap;

    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    int32_t* sel_b = sel + (size_t)b * S;
    pdl_trigger();
    pdl_wait();   // scores, histogram and candidates come from earlier kernels

    // The handed-in first-digit histogram is read once and left zeroed, so the
    // next scoring pass can add into it without clearing it first. Its loads
    // and the first keys of every thread are issued together: one round trip.
    static_assert(kHistBins == 4 * kSelThreads, "four histogram bins per thread");
    const int own = kHistBins - 4 - 4 * tid;   // bins own .. own + 3 belong to this thread
    uint32_t* hb = hist_in ? hist_in + (size_t)b * kHistBins : nullptr;
    uint4 h4 = make_uint4(0u, 0u, 0u, 0u);
    if (hb) h4 = *reinterpret_cast<const uint4*>(hb + own);

    // the key universe: a candidate list when one was made and did not overflow
    Src src{scores + (size_t)b * n, nullptr, n};
    if (cand_in) {
        const int nc = cand_cnt[b];
        if (nc >= 0 && nc <= cand_cap) {
            src.cl = cand_in + (size_t)b * cand_cap;
            src.n = nc;
        }
    }
    // keys tid + k * kSelThreads, k < kPre, stay in registers for every pass
    unsigned long long pre[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int i = tid + k * kSelThreads;
        pre[k] = i < src.n ? src.get(i) : 0ull;
    }
    auto each_key = [&](auto&& body) {
#pragma unroll
        for (int k = 0; k < kPre; ++k)
            if (tid + k * kSelThreads < src.n) body(pre[k]);
        for (int i = tid + kPre * kSelThreads; i < src.n; i += kSelThreads) body(src.get(i));
    };
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    if (hb) *reinterpret_cast<uint4*>(hb + own) = zero4;
    *reinterpret_cast<uint4*>(sh.fcnt + own) = zero4;

    if (tid == 0) {
        sh.n_out = 0;
        sh.n_cand = 0;
        sh.sq = 0u;
        sh.top_digit = 0;
    }
    __syncthreads();
    // every thread has read the candidate count: leave it zeroed for the next
    // candidate pass (which adds into it)
    if (cand_in && tid == 0) cand_cnt[b] = 0;

    int K;
    if (mode == SRH_SELECT_THRESH) {
        const uint32_t kt = ordered_key(thresh);
        each_key([&](unsigned long long c) {
            if ((uint32_t)(c >> 32) > kt) {
                const int pos = atomicAdd(&sh.n_cand, 1);
                if (pos < kCandCap) cand[pos] = c;
            }
        });
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
        uint4 c4;
        if (pbits == 0 && use_hist_in) {
            c4 = h4;
        } else {
            *reinterpret_cast<uint4*>(sh.hist + own) = zero4;
            __syncthreads();
            each_key([&](unsigned long long c) {
                if (pbits == 0 || (c >> (64 - pbits)) == (prefix >> (64 - pbits)))
                    atomicAdd(&sh.hist[(c >> shift) & mask], 1u);
            });
            __syncthreads();
            c4 = *reinterpret_cast<const uint4*>(sh.hist + own);
        }
        const uint32_t cb[4] = {c4.w, c4.z, c4.y, c4.x};   // digits own + 3 .. own
        const int local = (int)(cb[0] + cb[1] + cb[2] + cb[3]);
        int hist_total;
        const int incl = block_scan_1bar(local, sh.warp_buf, hist_total);
        int cum = incl - local;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int bin = own + 3 - j;
            const int c = (int)cb[j];
            if (c > 0 && cum < remaining && remaining <= cum + c) {
                sh.found_digit = bin;
                sh.found_above = cum;
                sh.found_cls = c;
            }
            if (pbits == 0 && c > 0 && cum == 0) sh.top_digit = bin;   // the first non-empty digit
            cum += c;
        }
        __syncthreads();
        const int digit = sh.found_digit;
        if (digit < 0 || (pbits == 0 && use_hist_in && hist_total != n)) {
            // the histogram handed in does not describe these scores (a count
            // that is not n means it was not cleared or not filled): rebuild it
            if (pbits == 0 && use_hist_in) {
                use_hist_in = false;
                __syncthreads();
                continue;
            }
            if (tid == 0) count[b] = 0;   // unreachable for consistent inputs
            return;
        }
        const int cls = sh.found_cls;
        remaining -= sh.found_above;
        prefix |= ((unsigned long long)digit) << shift;
        pbits += D;
        if (cls <= kCandCap || pbits >= 64) break;
        __syncthreads();
    }

    if (pbits == kDigit) {
        // ---- the first digit decides the class: place by fine buckets (no sort).
        // Keys at or above the cut-off digit span digits cut .. top, i.e. key32
        // in [cut << 20, (top + 1) << 20); a shift of fs = 8 + ceil(log2(top -
        // cut + 1)) maps that range onto 4096 ordered buckets.
        const uint32_t cut = (uint32_t)(prefix >> (64 - kDigit));
        const int nb = max(sh.top_digit - (int)cut + 1, 1);
        const int fs = 8 + (nb > 1 ? 32 - __clz(nb - 1) : 0);
        auto fine = [&](unsigned long long c) -> int {
            const uint32_t f = ((uint32_t)(c >> 32) - (cut << 20)) >> fs;
            return (int)min(f, (uint32_t)(kHistBins - 1));   // in range for consistent inputs
        };
        each_key([&](unsigned long long c) {
            if ((uint32_t)(c >> 52) >= cut) atomicAdd(&sh.fcnt[fine(c)], 1u);
        });
        __syncthreads();
        const uint4 f4 = *reinterpret_cast<const uint4*>(sh.fcnt + own);
        const uint32_t fb[4] = {f4.w, f4.z, f4.y, f4.x};   // buckets own + 3 .. own
        unsigned long long sq = 0ull;
#pragma unroll
        for (int j = 0; j < 4; ++j) sq += (unsigned long long)fb[j] * fb[j];
        const unsigned wsq = __reduce_add_sync(0xffffffffu, (unsigned)min(sq, (unsigned long long)(1u << 26)));
        if ((tid & 31) == 0 && wsq) atomicAdd(&sh.sq, min(wsq, 1u << 26));   // at most 2^31 in all
        const int flocal = (int)(fb[0] + fb[1] + fb[2] + fb[3]);
        int total;
        const int fincl = block_scan_1bar(flocal, sh.warp_buf, total);
        int fc = fincl - flocal;
        int4 st;
        st.w = fc;
        fc += (int)fb[0];
        st.z = fc;
        fc += (int)fb[1];
        st.y = fc;
        fc += (int)fb[2];
        st.x = fc;
        *reinterpret_cast<int4*>(sh.fpos + own) = st;
        __syncthreads();
        if (sh.sq <= kBucketWork && total <= kArr) {
            unsigned long long* arr = cand;               // cand and outk: kArr entries
            each_key([&](unsigned long long c) {
                if ((uint32_t)(c >> 52) >= cut) {
                    const int slot = atomicAdd(&sh.fpos[fine(c)], 1);
                    if (slot < kArr) arr[slot] = c;
                }
            });
            __syncthreads();
            // bucket f: [fpos[f] - fcnt[f], fpos[f]); keys in earlier buckets
            // are larger, so a key's position is its bucket start plus the
            // number of larger keys in its bucket
            for (int j = tid; j < total; j += kSelThreads) {
                const unsigned long long c = arr[j];
                const int f = fine(c);
                const int e = min(sh.fpos[f], total);
                const int s0 = max(e - (int)sh.fcnt[f], 0);
                if (s0 >= K) continue;
                int rank = 0;
                for (int q = s0; q < e; ++q) rank += arr[q] > c ? 1 : 0;
                const int pos = s0 + rank;
                if (pos < K) sel_b[pos] = (int32_t)(~(uint32_t)c);
            }
            if (tid == 0) count[b] = K;
            return;
        }
    }

    // ---- collect: keys above the class go out directly, class members to cand
    each_key([&](unsigned long long c) {
        const unsigned long long top = c >> (64 - pbits), cls = prefix >> (64 - pbits);
        if (top > cls) {
            const int pos = atomicAdd(&sh.n_out, 1);
            if (pos < K) outk[pos] = c;
        } else if (top == cls) {
            const int pos = atomicAdd(&sh.n_cand, 1);
            if (pos < kCandCap) cand[pos] = c;
        }
    });
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

// Candidate pass for large n, grid (ceil(n / 4096), B): append every chunk that
// can be selected to the sequence's list -- keys above the threshold, or keys
// whose first digit is at or above the digit holding the K-th largest key (from
// the first-digit histogram). Each CTA finds that digit itself, while its score
// loads are in flight, and reserves room for its keys with one atomic. The
// count keeps growing past the capacity so the select kernel can tell an
// overflow.
__global__ void __launch_bounds__(kCollectThreads)
collect_kernel(const float* scores, int n, int mode, int K, float thresh,
               const uint32_t* hist_in, unsigned long long* __restrict__ cand,
               int* __restrict__ cand_cnt, int cap) {
    __shared__ int warp_buf[32];
    __shared__ int cut_s, base_s, total_s;
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.y, tid = threadIdx.x;
    const float* sc = scores + (size_t)b * n;
    const int i0 = blockIdx.x * (kCollectThreads * kCollectPer) + tid;
    float v[kCollectPer];
#pragma unroll
    for (int j = 0; j < kCollectPer; ++j) {
        const int i = i0 + j * kCollectThreads;
        v[j] = i < n ? __ldg(sc + i) : 0.f;
    }
    uint32_t kt = 0, cut = 0;
    if (mode == SRH_SELECT_THRESH) {
        kt = ordered_key(thresh);
    } else {
        // thread t owns bins 4095-16t .. 4080-16t (descending)
        const uint32_t* h = hist_in + (size_t)b * kHistBins;
        uint32_t hv[16];
        int local = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            hv[j] = __ldg(h + kHistBins - 1 - 16 * tid - j);
            local += (int)hv[j];
        }
        if (tid == 0) cut_s = 0;
        const int incl = block_inclusive_scan(local, warp_buf);
        if (tid == kCollectThreads - 1) total_s = incl;
        int cum = incl - local;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = (int)hv[j];
            if (c > 0 && cum < K && K <= cum + c) cut_s = kHistBins - 1 - 16 * tid - j;
            cum += c;
        }
        __syncthreads();
        // a histogram that does not count n keys is stale: keep every key, so
        // the list overflows and the select kernel works on all the scores
        cut = total_s == n ? (uint32_t)cut_s : 0u;
    }
    uint32_t keys[kCollectPer];
    unsigned pass = 0;
    int np = 0;
#pragma unroll
    for (int j = 0; j < kCollectPer; ++j) {
        const int i = i0 + j * kCollectThreads;
        keys[j] = ordered_key(v[j]);
        const bool p = i < n && (mode == SRH_SELECT_THRESH ? keys[j] > kt : (keys[j] >> 20) >= cut);
        pass |= (p ? 1u : 0u) << j;
        np += p ? 1 : 0;
    }
    const int incl = block_inclusive_scan(np, warp_buf);
    if (tid == kCollectThreads - 1) base_s = incl ? atomicAdd(&cand_cnt[b], incl) : 0;
    __syncthreads();
    int pos = base_s + incl - np;
    unsigned long long* out = cand + (size_t)b * cap;
#pragma unroll
    for (int j = 0; j < kCollectPer; ++j) {
        if (pass & (1u << j)) {
            if (pos < cap) out[pos] = composite(keys[j], (uint32_t)(i0 + j * kCollectThreads));
            ++pos;
        }
    }
}

}  // namespace

cudaError_t launch_select(const float* scores, int n, int B, int mode, int k, float thresh,
                          int clamp, int S, uint32_t* hist, int32_t* sel, int32_t* count,
                          cudaStream_t st, const unsigned long long* cand, int* cand_cnt, int cand_cap,
                          bool chained) {
    const size_t smem = sizeof(SelShared) + sizeof(unsigned long long) * kArr;
    return launch_k(select_kernel, dim3(B), dim3(kSelThreads), smem, st, chained, scores, n, mode, k, thresh, clamp, S,
                    hist, cand, cand_cnt, cand_cap, sel, count);
}

int select_cand_cap() { return kCandCap; }

cudaError_t set_select_attrs() {
    return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(SelShared) + sizeof(unsigned long long) * kArr));
}

cudaError_t launch_collect(const float* scores, int n, int B, int mode, int K, float thresh,
                           const uint32_t* hist, unsigned long long* cand, int* cand_cnt, int cap,
                           cudaStream_t st, bool clear_count, bool chained) {
    if (clear_count) {
        const cudaError_t e = cudaMemsetAsync(cand_cnt, 0, sizeof(int) * B, st);
        if (e != cudaSuccess) return e;
    }
    const int per_cta = kCollectThreads * kCollectPer;
    const int bx = (n + per_cta - 1) / per_cta;
    return launch_k(collect_kernel, dim3((unsigned)bx, (unsigned)B), dim3(kCollectThreads), 0, st, chained, scores,
                    n, mode, K, thresh, hist, cand, cand_cnt, cap);
}

}  // namespace srh
