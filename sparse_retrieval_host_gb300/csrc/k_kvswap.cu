// K-lru + K-gather: the KV_SWAP Swap-in flow on the device.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section "KV_SWAP 实现细节":
// GgufKvSwapLayerState keeps, per sparse layer, the GPU slot of each logical
// chunk, the chunk of each slot and an LRU list of slots (front = most recently
// used). gguf_kv_swap_in_selected walks the selected logical ids in order: a hit
// moves its slot to the front; a miss pops the back slot, copies
// h_compressed_kv[logical] into it (H2D) and the slot becomes the front; the
// indices are then rewritten to physical = window + slot for the attention.
//
// Here that state lives in device memory and one CTA resolves one
// (layer, sequence) with no host round trip:
//   * slot_of[c]        chunk -> slot (-1 if absent), a direct map over the cap;
//   * slot_logical[s]   slot -> chunk (-1 if free);
//   * lru_order[q]      slots from least (q = 0) to most recently used.
// The walk is sequential on the pages, so a miss may pop the slot of a chunk
// that is selected later in the same list. The kernel first assumes that never
// happens (hits are the resident chunks; the i-th miss takes the i-th non-hit
// slot in LRU order), checks that assumption exactly in parallel, and only
// when it fails replays the list in order in shared memory, visiting just the
// misses (one warp: runs of up to 32 misses that pop unlisted slots at once,
// every other miss one at a time). Both paths produce the state and outputs of
// the sequential list.
//
// The miss gather reads the mapped pinned pool directly (zero-copy over the
// host link): each warp moves 2 KiB chunks with 16-byte loads, up to three
// chunks in flight, only for the layers that swap. A staged row is kept
// as fp16 (1 KiB): the attention rounds every row to fp16 for its tensor-core
// products anyway, so staging the rounded row gives the same results from half
// the bytes. A pool value beyond fp16's finite range (65504) sets kErrRange.
#include <climits>

#include "srh_internal.cuh"

namespace srh {
namespace {

constexpr int kLruThreads = 1024;
// Slot maps of at most this many chunks (32 KB) are prefetched whole; a larger
// map would cost far more DRAM reads than its 512 or so lookups (at 128K x 32
// sequences, 80 MB a step).
constexpr long long kPrefetchCap = 1 << 13;
constexpr uintptr_t kPrefetchChunk = 1 << 14;  // bytes per bulk prefetch

// Inclusive block scan of one int per thread; *total receives the block total.
// Two barriers; warp_buf must not be written again before the caller's next
// barrier.
__device__ __forceinline__ int block_scan_incl(int v, int* warp_buf, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_buf[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? warp_buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        warp_buf[lane] = w;
    }
    __syncthreads();
    *total = warp_buf[nwarps - 1];
    return v + (warp > 0 ? warp_buf[warp - 1] : 0);
}

// Exclusive block scan of one int per thread with a single barrier
// (blockDim.x == kLruThreads, 32 warps): each warp adds up the totals of the
// warps before it itself. `total` receives the block's sum. warp_buf must not
// be written again before the caller's next barrier.
__device__ __forceinline__ int block_scan_excl_1bar(int v, int* warp_buf, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
    }
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    const int w = warp_buf[lane];
    total = __reduce_add_sync(0xffffffffu, w);
    return x - v + __reduce_add_sync(0xffffffffu, lane < warp ? w : 0);
}

// In-place exclusive scan of a[0..len) in shared memory; returns the total.
// Three barriers; on return every thread sees the whole scanned array.
__device__ int block_scan_excl_array(int* a, int len, int* warp_buf) {
    const int per = (len + blockDim.x - 1) / blockDim.x;
    const int beg = threadIdx.x * per;
    const int end = min(beg + per, len);
    int local = 0;
    for (int i = beg; i < end; ++i) local += a[i];
    int total;
    const int incl = block_scan_incl(local, warp_buf, &total);
    int run = incl - local;
    for (int i = beg; i < end; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ void load_row(float4 (&v)[4], const float* __restrict__ src, int lane) {
    const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = s[k * 32 + lane];
}
__device__ __forceinline__ void store_row(float* __restrict__ dst, const float4 (&v)[4], int lane) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int k = 0; k < 4; ++k) d[k * 32 + lane] = v[k];
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// The row as fp16 (round to nearest even) into a staging row; a value beyond
// fp16's finite range sets kErrRange.
__device__ __forceinline__ void store_row_h(uint16_t* __restrict__ dst, const float4 (&v)[4], int lane,
                                            uint32_t* __restrict__ err) {
    uint2* d = reinterpret_cast<uint2*>(dst);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
        d[k * 32 + lane] = make_uint2(pack_h2(v[k].x, v[k].y), pack_h2(v[k].z, v[k].w));
    }
    if (__any_sync(0xffffffffu, !(amax <= 65504.f)) && lane == 0) atomicOr(err, kErrRange);
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

struct LruShared {
    int warp_buf[32];
    int nmiss;
    int conflict;
    unsigned version;   // the state's version read before the dependency wait
    int stale;          // it changed by the time the wait returned: state read again
};

constexpr int kLruPer = kMaxGpuChunks / kLruThreads;   // LRU entries per thread

// A swapped (layer, sequence)'s state into registers (thread t: entries
// t + k * kLruThreads of the LRU order and slot contents) and, when it fits,
// its slot map into shared memory.
__device__ __forceinline__ void lru_read_state(const AdaptState* as, const int* lru, const int* slot_logical,
                                               const int* slot_of, int* smap, bool mirror, long long cap, int G,
                                               int& g0, int& g, int (&lruv)[kLruPer], int (&slv)[kLruPer]) {
    g0 = as->g;
    g = as->g_next;
#pragma unroll
    for (int k = 0; k < kLruPer; ++k) {
        const int q = threadIdx.x + k * kLruThreads;
        lruv[k] = q < G ? lru[q] : 0;
        slv[k] = q < G ? slot_logical[q] : -1;
    }
    if (mirror)
        for (long long c = threadIdx.x; c < cap; c += blockDim.x) smap[c] = slot_of[c];
}
__device__ __forceinline__ void lru_keep_contents(int* sls, const int (&slv)[kLruPer], int G) {
#pragma unroll
    for (int k = 0; k < kLruPer; ++k) {
        const int q = threadIdx.x + k * kLruThreads;
        if (q < G) sls[q] = slv[k];
    }
}

__global__ void __launch_bounds__(kLruThreads)
lru_kernel(const LayerDev* __restrict__ layers, int l0, int B, int G, int S, int src_ratio, int dedup_tbl, int mirror_tbl,
           const int32_t* sel, const int32_t* count,
           int32_t* __restrict__ phys, int32_t* __restrict__ count_l, int2* __restrict__ miss,
           int* __restrict__ miss_count, unsigned long long* __restrict__ stats,
           uint32_t* __restrict__ err, AdaptParams ap) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    LruShared& sh = *reinterpret_cast<LruShared*>(smem_raw);
    int* r = reinterpret_cast<int*>(smem_raw + sizeof(LruShared));  // [S] layer list
    int* init_slot = r + S;      // [S]
    int* assign = init_slot + S; // [S]
    int* mr = assign + S;        // [S] miss rank / keep flags
    int* tk = mr + S;            // [S] position of the k-th miss
    int* is_miss = tk + S;       // [S]
    int* queue = is_miss + S;    // [G] lru order
    int* qpos = queue + G;       // [G]
    int* hit_time = qpos + G;    // [G]
    int* nh = hit_time + G;      // [G]
    int* victim = nh + G;        // [G]
    int* flag = victim + G;      // [G]
    int* sls = flag + G;         // [G] chunk held by each slot before this step
    int* first = sls + G;        // [dedup_tbl]: first list position of each mapped chunk
    int* smap = first + dedup_tbl;   // [mirror_tbl]: the slot map, when it fits

    const int tid = threadIdx.x;
    const int l = l0 + blockIdx.x / B;
    const int b = blockIdx.x % B;
    const LayerDev ld = layers[l];     // written once, at creation
    const long long cap = ld.cap;
    const size_t lb = (size_t)l * B + b;
    const int32_t* sel_b = sel + (size_t)b * S;
    int* lru = ld.swap ? ld.lru_order + (size_t)b * G : nullptr;   // swap layers only
    AdaptState* as = ld.swap ? ld.adapt + b : nullptr;
    pdl_trigger();                     // the gather kernel may launch (it waits for this one)
    // The layer's own state (capacity, LRU order, slot contents and, when it
    // fits in shared memory, the whole slot map) is written only by resolve
    // kernels of this (layer, sequence). It is read before the dependency wait,
    // while the earlier kernels finish, after a read of the state's version;
    // every resolve raises the version (release) after its last write. A
    // resolve still running at the first read (one chained right before this
    // one) has raised it by the time the wait returns, and the state is then
    // read again. host_ready is read only after the wait (for misses).
    for (int q = tid; q < G; q += blockDim.x) hit_time[q] = INT_MAX;
    const bool mirror = ld.swap && cap <= mirror_tbl;
    int* slot_of = ld.swap ? ld.slot_of + (size_t)b * cap : nullptr;
    int* slot_logical = ld.swap ? ld.slot_logical + (size_t)b * G : nullptr;
    if (ld.swap && tid == 0) sh.version = ld_acquire_u32(&as->version);
    if (ld.swap && tid < 2 && cap <= kPrefetchCap) {
        // L2 prefetches of the tables read after the wait: the host_ready bits
        // (for misses) and a slot map not copied into shared memory
        const void* base = nullptr;
        long long bytes = 0;
        if (tid == 0) {
            base = ld.host_ready + (size_t)b * cap;
            bytes = cap;
        } else if (!mirror) {
            base = slot_of;
            bytes = 4LL * cap;
        }
        // whole 16-byte units inside the range, from its first 16-byte boundary
        const uintptr_t a0 = ((uintptr_t)base + 15) & ~(uintptr_t)15;
        const uintptr_t a1 = ((uintptr_t)base + (uintptr_t)bytes) & ~(uintptr_t)15;
        for (uintptr_t a = a0; base && a < a1; a += kPrefetchChunk) {
            const uint32_t len = (uint32_t)min((uintptr_t)kPrefetchChunk, a1 - a);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(a), "r"(len) : "memory");
        }
    }
    __syncthreads();   // orders the version's acquire before every thread's state reads

    // Thread t holds entries t + k * 1024 of the selection row, the LRU order
    // and the slot contents.
    constexpr int kPer = kLruPer;
    static_assert(kMaxSelect <= kMaxGpuChunks, "selection entries per thread");
    int selv[kPer], lruv[kPer], slv[kPer];
    int g0 = G, g = G;
    if (ld.swap) lru_read_state(as, lru, slot_logical, slot_of, smap, mirror, cap, G, g0, g, lruv, slv);
    pdl_wait();                        // the selection comes from earlier kernels

    // one round of loads: the count and the whole selection row (entries past
    // the count are ignored), and the state's version again
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int p = tid + k * kLruThreads;
        selv[k] = p < S ? sel_b[p] : 0;
    }
    int m0 = count[b];
    if (ld.swap) {
        if (tid == 0) sh.stale = ld_acquire_u32(&as->version) != sh.version;
        lru_keep_contents(sls, slv, G);   // visible to every thread after the barrier of step 1
    }

    // ---- 1. the layer's ordered chunk list: c -> floor(c * src_ratio / ratio), first kept
    if (m0 < 0 || m0 > S) {
        if (tid == 0) atomicOr(err, kErrBounds);
        m0 = m0 < 0 ? 0 : S;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int p = tid + k * kLruThreads;
        if (p < m0) {
            const long long c = selv[k];
            long long v = (c * src_ratio) / ld.ratio;
            if (c < 0 || v >= cap) {
                // out-of-range id: flagged, then clamped so every access stays in bounds
                atomicOr(err, kErrBounds);
                v = 0;
            }
            r[p] = (int)v;
        }
    }
    __syncthreads();
    int m;
    if (ld.ratio == src_ratio) {
        m = m0;
    } else {
        if (cap <= dedup_tbl) {
            // keep the first position of each mapped chunk: min position per chunk
            for (int v = tid; v < cap; v += blockDim.x) first[v] = INT_MAX;
            __syncthreads();
            for (int p = tid; p < m0; p += blockDim.x) atomicMin(&first[r[p]], p);
            __syncthreads();
            for (int p = tid; p < m0; p += blockDim.x) mr[p] = first[r[p]] == p ? 1 : 0;
        } else {
            for (int p = tid; p < m0; p += blockDim.x) {
                const int v = r[p];
                int keep = 1;
                for (int q = 0; q < p; ++q)
                    if (r[q] == v) {
                        keep = 0;
                        break;
                    }
                mr[p] = keep;
            }
        }
        __syncthreads();
        // stable compaction (read all, scan, then write)
        for (int p = tid; p < m0; p += blockDim.x) tk[p] = mr[p];
        __syncthreads();
        m = block_scan_excl_array(mr, m0, sh.warp_buf);
        for (int p = tid; p < m0; p += blockDim.x) is_miss[p] = r[p];
        __syncthreads();
        for (int p = tid; p < m0; p += blockDim.x)
            if (tk[p]) r[mr[p]] = is_miss[p];
        __syncthreads();
    }

    if (ld.swap && sh.stale) {
        // a resolve of this state ran past the first read: read it again
        __syncthreads();
        lru_read_state(as, lru, slot_logical, slot_of, smap, mirror, cap, G, g0, g, lruv, slv);
        lru_keep_contents(sls, slv, G);
        __syncthreads();
    }

    int32_t* phys_lb = phys + lb * S;
    if (!ld.swap) {
        // swap disabled: every chunk is resident at its own row
        for (int p = tid; p < m; p += blockDim.x) {
            const int c = r[p];
            if (!ld.host_ready[(size_t)b * cap + c]) atomicOr(err, kErrNotStored);
            phys_lb[p] = kWindow + c;
        }
        if (tid == 0) {
            count_l[lb] = m;
            miss_count[lb] = 0;
            atomicAdd(&stats[kStatSelected], (unsigned long long)m);
        }
        return;
    }

    // ---- 2a. slots in use: the last step's range g0, resized to g when the
    // hit-rate policy (or the host) asked for it. No staged row moves.
    if (g0 < 1 || g0 > G || g < 1 || g > G) {
        if (tid == 0) atomicOr(err, kErrBounds);
        g0 = (g0 < 1 || g0 > G) ? G : g0;
        g = (g < 1 || g > G) ? g0 : g;
    }
    if (g > g0) {
        // the new slots, empty, go to the least recently used end, lowest first
        const int add = g - g0;
        for (int q = tid; q < add; q += blockDim.x) {
            const int s = g0 + q;
            const int c = sls[s];
            if (c >= 0 && c < cap && (mirror ? smap[c] : slot_of[c]) == s) {
                slot_of[c] = -1;
                if (mirror) smap[c] = -1;
            }
            slot_logical[s] = -1;
            sls[s] = -1;
            queue[q] = s;
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int q = tid + k * kLruThreads;
            if (q < g0) {
                int s = lruv[k];
                if (s < 0 || s >= g0) {
                    atomicOr(err, kErrBounds);
                    s = q;
                }
                queue[add + q] = s;
            }
        }
        __syncthreads();
    } else if (g < g0) {
        // keep the slots below g in their order; the others forget their chunks
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int q = tid + k * kLruThreads;
            if (q < g0) {
                int s = lruv[k];
                if (s < 0 || s >= g0) {
                    atomicOr(err, kErrBounds);
                    s = q;
                }
                victim[q] = s;
                nh[q] = s < g ? 1 : 0;
            }
        }
        __syncthreads();
        block_scan_excl_array(nh, g0, sh.warp_buf);
        for (int q = tid; q < g0; q += blockDim.x) {
            const int s = victim[q];
            if (s < g) {
                queue[nh[q]] = s;
            } else {
                const int c = sls[s];
                if (c >= 0 && c < cap && (mirror ? smap[c] : slot_of[c]) == s) {
                    slot_of[c] = -1;
                    if (mirror) smap[c] = -1;
                }
                slot_logical[s] = -1;
            }
        }
        __syncthreads();
    } else {
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int q = tid + k * kLruThreads;
            if (q < g) {
                int s = lruv[k];
                if (s < 0 || s >= g) {
                    atomicOr(err, kErrBounds);
                    s = q;
                }
                queue[q] = s;
            }
        }
    }
    // a swapped layer stages at most g chunks per step (reachable with
    // allow_topk_reduction or a small adaptive range): it keeps the first g
    if (m > g) m = g;

    // ---- 2b. resident lookups (hit_time was set to INT_MAX before the wait)
    for (int p = tid; p < m; p += blockDim.x) {
        const int c = r[p];
        int s = mirror ? smap[c] : slot_of[c];
        if (s >= g) {
            atomicOr(err, kErrBounds);
            s = -1;
        }
        init_slot[p] = s;
        if (s >= 0) hit_time[s] = p;
    }
    for (int q = tid; q < g; q += blockDim.x) qpos[queue[q]] = q;
    if (tid == 0) sh.conflict = 0;
    __syncthreads();

    // ---- 3. optimistic assignment: hits keep their slots, the i-th miss takes
    // the i-th non-hit slot in LRU order. One scan ranks both: the non-hit slots
    // (high 16 bits) and the misses (low 16 bits); both counts are <= 4096.
    const int nk = max(g, m);
    int nmiss0;
    if (nk <= kLruThreads) {
        // one entry per thread: one scan with a single barrier, ranks used in place
        const bool free_q = tid < g && hit_time[queue[tid]] == INT_MAX;
        const bool miss_p = tid < m && init_slot[tid] < 0;
        const int v = (free_q ? (1 << 16) : 0) | (miss_p ? 1 : 0);
        int both;
        const int ex = block_scan_excl_1bar(v, sh.warp_buf, both);
        nmiss0 = both & 0xffff;
        if (tid < nk) nh[tid] = ex;
        if (free_q) victim[ex >> 16] = queue[tid];
        if (miss_p) tk[ex & 0xffff] = tid;
    } else {
        for (int i = tid; i < nk; i += blockDim.x)
            nh[i] = ((i < g && hit_time[queue[i]] == INT_MAX) ? (1 << 16) : 0) | ((i < m && init_slot[i] < 0) ? 1 : 0);
        __syncthreads();
        const int both = block_scan_excl_array(nh, nk, sh.warp_buf);
        nmiss0 = both & 0xffff;
        for (int q = tid; q < g; q += blockDim.x)
            if (hit_time[queue[q]] == INT_MAX) victim[nh[q] >> 16] = queue[q];
        for (int p = tid; p < m; p += blockDim.x)
            if (init_slot[p] < 0) tk[nh[p] & 0xffff] = p;
    }
    __syncthreads();
    // a hit slot j lying before the kj-th non-hit slot is reached by that pop if
    // the pop happens before j is touched: the sequential list would take j
    for (int p = tid; p < m; p += blockDim.x) {
        const int j = init_slot[p];
        if (j >= 0) {
            const int kj = nh[qpos[j]] >> 16;
            if (kj < nmiss0 && tk[kj] < p) sh.conflict = 1;
        }
    }
    __syncthreads();
    int nmiss;
    int2* miss_lb = miss + lb * S;
    if (!sh.conflict) {
        nmiss = nmiss0;
        // ---- 4+5 (no conflict). The victims are the first nmiss non-hit slots,
        // so the untouched slots are the other non-hit ones, in their old order;
        // the touched slots follow by list position. A victim's old chunk is not
        // listed (it would have been a hit), so clearing it never meets a new entry.
        for (int q = tid; q < g; q += blockDim.x) {
            const int s = queue[q];
            const int k = nh[q] >> 16;
            if (hit_time[s] == INT_MAX && k >= nmiss) lru[k - nmiss] = s;
        }
        for (int p = tid; p < m; p += blockDim.x) {
            int s = init_slot[p];
            if (s < 0) {
                const int i = nh[p] & 0xffff;
                s = victim[i];
                const int c = r[p];
                const int old = sls[s];
                if (old >= 0 && old < cap) slot_of[old] = -1;
                slot_of[c] = s;
                slot_logical[s] = c;
                miss_lb[i] = make_int2(c, s);
                if (!ld.host_ready[(size_t)b * cap + c]) atomicOr(err, kErrNotStored);
            }
            phys_lb[p] = kWindow + s;
            lru[g - m + p] = s;
        }
    } else {
        // Replay the list in order, visiting only the misses (warp 0). The LRU
        // pointer skips the slot at queue position q exactly when that slot's
        // listed position T[q] comes before the current miss (it was hit
        // already); otherwise it pops it, and a popped slot's later listed
        // position T[q] becomes a miss too. The next miss is the smaller of the
        // next initial miss and the earliest pending induced one (kept sorted
        // in mr[hs..he)). A run of initial misses that all come before the
        // earliest pending one, at queue positions whose slots are not listed
        // (T = INT_MAX), pops those positions in order: up to 32 of them are
        // placed at once; every other miss is taken one at a time. All lanes
        // hold the same state; lane 0 writes the pending list.
        for (int q = tid; q < g; q += blockDim.x) flag[q] = hit_time[queue[q]];   // T[q]
        for (int p = tid; p < m; p += blockDim.x) {
            assign[p] = init_slot[p];
            is_miss[p] = 0;
        }
        __syncthreads();
        if (tid < 32) {
            const int lane = tid;
            int i0 = 0, hs = 0, he = 0, nm = 0, ptr = 0;
            int hmin = INT_MAX;   // earliest pending induced miss
            for (;;) {
                // a run of misses i0 + j popping positions ptr + j (j < 32)
                const int q = ptr + lane;
                const int pj = i0 + lane < nmiss0 ? tk[i0 + lane] : INT_MAX;
                const bool ok = q < g && pj < hmin && flag[q] == INT_MAX;
                const unsigned run = __ballot_sync(0xffffffffu, ok);
                const int k = run == 0xffffffffu ? 32 : __ffs(~run) - 1;
                if (k > 0) {
                    if (lane < k) {
                        assign[pj] = queue[q];
                        is_miss[pj] = 1;
                    }
                    nm += k;
                    ptr += k;
                    i0 += k;
                    continue;
                }
                // one miss: the next initial or pending one
                const int ni = i0 < nmiss0 ? tk[i0] : INT_MAX;
                int P;
                if (ni < hmin) {
                    P = ni;
                    ++i0;
                } else if (hmin != INT_MAX) {
                    P = hmin;
                    ++hs;
                    hmin = hs < he ? mr[hs] : INT_MAX;
                } else {
                    break;
                }
                while (ptr < g && flag[ptr] < P) ++ptr;   // hit before P: skipped
                if (ptr >= g) {   // no slot left: unreachable (at most g misses among g slots)
                    if (lane == 0) atomicOr(err, kErrBounds);
                    break;
                }
                const int tv = flag[ptr];
                if (lane == 0) {
                    assign[P] = queue[ptr];
                    is_miss[P] = 1;
                }
                ++nm;
                ++ptr;
                if (tv != INT_MAX) {
                    // the popped slot's own listed position (> P) misses too
                    if (lane == 0) {
                        int j = he;
                        while (j > hs && mr[j - 1] > tv) {
                            mr[j] = mr[j - 1];
                            --j;
                        }
                        mr[j] = tv;
                    }
                    ++he;
                    __syncwarp();
                    hmin = mr[hs];
                }
            }
            if (lane == 0) sh.nmiss = nm;
        }
        __syncthreads();
        nmiss = sh.nmiss;
        for (int p = tid; p < m; p += blockDim.x) mr[p] = is_miss[p];
        __syncthreads();
        block_scan_excl_array(mr, m, sh.warp_buf);

        // ---- 4. new LRU order: untouched slots in old order, then touched ones by position
        for (int q = tid; q < g; q += blockDim.x) flag[q] = 0;
        __syncthreads();
        for (int p = tid; p < m; p += blockDim.x) flag[assign[p]] = 1;
        __syncthreads();
        for (int q = tid; q < g; q += blockDim.x) nh[q] = flag[queue[q]] ? 0 : 1;
        __syncthreads();
        block_scan_excl_array(nh, g, sh.warp_buf);
        for (int q = tid; q < g; q += blockDim.x)
            if (!flag[queue[q]]) lru[nh[q]] = queue[q];
        for (int p = tid; p < m; p += blockDim.x) lru[g - m + p] = assign[p];

        // ---- 5. slot maps: clear evicted chunks first, then record the new ones
        for (int p = tid; p < m; p += blockDim.x)
            if (is_miss[p]) {
                const int old = sls[assign[p]];
                if (old >= 0 && old < cap) slot_of[old] = -1;
            }
        __syncthreads();
        for (int p = tid; p < m; p += blockDim.x) {
            const int s = assign[p];
            phys_lb[p] = kWindow + s;
            if (is_miss[p]) {
                const int c = r[p];
                slot_of[c] = s;
                slot_logical[s] = c;
                miss_lb[mr[p]] = make_int2(c, s);
                if (!ld.host_ready[(size_t)b * cap + c]) atomicOr(err, kErrNotStored);
            }
        }
    }
    __syncthreads();   // every thread's state writes precede the version's release below
    if (tid == 0) {
        count_l[lb] = m;
        miss_count[lb] = nmiss;
        atomicAdd(&stats[kStatHits], (unsigned long long)(m - nmiss));
        atomicAdd(&stats[kStatMisses], (unsigned long long)nmiss);
        atomicAdd(&stats[kStatSelected], (unsigned long long)m);
        // ---- 6. hit-rate window of the adaptive policy
        as->g = g;
        if (ap.on) {
            int en = as->ep_steps + 1;
            long long eh = as->ep_hits + (m - nmiss);
            long long es = as->ep_sel + m;
            int gn = g;
            if (en >= ap.epoch) {
                if (eh * 1000 < (long long)ap.lo_pm * es)
                    gn = min(ap.g_max, g + ap.delta);
                else if (eh * 1000 > (long long)ap.hi_pm * es)
                    gn = max(ap.g_min, g - ap.delta);
                en = 0;
                eh = es = 0;
            }
            as->ep_steps = en;
            as->ep_hits = eh;
            as->ep_sel = es;
            as->g_next = gn;
        } else {
            as->g_next = g;
        }
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(&as->version) : "memory");
    }
}

constexpr int kGatherWarps = 8;
constexpr int kGatherRows = 3;   // rows in flight per gather warp

// at most 85 registers: three gather CTAs per SM, so that the whole grid is
// resident beside the resolve CTAs and the attention behind it can launch
__global__ void __launch_bounds__(kGatherWarps * 32, 3)
gather_kernel(const LayerDev* __restrict__ layers, const int* __restrict__ swap_layers, int B, int G, int S,
              const int2* miss, const int* miss_count,
              uint16_t* __restrict__ staging, uint32_t* __restrict__ err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    // blockIdx.y: (swapped layer, sequence); the list is written once, at creation
    const int l = swap_layers[blockIdx.y / B], b = (int)(blockIdx.y % B);
    const size_t lb = (size_t)l * B + b;
    pdl_wait();                        // the miss lists come from the resolve kernel
    const int nm = miss_count[lb];
    const LayerDev ld = layers[l];
    const int2* ml = miss + lb * S;
    // up to kGatherRows rows per warp in flight: their loads are all issued
    // before the first store (a host row's first read may wait on the
    // translation of its page)
    const int step = gridDim.x * kGatherWarps;
    for (int i0 = blockIdx.x * kGatherWarps + warp; i0 < nm; i0 += kGatherRows * step) {
        int2 e[kGatherRows];
        bool ok[kGatherRows];
#pragma unroll
        for (int r = 0; r < kGatherRows; ++r) {
            const int i = i0 + r * step;
            e[r] = i < nm ? ml[i] : make_int2(-1, -1);
            ok[r] = i < nm && e[r].x >= 0 && e[r].x < ld.cap && e[r].y >= 0 && e[r].y < G;
            if (i < nm && !ok[r] && lane == 0) atomicOr(err, kErrBounds);
        }
        float4 v[kGatherRows][4];
#pragma unroll
        for (int r = 0; r < kGatherRows; ++r)
            if (ok[r]) load_row(v[r], ld.pool + ((size_t)b * ld.cap + e[r].x) * kKvDim, lane);
#pragma unroll
        for (int r = 0; r < kGatherRows; ++r)
            if (ok[r]) store_row_h(staging + (((size_t)l * B + b) * G + e[r].y) * kKvDim, v[r], lane, err);
    }
}

__global__ void __launch_bounds__(kGatherWarps * 32)
resident_fill_kernel(const float* __restrict__ pool, const uint8_t* __restrict__ ready,
                     long long cap, int layer, int B, int G, uint16_t* __restrict__ staging,
                     uint32_t* __restrict__ err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    for (long long c = (long long)blockIdx.x * kGatherWarps + warp; c < cap;
         c += (long long)gridDim.x * kGatherWarps) {
        if (!ready[(size_t)b * cap + c]) continue;
        float4 v[4];
        load_row(v, pool + ((size_t)b * cap + c) * kKvDim, lane);
        store_row_h(staging + (((size_t)layer * B + b) * G + c) * kKvDim, v, lane, err);
    }
}


// Store flow: rows [n][512] of chunks c0.. of (layer, seq) go to the pinned pool
// (zero-copy writes over the host link), host_ready is set, and the staging
// stays consistent: a staged chunk keeps its slot with the new row; a layer
// that does not swap gets row c. One warp per row.
__global__ void __launch_bounds__(kGatherWarps * 32)
store_kernel(const LayerDev* __restrict__ layers, int l, int B, int G, int seq, long long c0, int n,
             const float* __restrict__ rows, uint16_t* __restrict__ staging, uint32_t* __restrict__ err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const LayerDev ld = layers[l];
    float* pool = const_cast<float*>(ld.pool) + (size_t)seq * ld.cap * kKvDim;
    uint16_t* stg = staging ? staging + ((size_t)l * B + seq) * G * kKvDim : nullptr;
    for (int i = blockIdx.x * kGatherWarps + warp; i < n; i += gridDim.x * kGatherWarps) {
        const long long c = c0 + i;
        if (c < 0 || c >= ld.cap) {
            if (lane == 0) atomicOr(err, kErrBounds);
            continue;
        }
        float4 v[4];
        load_row(v, rows + (size_t)i * kKvDim, lane);
        store_row(pool + c * kKvDim, v, lane);
        if (stg) {
            long long row = -1;
            if (ld.swap) {
                const int s = ld.slot_of[(size_t)seq * ld.cap + c];
                if (s >= 0 && s < G) row = s;
            } else if (c < G) {
                row = c;
            }
            if (row >= 0) store_row_h(stg + row * kKvDim, v, lane, err);
        }
        __syncwarp();
        if (lane == 0) ld.host_ready[(size_t)seq * ld.cap + c] = 1;
    }
    __threadfence_system();   // the pool rows are host memory read by later kernels
}

// One read per 4 KiB of a pool range, so the device side of the host page
// mappings is set up before the first miss gathers need them (random rows of
// pages the GPU has never read are several times slower to fetch).
__global__ void touch_kernel(const float* __restrict__ p, long long n_pages, uint32_t* __restrict__ sink) {
    uint32_t acc = 0;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_pages;
         i += (long long)gridDim.x * blockDim.x)
        acc ^= __float_as_uint(p[i * 1024]);
    if (acc == 0x9e3779b9u) *sink = acc;   // keeps the loads; practically never taken
}
}  // namespace

cudaError_t set_lru_attrs() {
    return cudaFuncSetAttribute(lru_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

size_t lru_smem_bytes(int S, int G) {
    return sizeof(LruShared) + sizeof(int) * (6 * (size_t)S + 7 * (size_t)G);
}

cudaError_t launch_lru(const LayerDev* layers, int l0, int nl, int B, int G, int S, int src_ratio,
                       long long max_dedup_cap, long long max_mirror_cap, const int32_t* sel, const int32_t* count,
                       int32_t* phys, int32_t* count_l, int2* miss, int* miss_count,
                       unsigned long long* stats, uint32_t* err, AdaptParams ap, cudaStream_t st,
                       bool chained) {
    // a shared-memory table of first positions for layers whose ratio differs from
    // src_ratio, when it fits; otherwise those layers fall back to pairwise checks
    int tbl = 0;
    if (max_dedup_cap > 0 &&
        lru_smem_bytes(S, G) + sizeof(int) * (size_t)max_dedup_cap <= 227 * 1024)
        tbl = (int)max_dedup_cap;
    // a shared-memory copy of the slot map for swapped layers of at most
    // kLruMirrorMax chunks, when it fits beside the rest and the launch is
    // chained (the copy then overlaps the earlier kernels; unchained it would
    // only add its reads ahead of the lookups)
    int mir = 0;
    if (chained && max_mirror_cap > 0 && max_mirror_cap <= kLruMirrorMax &&
        lru_smem_bytes(S, G) + sizeof(int) * ((size_t)tbl + (size_t)max_mirror_cap) <= 227 * 1024)
        mir = (int)max_mirror_cap;
    const size_t smem = lru_smem_bytes(S, G) + sizeof(int) * ((size_t)tbl + (size_t)mir);   // <= 227 KB
    return launch_k(lru_kernel, dim3(nl * B), dim3(kLruThreads), smem, st, chained, layers, l0, B, G, S, src_ratio,
                    tbl, mir, sel, count, phys, count_l, miss, miss_count, stats, err, ap);
}

cudaError_t launch_gather(const LayerDev* layers, const int* swap_layers, int n_sw, int nl_call, int B, int G, int S,
                          const int2* miss, const int* miss_count, uint16_t* staging, uint32_t* err,
                          int sm_count, cudaStream_t st, bool chained) {
    if (n_sw <= 0) return cudaSuccess;
    // CTAs per (layer, sequence) as if every layer of the call swapped: a
    // lookahead boundary's misses keep that many rows in flight per layer
    int bx = (4 * sm_count + nl_call * B - 1) / (nl_call * B);
    if (bx < 1) bx = 1;
    if (bx > 64) bx = 64;
    return launch_k(gather_kernel, dim3(bx, n_sw * B), dim3(kGatherWarps * 32), 0, st, chained, layers, swap_layers, B,
                    G, S, miss, miss_count, staging, err);
}

cudaError_t launch_touch(const float* p, long long n_floats, uint32_t* sink, int sm_count, cudaStream_t st) {
    const long long pages = (n_floats + 1023) / 1024;
    if (pages <= 0) return cudaSuccess;
    long long bx = (pages + 255) / 256;
    if (bx > 8LL * sm_count) bx = 8LL * sm_count;
    touch_kernel<<<(unsigned)bx, 256, 0, st>>>(p, pages, sink);
    return cudaGetLastError();
}

cudaError_t launch_store(const LayerDev* layers, int l, int B, int G, int seq, long long c0, int n,
                         const float* rows, uint16_t* staging, uint32_t* err, cudaStream_t st) {
    int bx = (n + kGatherWarps - 1) / kGatherWarps;
    if (bx > 1024) bx = 1024;
    store_kernel<<<bx, kGatherWarps * 32, 0, st>>>(layers, l, B, G, seq, c0, n, rows, staging, err);
    return cudaGetLastError();
}

cudaError_t launch_resident_fill(const float* pool_dev, const uint8_t* ready, long long cap,
                                 int layer, int B, int G, uint16_t* staging, uint32_t* err, cudaStream_t st) {
    long long bx = (cap + kGatherWarps - 1) / kGatherWarps;
    if (bx > 256) bx = 256;
    if (bx < 1) bx = 1;
    resident_fill_kernel<<<dim3((unsigned)bx, B), kGatherWarps * 32, 0, st>>>(pool_dev, ready, cap,
                                                                              layer, B, G, staging, err);
    return cudaGetLastError();
}

}  // namespace srh
