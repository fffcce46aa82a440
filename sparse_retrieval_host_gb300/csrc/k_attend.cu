// K-attend + K-combine: split-K flash-decode over the window and the staged rows.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 技术细节 / 架构概览,
// per-layer box step 3 (indexed_cached_attention over window + selected) and
// "Memory Layout" (window KV [128, kv_dim] plus staging slots [gpu_chunks,
// kv_dim], one fp32 latent row per entry). Every head attends over the same rows
// (MQA over the latent, K = V = row):
//   o_h = sum_j softmax_j(<q_h, e_j> / sqrt(512)) e_j.
//
// Work: the rows of one (layer, sequence) -- 128 window rows, then the layer's
// staged rows in selection order -- are cut into fixed splits of `split_rows`;
// one CTA (8 warps) runs one split for all heads. Rows stream through a
// two-stage cp.async ring of 32-row tiles (16-byte copies into an XOR-swizzled
// layout); the query block sits in shared memory as bf16. Per tile:
//   S = Q E^T     (tf32 m16n8k8 MMAs, fp32 accumulate; q in bf16 is exact in tf32),
//   online softmax in base 2 with a running max per head,
//   O = O * alpha + P E  (tf32 MMAs; O stays in registers, each warp owns 64
//   latent columns for all heads).
// A split writes (m, l, O) partials; the last CTA of a (layer, sequence) to
// finish (atomic ticket, no waiting) merges the partials in split order. The
// split layout depends only on the row count, so identical rows give identical
// bits whatever slots they occupy.
#include <cmath>

#include "srh_internal.cuh"

namespace srh {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = kAttnTile;   // 32 rows
constexpr int kPStride = 40;       // floats per P row (bank-conflict-free fragment loads)
constexpr int kMaxSplits = (kWindow + kMaxSelect + kTile - 1) / kTile;

template <int H>
struct __align__(16) AttnSmem {
    uint16_t q[H * kKvDim];              // bf16, 16-byte chunk c of row r at c ^ (r & 7)
    float e[2][kTile * kKvDim];          // fp32, 16-byte chunk c of row r at c ^ (r & 7)
    float p[H * kPStride];               // S, then P, of the current tile
    float m_run[H];
    float l_run[H];
    float alpha[H];
    unsigned ticket;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int e_off(int row, int d) {  // float offset in an E tile
    return row * kKvDim + ((((d >> 2) ^ (row & 7))) << 2) + (d & 3);
}
__device__ __forceinline__ int q_off(int row, int d) {  // bf16 offset in Q
    return row * kKvDim + ((((d >> 3) ^ (row & 7))) << 3) + (d & 7);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

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

template <int H>
__global__ void __launch_bounds__(kThreads, 1) attend_kernel(AttnArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<H>& sm = *reinterpret_cast<AttnSmem<H>*>(smem_raw);
    constexpr int MT = H / 16;                       // m-tiles of heads
    constexpr int NTW = (MT * 4 >= 8) ? (MT * 4 / 8) : 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int item_idx = a.item0 + blockIdx.x;
    const AttnItem it = a.items[item_idx];
    const int l = it.layer, b = it.seq;
    const size_t lb = (size_t)l * a.B + b;
    int cnt = a.count_l[lb];
    if (cnt < 0 || cnt > a.S) {
        if (tid == 0) atomicOr(a.err, kErrBounds);
        cnt = cnt < 0 ? 0 : a.S;
    }
    const int R = kWindow + cnt;
    const int row0 = it.split * a.split_rows;
    const int row1 = min(R, row0 + a.split_rows);
    const int n_tiles = row1 > row0 ? (row1 - row0 + kTile - 1) / kTile : 0;

    const float* win = a.window + lb * kWindow * kKvDim;
    const float* stg = a.staging + lb * (size_t)a.G * kKvDim;
    const int32_t* ph = a.phys + lb * a.S;

    for (int h = tid; h < H; h += kThreads) {
        sm.m_run[h] = -INFINITY;
        sm.l_run[h] = 0.f;
        sm.alpha[h] = 1.f;
    }

    // ---- queries: H x 64 chunks of 16 B
    const uint16_t* qg = a.q + lb * H * kKvDim;
    for (int i = tid; i < H * (kKvDim / 8); i += kThreads) {
        const int row = i >> 6, c = i & 63;
        cp_async16(&sm.q[row * kKvDim + ((c ^ (row & 7)) << 3)], qg + row * kKvDim + c * 8, 16);
    }

    // each thread copies 16 chunks of one tile row: row = tid / 8, chunks (tid % 8) + 8j
    auto load_tile = [&](int tile, int buf) {
        const int rr = tid >> 3, cg = tid & 7;
        const int row = row0 + tile * kTile + rr;
        const float* src = win;
        int bytes = 16;
        if (row >= row1) {
            bytes = 0;                       // zero-fill past the split
        } else if (row < kWindow) {
            src = win + (size_t)row * kKvDim;
        } else {
            const int slot = ph[row - kWindow] - kWindow;
            if (slot < 0 || slot >= a.G) {
                atomicOr(a.err, kErrBounds);
                bytes = 0;
            } else {
                src = stg + (size_t)slot * kKvDim;
            }
        }
        float* dst = sm.e[buf] + rr * kKvDim;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = cg + 8 * j;
            cp_async16(dst + ((c ^ (rr & 7)) << 2), src + (bytes ? c * 4 : 0), bytes);
        }
    };

    if (n_tiles > 0) load_tile(0, 0);
    cp_async_commit();

    float acc[MT][8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nn = 0; nn < 8; ++nn) acc[mt][nn][0] = acc[mt][nn][1] = acc[mt][nn][2] = acc[mt][nn][3] = 0.f;

    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(sm.q);

    for (int tile = 0; tile < n_tiles; ++tile) {
        const int buf = tile & 1;
        if (tile + 1 < n_tiles) {
            load_tile(tile + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float* E = sm.e[buf];

        // ---- S = Q E^T for this tile (H x 32)
        {
            const int first = warp * NTW;
            if (first < MT * 4) {
                const int mt = first >> 2, nt0 = first & 3;
                const int h0 = mt * 16 + g, h1 = h0 + 8;
                float s[NTW][4];
#pragma unroll
                for (int u = 0; u < NTW; ++u) s[u][0] = s[u][1] = s[u][2] = s[u][3] = 0.f;
#pragma unroll 4
                for (int j = 0; j < kKvDim / 8; ++j) {
                    const uint32_t wa = q32[q_off(h0, 8 * j + 2 * t) >> 1];
                    const uint32_t wb = q32[q_off(h1, 8 * j + 2 * t) >> 1];
                    const uint32_t a0 = wa << 16, a2 = wa & 0xffff0000u;
                    const uint32_t a1 = wb << 16, a3 = wb & 0xffff0000u;
#pragma unroll
                    for (int u = 0; u < NTW; ++u) {
                        const int rrow = (nt0 + u) * 8 + g;
                        const float2 ev = *reinterpret_cast<const float2*>(&E[e_off(rrow, 8 * j + 2 * t)]);
                        mma_tf32(s[u], a0, a1, a2, a3, to_tf32(ev.x), to_tf32(ev.y));
                    }
                }
#pragma unroll
                for (int u = 0; u < NTW; ++u) {
                    const int col = (nt0 + u) * 8 + 2 * t;
                    *reinterpret_cast<float2*>(&sm.p[h0 * kPStride + col]) = make_float2(s[u][0], s[u][1]);
                    *reinterpret_cast<float2*>(&sm.p[h1 * kPStride + col]) = make_float2(s[u][2], s[u][3]);
                }
            }
        }
        __syncthreads();

        // ---- online softmax (base 2): one warp per head, lane = row
        {
            const bool valid = row0 + tile * kTile + lane < row1;
            for (int h = warp; h < H; h += kThreads / 32) {
                const float v = valid ? sm.p[h * kPStride + lane] * a.sl2 : -INFINITY;
                const float mx = warp_max(v);
                const float m_old = sm.m_run[h];
                const float m_new = fmaxf(m_old, mx);
                const float alpha = exp2f(m_old - m_new);
                const float p = valid ? exp2f(v - m_new) : 0.f;
                const float sum = warp_sum(p);
                sm.p[h * kPStride + lane] = p;
                __syncwarp();
                if (lane == 0) {
                    sm.l_run[h] = sm.l_run[h] * alpha + sum;
                    sm.m_run[h] = m_new;
                    sm.alpha[h] = alpha;
                }
            }
        }
        __syncthreads();

        // ---- O = O * alpha + P E (this warp: latent columns [64 warp, 64 warp + 64))
        {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float al0 = sm.alpha[mt * 16 + g], al1 = sm.alpha[mt * 16 + g + 8];
#pragma unroll
                for (int nn = 0; nn < 8; ++nn) {
                    acc[mt][nn][0] *= al0;
                    acc[mt][nn][1] *= al0;
                    acc[mt][nn][2] *= al1;
                    acc[mt][nn][3] *= al1;
                }
            }
#pragma unroll
            for (int jj = 0; jj < kTile / 8; ++jj) {
                const int r0 = 8 * jj + 2 * t;
                uint32_t pa[MT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const float2 x0 = *reinterpret_cast<const float2*>(&sm.p[(mt * 16 + g) * kPStride + r0]);
                    const float2 x1 = *reinterpret_cast<const float2*>(&sm.p[(mt * 16 + g + 8) * kPStride + r0]);
                    pa[mt][0] = to_tf32(x0.x);
                    pa[mt][2] = to_tf32(x0.y);
                    pa[mt][1] = to_tf32(x1.x);
                    pa[mt][3] = to_tf32(x1.y);
                }
#pragma unroll
                for (int nn = 0; nn < 8; ++nn) {
                    const int d = warp * 64 + nn * 8 + g;
                    const uint32_t b0 = to_tf32(E[e_off(r0, d)]);
                    const uint32_t b1 = to_tf32(E[e_off(r0 + 1, d)]);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        mma_tf32(acc[mt][nn], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- epilogue
    const bool single = it.n_splits == 1;
    if (single) {
        float* o = a.out + lb * H * kKvDim;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int h0 = mt * 16 + g, h1 = h0 + 8;
            const float i0 = 1.f / sm.l_run[h0], i1 = 1.f / sm.l_run[h1];
#pragma unroll
            for (int nn = 0; nn < 8; ++nn) {
                const int d = warp * 64 + nn * 8 + 2 * t;
                *reinterpret_cast<float2*>(&o[h0 * kKvDim + d]) = make_float2(acc[mt][nn][0] * i0, acc[mt][nn][1] * i0);
                *reinterpret_cast<float2*>(&o[h1 * kKvDim + d]) = make_float2(acc[mt][nn][2] * i1, acc[mt][nn][3] * i1);
            }
        }
        return;
    }
    float* po = a.part_o + (size_t)item_idx * H * kKvDim;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int h0 = mt * 16 + g, h1 = h0 + 8;
#pragma unroll
        for (int nn = 0; nn < 8; ++nn) {
            const int d = warp * 64 + nn * 8 + 2 * t;
            __stcg(reinterpret_cast<float2*>(&po[h0 * kKvDim + d]), make_float2(acc[mt][nn][0], acc[mt][nn][1]));
            __stcg(reinterpret_cast<float2*>(&po[h1 * kKvDim + d]), make_float2(acc[mt][nn][2], acc[mt][nn][3]));
        }
    }
    float* pml = a.part_ml + (size_t)item_idx * 2 * H;
    for (int h = tid; h < H; h += kThreads) {
        __stcg(&pml[h], sm.m_run[h]);
        __stcg(&pml[H + h], sm.l_run[h]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.ticket = atomicAdd(&a.counters[lb], 1u);
    __syncthreads();
    if (sm.ticket != (unsigned)(it.n_splits - 1)) return;
    __threadfence();

    // ---- last CTA: merge the splits of this (layer, sequence) in split order
    const int ns = it.n_splits;
    const int base = item_idx - it.split;
    float* wts = sm.e[0];   // [ns][H] merge weights (reuses the tile buffer)
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
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < ns; ++s) {
            const float w = wts[s * H + h];
            if (w == 0.f) continue;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part_o + (size_t)(base + s) * H * kKvDim) + i);
            r.x += w * v.x;
            r.y += w * v.y;
            r.z += w * v.z;
            r.w += w * v.w;
        }
        reinterpret_cast<float4*>(o)[i] = r;
    }
    if (tid == 0) a.counters[lb] = 0u;
}

template <int H>
cudaError_t launch_h(const AttnArgs& args, int n_items, cudaStream_t st) {
    const size_t smem = sizeof(AttnSmem<H>);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    attend_kernel<H><<<n_items, kThreads, smem, st>>>(args);
    return cudaGetLastError();
}

}  // namespace

int attend_max_splits() { return kMaxSplits; }

cudaError_t launch_attend(const AttnItem* items, int item0, int n_items, int split_rows,
                          int n_heads, int B, int G, int S, const uint16_t* q, const float* window,
                          const float* staging, const int32_t* phys, const int32_t* count_l,
                          float* out, float* part_o, float* part_ml, unsigned* counters,
                          uint32_t* err, cudaStream_t st) {
    if (n_items <= 0) return cudaSuccess;
    AttnArgs args{items, item0, split_rows, B, G, S, q, window, staging, phys, count_l,
                  out, part_o, part_ml, counters, err,
                  (float)(1.4426950408889634 / std::sqrt((double)kKvDim))};
    switch (n_heads) {
        case 16: return launch_h<16>(args, n_items, st);
        case 32: return launch_h<32>(args, n_items, st);
        case 64: return launch_h<64>(args, n_items, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace srh
