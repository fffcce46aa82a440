// K-score on the 5th-generation tensor cores: memory-indexer scoring +
// ensemble for every compressed chunk, one key set shared by the three
// indexers.
//
// PocketLLM "FlashMemory 1M 上下文显存优化使用文档", section 技术细节 / 架构概览,
// scoring box steps 1-3, and the FlashMemory-DeepSeek-V4 summary, sections
// "LSA 让模型预判 KV chunk" and "Memory Indexer 放哪里":
//   s_{i,h}(c) = <Q[i,h,:], K[c,:]>, s_i(c) = scale * max_h s_{i,h}(c) + b_i,
//   s(c) = max_i s_i(c) (OR-mode) or mean_i s_i(c).
//
// The keys are the only large operand (256 B per chunk, read once per pass),
// so the kernel is a TMA stream: a tile is 128 chunks (32 KB), and each CTA
// runs a contiguous range of one sequence's tiles through a ring of shared
// memory stages. Roles (192 threads, two CTAs per SM):
//   warp 0   one thread issues the TMA loads: the sequence's query block once
//            (24 rows, padded to 32 with zeros by the tensor map), then every
//            tile, each as two 128B-swizzled boxes of 128 chunks x 64 d; the
//            query block and the first two tiles as soon as the barriers are
//            initialized, before the CTA's set-up barrier;
//   warp 1   allocates TMEM; one thread issues, per tile, the eight
//            tcgen05.mma kind::f16 (bf16) steps S[c, i*8+h] = K[c, :] . Q[i,h, :]
//            (M = 128 chunks, N = 32, K = 128) into one of two TMEM
//            accumulators, and commits to the stage's "empty" barrier and the
//            accumulator's "full" barrier;
//   warps 2-5  the epilogue: thread = TMEM lane = chunk of the tile; it reads
//            its 24 products, takes the head max per indexer, scales, biases,
//            ensembles, writes the fp32 score (coalesced) and bumps the
//            4096-bin histogram of the score's order-preserving key (top 12
//            bits) that the selector uses for its first radix digit.
// Every wait is bounded. On a timeout the CTA records kErrTimeout, waits for
// its copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>

#include "srh_internal.cuh"
#include "umma.cuh"

namespace srh {
namespace {

using namespace umma;

constexpr int kTile = 128;                          // chunks per tile (MMA M)
constexpr int kN = 32;                              // MMA N: 24 query rows + 8 zero rows
constexpr int kStages = 2;                          // key tiles in flight per CTA
constexpr int kAcc = 2;                             // TMEM accumulators
constexpr int kThreadsTc = 192;                     // 6 warps
constexpr int kEpiThreads = 128;                    // warps 2-5
constexpr int kStageBytes = kTile * kIdxDim * 2;    // 32 KB
constexpr int kHalfBytes = kStageBytes / 2;         // one 64-d box: 128 rows x 128 B
constexpr int kQBytes = kN * kIdxDim * 2;           // 8 KB
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffHist = kOffQ + kQBytes;
constexpr int kOffBar = kOffHist + kHistBins * 4;

struct Bars {
    uint64_t full[kStages];    // TMA bytes of a tile landed
    uint64_t empty[kStages];   // the tile's MMAs completed
    uint64_t tfull[kAcc];      // the accumulator's MMAs completed
    uint64_t tempty[kAcc];     // the epilogue read the accumulator
    uint64_t qfull;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
constexpr int kSmemTc = kOffBar + (int)sizeof(Bars) + 1024;   // + base alignment slack
static_assert(2 * kSmemTc <= 232448, "two scoring CTAs must fit one SM");

struct ScoreTcArgs {
    int n;
    int tiles;        // tiles per sequence
    int parts;        // CTAs per sequence
    float scale;
    float bias[3];
    int ensemble;
    float* scores;
    uint32_t* hist;           // nullptr: no histogram
    uint32_t* err;
    CandSink sink;            // sink.cand == nullptr: no candidate list
};

// Bounded wait that also leaves when another role has aborted the CTA.
__device__ __forceinline__ bool wait_tc(uint64_t* bar, uint32_t parity, volatile int* abort) {
    return mbar_wait_abort(bar, parity, abort) > 0;
}

__global__ void __launch_bounds__(kThreadsTc, 2)
score_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                const __grid_constant__ ScoreTcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars& bs = *reinterpret_cast<Bars*>(sm + kOffBar);
    uint32_t* h_s = reinterpret_cast<uint32_t*>(sm + kOffHist);
    volatile int* abort = &bs.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y;
    const int t0 = (int)((long long)blockIdx.x * a.tiles / a.parts);
    const int t1 = (int)((long long)(blockIdx.x + 1) * a.tiles / a.parts);
    const int nt = t1 - t0;
    pdl_trigger();
    // tile i of this CTA's range into stage i % kStages (thread 0)
    auto issue_tile = [&](int i) {
        const int s = i % kStages;
        const uint32_t dst = smem_u32(sm + s * kStageBytes);
        const int y = (t0 + i) * kTile;
        mbar_arrive_expect_tx(&bs.full[s], kStageBytes);
        tma_load_3d(dst, &kmap, 0, y, b, &bs.full[s]);
        tma_load_3d(dst + kHalfBytes, &kmap, 64, y, b, &bs.full[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bs.full[s], 1);
            mbar_init(&bs.empty[s], 1);
        }
        for (int x = 0; x < kAcc; ++x) {
            mbar_init(&bs.tfull[x], 1);
            mbar_init(&bs.tempty[x], kEpiThreads);
        }
        mbar_init(&bs.qfull, 1);
        mbar_init(&bs.drain, 1);
        bs.abort = 0;
        fence_mbar_init();
        if (nt > 0) {
            // the queries and the first tiles are requested before the set-up
            // barrier, so that HBM starts streaming while TMEM and the histogram
            // are set up (the barriers' initialization is ordered before the
            // copies' completions by the proxy fence)
            fence_async_smem();
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(&kmap) : "memory");
            const uint32_t q0 = smem_u32(sm + kOffQ);
            mbar_arrive_expect_tx(&bs.qfull, kQBytes);
            tma_load_3d(q0, &qmap, 0, 0, b, &bs.qfull);
            tma_load_3d(q0 + kQBytes / 2, &qmap, 64, 0, b, &bs.qfull);
            for (int i = 0; i < nt && i < kStages; ++i) issue_tile(i);
        }
    }
    if (warp == 1) tmem_alloc(&bs.tmem_base, kAcc * kN);
    if (a.hist)
        for (int i = tid; i < kHistBins; i += kThreadsTc) h_s[i] = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && nt > 0) {
            // the queries and tiles 0 .. kStages - 1 were issued before the set-up barrier
            int issued = nt < kStages ? nt : kStages;
            for (int i = issued; i < nt; ++i) {
                const int s = i % kStages;
                if (!wait_tc(&bs.empty[s], ((i / kStages) + 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                issue_tile(i);
                issued = i + 1;
            }
            if (!ok) {
                // an aborted CTA: every copy issued above lands before the CTA may leave
                mbar_wait(&bs.qfull, 0);
                for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                    mbar_wait(&bs.full[i % kStages], (i / kStages) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nt > 0) {
            constexpr uint32_t idesc = idesc_f32acc(1, 0, 0, kTile, kN);   // bf16 x bf16 -> f32, K-major
            const uint32_t tmem = bs.tmem_base;
            const uint32_t q0 = smem_u32(sm + kOffQ);
            if (!wait_tc(&bs.qfull, 0, abort)) ok = false;
            for (int i = 0; ok && i < nt; ++i) {
                const int s = i % kStages, x = i % kAcc;
                if (!wait_tc(&bs.full[s], (i / kStages) & 1, abort)) { ok = false; break; }
                if (i >= kAcc && !wait_tc(&bs.tempty[x], ((i / kAcc) + 1) & 1, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sm + s * kStageBytes);
#pragma unroll
                for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (uint32_t)(kk & 3) * 32;
                    const uint32_t qoff = (uint32_t)(kk >> 2) * (kQBytes / 2) + (uint32_t)(kk & 3) * 32;
                    mma_f16kind(tmem + x * kN, desc_sw128(a0 + off, 16, 1024), desc_sw128(q0 + qoff, 16, 1024),
                                idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bs.empty[s]);
                mma_commit(&bs.tfull[x]);
            }
            // every MMA issued above completes before TMEM is freed
            mma_commit(&bs.drain);
            if (!mbar_wait(&bs.drain, 0)) ok = false;
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int r = (warp & 3) * 32 + lane;   // tile row = TMEM lane
        float* scores_b = a.scores + (size_t)b * a.n;
        for (int i = 0; i < nt; ++i) {
            const int x = i % kAcc;
            // warp-uniform: the candidate append below is a warp collective
            const bool got = wait_tc(&bs.tfull[x], (i / kAcc) & 1, abort);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[32];
            tmem_ld16(bs.tmem_base + lane_base + x * kN, *reinterpret_cast<float(*)[16]>(v));
            tmem_ld16(bs.tmem_base + lane_base + x * kN + 16, *reinterpret_cast<float(*)[16]>(v + 16));
            tmem_ld_wait();
            tmem_regs_ready(v);
            tmem_regs_ready(v + 16);
            tc_fence_before();
            mbar_arrive(&bs.tempty[x]);
            float si[kIdx];
#pragma unroll
            for (int q = 0; q < kIdx; ++q) {
                float m = v[8 * q];
#pragma unroll
                for (int h = 1; h < kIdxHeads; ++h) m = fmaxf(m, v[8 * q + h]);
                si[q] = fmaf(a.scale, m, a.bias[q]);
            }
            const float e = a.ensemble == SRH_ENSEMBLE_MAX ? fmaxf(fmaxf(si[0], si[1]), si[2])
                                                           : (si[0] + si[1] + si[2]) / 3.0f;
            const int c = (t0 + i) * kTile + r;
            const uint32_t key = ordered_key(e);
            if (c < a.n) {
                scores_b[c] = e;
                if (a.hist) atomicAdd(&h_s[key >> 20], 1u);
            }
            if (a.sink.cand) append_candidate(a.sink, b, c < a.n && key > a.sink.key, key, (uint32_t)c);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    const bool failed = __syncthreads_or(!ok);
    if (failed && tid == 0) atomicOr(a.err, kErrTimeout);
    if (a.hist) {
        uint32_t* hb = a.hist + (size_t)b * kHistBins;
        for (int i = tid; i < kHistBins; i += kThreadsTc)
            if (h_s[i]) atomicAdd(&hb[i], h_s[i]);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(bs.tmem_base, kAcc * kN);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = []() -> EncodeTiled {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// bf16 tensor [dim2][dim1][128] (row pitch 256 B) read in boxes of 64 x rows x 1
// with the 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* base, long long dim1, long long dim2, int rows) {
    const EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kIdxDim, (cuuint64_t)dim1, (cuuint64_t)dim2};
    const cuuint64_t strides[2] = {(cuuint64_t)kIdxDim * 2, (cuuint64_t)dim1 * kIdxDim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {
// The bounded-wait path of the kernels above, on its own: the barrier expects
// one arrival that never comes, so mbar_wait gives up after limit_ns.
__global__ void wait_selftest_kernel(uint32_t* err, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) atomicOr(err, kErrTimeout);
}
}  // namespace

cudaError_t launch_wait_selftest(uint32_t* err, unsigned long long limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

cudaError_t set_score_tc_attrs() {
    return cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
}

cudaError_t launch_score_tc(const uint16_t* keys, int n, int B, const uint16_t* q, float scale, const float* bias3,
                            int ensemble, float* scores, uint32_t* hist, uint32_t* err, int sm_count,
                            cudaStream_t st, CandSink sink) {
    CUtensorMap kmap, qmap;
    if (!encode_rows(&kmap, keys, n, B, kTile) || !encode_rows(&qmap, q, kIdx * kIdxHeads, B, kN))
        return cudaErrorNotSupported;
    ScoreTcArgs args{};
    args.n = n;
    args.tiles = (n + kTile - 1) / kTile;
    // two CTAs per SM over all sequences; a CTA never spans two sequences
    long long parts = (2LL * sm_count) / B;
    if (parts > args.tiles) parts = args.tiles;
    if (parts < 1) parts = 1;
    args.parts = (int)parts;
    args.scale = scale;
    args.bias[0] = bias3[0];
    args.bias[1] = bias3[1];
    args.bias[2] = bias3[2];
    args.ensemble = ensemble;
    args.scores = scores;
    args.hist = hist;
    args.err = err;
    args.sink = sink;
    score_tc_kernel<<<dim3((unsigned)parts, (unsigned)B), kThreadsTc, kSmemTc, st>>>(kmap, qmap, args);
    return cudaGetLastError();
}

}  // namespace srh
