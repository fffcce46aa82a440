// Internal declarations shared by the translation units of libsrh.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/srh.h"

namespace srh {

// Programmatic dependent launch. A kernel launched with `chained` may start
// while the previous kernel on the stream is still running: it must call
// pdl_wait() before it reads anything that kernel (or an earlier one) wrote.
// pdl_trigger() lets the next chained kernel start as soon as every CTA of
// this one has issued it. Both are no-ops for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            bool chained, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kKvDim = SRH_KV_DIM;
constexpr int kWindow = SRH_WINDOW;
constexpr int kIdx = SRH_N_INDEXERS;
constexpr int kIdxHeads = SRH_INDEXER_HEADS;
constexpr int kIdxDim = SRH_INDEXER_DIM;
constexpr int kHistBins = 4096;        // score histogram: top 12 bits of the ordered key
constexpr int kMaxSelect = 4096;       // largest S
constexpr int kMaxGpuChunks = 4096;    // largest G
constexpr int kAttnTile = 128;         // rows per attention tile
constexpr int kAttnMlStride = 2 * SRH_MAX_HEADS + 4;   // floats per attention partial's statistics: m, l, scale

// Bits of the sticky device error word.
enum : uint32_t {
    kErrNotStored = 1u,
    kErrBounds = 2u,
    kErrTimeout = 4u,
    kErrRange = 8u,      // an attention operand beyond fp16's finite range
};

// Device-side counters (one array of unsigned long long).
enum : int {
    kStatHits = 0,
    kStatMisses,
    kStatSelected,
    kStatResidentFill,
    kStatCount
};

// Adaptive capacity of one swapped (layer, sequence): slots [0, g) are in use.
struct AdaptState {
    int g;               // slots used by the last resolve
    int g_next;          // slots the next resolve uses (policy decision or host setting)
    int ep_steps;        // swap steps in the current hit-rate window
    unsigned version;    // resolves of this (layer, sequence) so far (raised by each, with release)
    long long ep_hits;   // hits in the window
    long long ep_sel;    // chunks resolved in the window
};

// The hit-rate policy, passed by value to the resolve kernel (on == 0: none).
struct AdaptParams {
    int on;
    int g_min, g_max;
    int epoch;
    int lo_pm, hi_pm;
    int delta;
};

// Per-layer facts and state pointers, kept in device memory ([L] array).
struct LayerDev {
    long long cap;           // chunks of this layer
    int ratio;               // compression ratio
    int swap;                // 1 if cap > G
    const float* pool;       // device alias of the mapped pinned pool [B][cap][D]
    uint8_t* host_ready;     // [B][cap]
    int* slot_of;            // [B][cap]: slot holding chunk c, -1 if none (swap layers)
    int* slot_logical;       // [B][G]: chunk in slot s, -1 if free (swap layers)
    int* lru_order;          // [B][G]: slots in use from least (0) to most recently used
    AdaptState* adapt;       // [B] (swap layers)
};

// One segment of the attention plan: rows [r0, r1) of one (layer, seq) (rows
// 0-127 are the window rows, then the staged rows in selection order), run in
// tiles of up to 128 rows from r0. A CTA runs one or more segments. A segment
// holding every row of its pair writes the output; the others write partials
// to `slot`, and the CTA merges share `part` of the pair's output once every
// partial is in.
struct AttnSeg {
    int lb;      // layer * B + seq
    int r0;
    int r1;
    int slot;    // partial slot, or -1
    int merge;   // index of the pair's MergeItem in its plan, or -1
    int part;    // this segment's place among the pair's partials (its merge share)
};

// One (layer, seq) whose tiles were cut across ns > 1 CTAs: its partial
// slots first .. first + ns - 1 are combined in row order.
struct MergeItem {
    int lb;      // layer * B + seq
    int first;
    int ns;
    int pad;
};

// The static attention plan of one lsa_attend scope (all layers, or one).
struct AttnPlan {
    int seg0, n_segs;      // into Ctx::d_segs
    int cta0, n_ctas;      // into Ctx::d_cta_begin (n_ctas + 1 entries from cta0)
    int merge0, n_merges;  // into Ctx::d_merges
    int n_slots;
    int one_wave;          // 1: each pair cut into chunks of equal bytes; 0: stream-K tile ranges
};

struct Ctx {
    srh_config cfg{};
    std::vector<int> ratios;
    std::vector<long long> caps;
    std::vector<int> swap;
    int S = 0;           // selection row stride
    int G = 0;
    int B = 0;
    int L = 0;
    long long n_src = 0; // scored chunks (ratio src_ratio)
    int device = 0;
    int sm_count = 0;

    // pinned pools: one per layer, [B][cap][D]
    std::vector<float*> pool_host;
    std::vector<float*> pool_dev;
    // host_ready mirror (host) per layer [B][cap]
    std::vector<std::vector<uint8_t>> ready_host;
    // swap-disabled layers whose staging rows need a (re)fill, per layer
    std::vector<uint8_t> resident_dirty;

    // device state
    LayerDev* d_layers = nullptr;
    int* d_swap_layers = nullptr;       // the swapped layers' indices, ascending (the gather's rows)
    std::vector<int> swap_pos;          // each layer's place in that list, -1 if it does not swap
    int n_swap = 0;
    std::vector<LayerDev> h_layers;
    unsigned long long* d_stats = nullptr;
    uint32_t* d_err = nullptr;
    bool chained = false;               // srh_set_chained: step kernels may launch early
    AdaptParams adapt{};                // srh_set_adaptive
    uint32_t* d_hist = nullptr;         // [B][kHistBins]
    bool hist_clean = true;             // d_hist is all zeros (cleared, or consumed by a selection)
    unsigned long long* d_cand = nullptr; // [B][select_cand_cap()] candidate composites
    int* d_cand_cnt = nullptr;          // [B]
    bool cand_clean = true;             // d_cand_cnt is zero (cleared, or consumed by a selection)
    // threshold selection: the threshold of the last fm_select in that mode; the
    // next scoring pass appends the chunks above it to d_cand, and a selection
    // with that threshold on those scores uses the list (no candidate pass)
    bool thresh_hint_valid = false;
    float thresh_hint = 0.f;
    const float* cand_scores = nullptr; // the d_scores d_cand was built from by a scoring pass
    int cand_n = -1;
    float cand_thresh = 0.f;
    const float* hist_scores = nullptr; // the d_scores the histogram describes
    int hist_n = -1;
    int2* d_miss = nullptr;             // [L][B][S] (chunk, slot)
    int* d_miss_count = nullptr;        // [L][B]
    uint32_t* d_sink = nullptr;         // write target that keeps the page-touch loads alive
    // attention plans: [0] all layers, [1 + l] layer l alone
    std::vector<AttnPlan> plans;
    AttnSeg* d_segs = nullptr;
    int* d_cta_begin = nullptr;
    MergeItem* d_merges = nullptr;
    int max_slots = 0;
    uint16_t* d_part_o = nullptr;       // fp16 [max_slots][SRH_MAX_HEADS][D]
    float* d_part_ml = nullptr;         // [max_slots][kAttnMlStride]
    unsigned long long* d_merge_cnt = nullptr;   // arrivals per split pair, all plans
    // bookkeeping
    uint16_t* staging = nullptr;        // the staging buffer (fp16 rows) bound to this context
    cudaEvent_t ev_resolved = nullptr;
    cudaEvent_t ev_gathered = nullptr;
    unsigned long long stage_calls = 0;
    unsigned long long resident_fill_bytes = 0;
    unsigned long long stored_bytes = 0;   // kvswap_store: rows written to the host pool
    std::string last_error;
};

#ifdef __CUDACC__
// Order-preserving 32-bit key of a score: a larger score gives a larger key and
// -0 maps like +0, so equal scores give equal keys.
__host__ __device__ __forceinline__ uint32_t ordered_key(float s) {
    s = (s == 0.0f) ? 0.0f : s;
    uint32_t u;
    memcpy(&u, &s, sizeof u);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The selection's unique 64-bit key of chunk idx: larger = (score descending,
// index ascending).
__host__ __device__ __forceinline__ unsigned long long candidate_key(uint32_t key, uint32_t idx) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~idx);
}

// Where a scoring pass appends the chunks whose key exceeds `key` (the
// selection's threshold): the candidate list [B][cap] and counts [B] that the
// select kernel consumes. A count past `cap` means the list overflowed (the
// select kernel then scans all the scores). cand == nullptr: no list.
struct CandSink {
    uint32_t key;
    unsigned long long* cand;
    int* cnt;
    int cap;
};

// Appends (key, idx) to the sequence's list when `pass`; every lane of the warp
// calls it (one atomic per warp).
__device__ __forceinline__ void append_candidate(const CandSink& sk, int b, bool pass, uint32_t key,
                                                 uint32_t idx) {
    const unsigned m = __ballot_sync(0xffffffffu, pass);
    if (!m) return;
    const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(&sk.cnt[b], __popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (pass) {
        const int pos = base + __popc(m & ((1u << lane) - 1u));
        if (pos < sk.cap) sk.cand[(size_t)b * sk.cap + pos] = candidate_key(key, idx);
    }
}
#endif

// ---------------------------------------------------------------- launchers
// The scoring launchers add into the first-digit histogram `hist`; with
// `clear_hist` they zero it first (the select kernel leaves the rows it reads
// zeroed, so a histogram consumed by a selection needs no clearing).
// With sink.cand set, the scoring kernels also append the chunks above
// sink.key to the candidate list (the counts are zeroed first with
// clear_cand); hist may be nullptr (no histogram).
cudaError_t launch_score(const uint16_t* keys, int n, int B, const uint16_t* q, float scale,
                         const float* bias3, int ensemble, float* scores, uint32_t* hist, uint32_t* err,
                         int sm_count, cudaStream_t st, int key_sets, bool clear_hist, CandSink sink,
                         bool clear_cand);
// One key set on the tensor cores (TMA-streamed key tiles, tcgen05, TMEM);
// launch_score uses it from this many chunks per call (all sequences) up.
constexpr long long kTcMinChunks = 1LL << 18;
cudaError_t launch_score_tc(const uint16_t* keys, int n, int B, const uint16_t* q, float scale, const float* bias3,
                            int ensemble, float* scores, uint32_t* hist, uint32_t* err, int sm_count,
                            cudaStream_t st, CandSink sink);
cudaError_t launch_hist(const float* scores, int n, int B, uint32_t* hist, cudaStream_t st, bool clear_hist);
cudaError_t launch_quantize_keys(const uint16_t* keys, long long total, uint8_t* codes, float* kscale,
                                 int sm_count, cudaStream_t st);
cudaError_t launch_score_fp8(const uint8_t* codes, const float* kscale, int n, int B, const uint16_t* q, float scale,
                             const float* bias3, int ensemble, float* scores, uint32_t* hist, int sm_count,
                             cudaStream_t st, bool clear_hist);
// Candidate pass for large n: appends the selectable keys to cand, counting in
// cand_cnt (zeroed first with clear_count; the select kernel leaves it zeroed).
cudaError_t launch_collect(const float* scores, int n, int B, int mode, int K, float thresh,
                           const uint32_t* hist, unsigned long long* cand, int* cand_cnt, int cap,
                           cudaStream_t st, bool clear_count, bool chained);
int select_cand_cap();
constexpr int kCollectMinN = 16384;    // fm_select runs the candidate pass above this n
cudaError_t launch_select(const float* scores, int n, int B, int mode, int k, float thresh,
                          int clamp, int S, uint32_t* hist, int32_t* sel, int32_t* count,
                          cudaStream_t st, const unsigned long long* cand = nullptr,
                          int* cand_cnt = nullptr, int cand_cap = 0, bool chained = false);
// Swapped layers of at most this many chunks keep a shared-memory copy of their
// slot map in the resolve kernel (read before its dependency wait).
constexpr long long kLruMirrorMax = 1 << 13;
cudaError_t launch_lru(const LayerDev* layers, int l0, int nl, int B, int G, int S, int src_ratio,
                       long long max_dedup_cap, long long max_mirror_cap, const int32_t* sel, const int32_t* count,
                       int32_t* phys, int32_t* count_l, int2* miss, int* miss_count,
                       unsigned long long* stats, uint32_t* err, AdaptParams ap, cudaStream_t st,
                       bool chained);
// Gathers the misses of the swapped layers swap_layers[0 .. n_sw) (every
// sequence); nl_call is the call's layer count, which sizes the grid per layer.
cudaError_t launch_gather(const LayerDev* layers, const int* swap_layers, int n_sw, int nl_call, int B, int G, int S,
                          const int2* miss, const int* miss_count, uint16_t* staging,
                          uint32_t* err, int sm_count, cudaStream_t st, bool chained);
cudaError_t launch_touch(const float* p, long long n_floats, uint32_t* sink, int sm_count, cudaStream_t st);
cudaError_t launch_store(const LayerDev* layers, int l, int B, int G, int seq, long long c0, int n,
                         const float* rows, uint16_t* staging, uint32_t* err, cudaStream_t st);
cudaError_t launch_resident_fill(const float* pool_dev, const uint8_t* ready, long long cap,
                                 int layer, int B, int G, uint16_t* staging, uint32_t* err, cudaStream_t st);
cudaError_t launch_attend(const AttnSeg* segs, const int* cta_begin, int n_ctas, const MergeItem* merges,
                          unsigned long long* merge_cnt, int n_heads, int B, int G, int S, const uint16_t* q,
                          const float* window, const uint16_t* staging, const int32_t* phys, const int32_t* count_l,
                          float* out, uint16_t* part_o, float* part_ml, uint32_t* err, cudaStream_t st,
                          bool chained);
size_t lru_smem_bytes(int S, int G);
int attend_max_splits();
int attend_max_duties();   // split pairs one attention CTA may take part in
// One CTA waits (limit_ns) on an mbarrier phase nothing completes and records
// kErrTimeout in err: the self-test of the kernels' bounded waits.
cudaError_t launch_wait_selftest(uint32_t* err, unsigned long long limit_ns, cudaStream_t st);

// Shared-memory limits of the kernels that need more than the default 48 KB,
// set on the current device once, outside any launch sequence: changing a
// kernel's limit between two chained launches let the second start before the
// first had finished (seen with the resolve kernel). srh_create sets all of
// them; fm_select_noalloc sets the select kernel's in its per-device set-up.
cudaError_t set_select_attrs();
cudaError_t set_lru_attrs();
cudaError_t set_attend_attrs();
cudaError_t set_score_tc_attrs();

}  // namespace srh

struct srh_ctx : public srh::Ctx {};
