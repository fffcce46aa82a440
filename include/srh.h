/*
 * srh.h -- C ABI of the FlashMemory lookahead-sparse-attention + KV_SWAP
 * decode-step hot path, for one NVIDIA GB300 (sm_103a).
 *
 * One decode step is four calls, in this order:
 *
 *   fm_score      score every compressed chunk with 3 memory-indexer query
 *                 sets against the frozen bf16 indexer keys and ensemble the
 *                 three per-indexer logits (max = OR-mode, or mean);
 *   fm_select     pick chunks by top-k or by sigmoid threshold, ordered by
 *                 (score descending, chunk index ascending);
 *   kvswap_stage  per sparse layer, map the global selection to the layer's
 *                 chunks, resolve them against the GPU staging slots with the
 *                 LRU of the Swap-in flow, and gather the misses from the
 *                 pinned host pool;
 *   lsa_attend    per sparse layer, attention of every head over the
 *                 128-row window plus the staged selected chunks.
 *
 * Sources (the pages this interface restates):
 *   [P1] PocketLLM, "FlashMemory 1M 上下文显存优化使用文档": sections
 *        "配置说明" (flags), "关键参数调优" (GPU_CHUNKS rule, pinned-size
 *        formula), "故障排查" (the four errors and swap auto-disable),
 *        "技术细节 / 架构概览" (scoring box and per-layer attention box,
 *        memory layout), "KV_SWAP 实现细节" (GgufKvSwapLayerState, Swap-in
 *        and Store flows).
 *   [P2] FlashMemory-DeepSeek-V4 summary (wmrh.cn/news/1094): sections
 *        "LSA 让模型预判 KV chunk" (cold pool, indexer queries vs compressed
 *        indexer keys, sigmoid threshold recall), "Memory Indexer 放哪里"
 *        (3 indexers, OR-mode routing).
 *
 * Conventions
 *   - "d_" pointers are device memory owned by the caller; "h_" pointers
 *     are host memory. bf16 tensors are passed as their uint16_t bit
 *     patterns. All device arrays are dense, row-major, with the shapes
 *     given at each call.
 *   - Streams are cudaStream_t values passed as srh_stream_t (void*); NULL
 *     means the legacy default stream.
 *   - Every call returns SRH_OK (0) or a negative SRH_ERR_* code, and
 *     validates its arguments before it launches anything. Kernel work is
 *     asynchronous: errors found on the device (a selected chunk not yet
 *     stored, an index out of range) are recorded in a sticky device error
 *     word and reported by srh_check_error(). No kernel traps; every
 *     device-side wait gives up after 2 s (SRH_ERR_TIMEOUT).
 *   - Nothing is allocated in the per-step calls: srh_create() allocates
 *     the pinned host pools, the device slot tables and all scratch.
 *   - A context is not thread-safe; calls on one context must be issued
 *     from one host thread. Streams passed to consecutive calls of one
 *     step must be ordered by the caller (the usual case is one stream).
 */
#ifndef SRH_H
#define SRH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SRH_KV_DIM 512        /* latent row width, fp32 ([P1] 关键参数调优: kv_dim = 512) */
#define SRH_WINDOW 128        /* sliding-window rows ([P1] 概述, item 3) */
#define SRH_N_INDEXERS 3      /* memory indexers (layers 10/12/20) ([P2] Memory Indexer 放哪里) */
#define SRH_INDEXER_HEADS 8   /* query heads per indexer */
#define SRH_INDEXER_DIM 128   /* indexer key width, bf16 */
#define SRH_MAX_HEADS 64      /* largest attention head count lsa_attend accepts */

/* Return codes. */
#define SRH_OK 0
#define SRH_ERR_INVALID -1     /* bad argument or shape; GPU_CHUNKS < index_topk without
                                  allow_topk_reduction ([P1] 故障排查, error 2) */
#define SRH_ERR_PINNED_CAP -2  /* pinned pools would exceed pinned_cap_bytes ([P1] 故障排查,
                                  error 3; srh_last_error() gives required_mib / cap_mib) */
#define SRH_ERR_NOT_STORED -3  /* a selected chunk was never stored to the host pool
                                  ([P1] 故障排查, error 4); reported by srh_check_error() */
#define SRH_ERR_CUDA -4        /* a CUDA runtime call failed */
#define SRH_ERR_TIMEOUT -5     /* a bounded device-side wait gave up */
#define SRH_ERR_NOMEM -6       /* host or device allocation failed */
#define SRH_ERR_BOUNDS -7      /* a device kernel met an index outside its buffer (the
                                  access was skipped); reported by srh_check_error() */
#define SRH_ERR_RANGE -8       /* lsa_attend met a query or latent value beyond +-65504, the
                                  finite range of its fp16 tensor-core operands; that call's
                                  outputs are not valid; reported by srh_check_error() */

#define SRH_ENSEMBLE_MAX 0     /* s = max_i s_i: OR-mode ([P1] 配置说明 ENSEMBLE=max; [P2]) */
#define SRH_ENSEMBLE_MEAN 1    /* s = (s_0 + s_1 + s_2) / 3 */

#define SRH_SELECT_TOPK 0      /* top-k by (score desc, index asc) ([P1] 架构概览 step 3) */
#define SRH_SELECT_THRESH 1    /* sigmoid(s) > tau, taken as s > ln(tau/(1-tau)) ([P2] LSA) */

/* srh_config.flags */
#define SRH_FLAG_TEST_FAIL_HOST_ALLOC 1u  /* testing only: the last layer's pinned pool allocation
                                             fails (after every earlier layer's pool and device
                                             state were allocated): srh_create returns
                                             SRH_ERR_NOMEM and frees all of it */

typedef void* srh_stream_t;
typedef struct srh_ctx srh_ctx;

/*
 * Static shape of one decode loop ([P1] 配置说明 and 关键参数调优).
 *   batch            B, independent sequences
 *   n_layers         L, sparse layers
 *   kv_dim           must be SRH_KV_DIM
 *   window           must be SRH_WINDOW
 *   gpu_chunks       G, staging slots per (layer, sequence) (KV_SWAP_GPU_CHUNKS)
 *   index_topk       k, the top-k size (512 on the pages)
 *   src_ratio        compression ratio of the scored chunks (4)
 *   layer_ratio      [n_layers] host array, each a multiple of src_ratio;
 *                    copied by srh_create
 *   context_len      tokens; a layer of ratio r holds cap = ceil(context_len / r)
 *                    chunks ([P1] 关键参数调优, layer_compressed_cap)
 *   pinned_cap_bytes upper bound of the pinned host pools (KV_SWAP_PINNED_MIB
 *                    in bytes); 0 = no bound
 *   allow_topk_reduction  accept gpu_chunks < index_topk
 *                    (KV_SWAP_TEST_ALLOW_TOPK_REDUCTION, tests only)
 *   max_select       S, the row stride of every selection-shaped array
 *                    ([B][S] and [L][B][S]); 0 means max(index_topk, gpu_chunks).
 *                    Must be >= index_topk and <= 4096.
 *   flags            SRH_FLAG_* bits; 0 normally
 */
typedef struct {
    int batch;
    int n_layers;
    int kv_dim;
    int window;
    int gpu_chunks;
    int index_topk;
    int src_ratio;
    const int* layer_ratio;
    long long context_len;
    size_t pinned_cap_bytes;
    int allow_topk_reduction;
    int max_select;
    unsigned flags;
} srh_config;

/* Swap counters, summed over swapped layers and sequences since creation or the
 * last srh_reset_stats() ([P1] 使用示例: gguf_kv_swap_stats hits/misses/h2d_mib/d2h_mib). */
typedef struct {
    unsigned long long hits;                 /* selected chunks found in a staging slot */
    unsigned long long misses;               /* selected chunks gathered from the host pool */
    unsigned long long h2d_bytes;            /* misses * kv_dim * 4 */
    unsigned long long d2h_bytes;            /* bytes written to the host pool by the store path */
    unsigned long long resident_fill_bytes;  /* one-time fills of swap-disabled layers */
    unsigned long long stage_calls;          /* kvswap_stage calls */
    unsigned long long selected;             /* chunks resolved, all layers and sequences */
    int swapped_layers;                      /* layers with cap > gpu_chunks */
    int n_layers;
} srh_stats;

/*
 * Create a context: validates the config (GPU_CHUNKS >= index_topk unless
 * allow_topk_reduction, [P1] 故障排查 error 2; required pinned bytes <=
 * pinned_cap_bytes, error 3), allocates one mapped pinned pool per layer of
 * [batch][cap][kv_dim] fp32 (the host "full compressed cache", [P1] Memory
 * Layout), the device slot tables (all slots free), and the scratch of every
 * kernel. The pools start zeroed and unstored. Uses the current CUDA device.
 * On success *out owns everything; release it with srh_destroy().
 * Errors: SRH_ERR_INVALID, SRH_ERR_PINNED_CAP, SRH_ERR_NOMEM, SRH_ERR_CUDA.
 */
int srh_create(const srh_config* cfg, srh_ctx** out);

/* Free everything the context owns. Waits for the device first. NULL is a no-op. */
void srh_destroy(srh_ctx* ctx);

/* Bytes of pinned host memory a config needs: sum over layers of
 * batch * ceil(context_len / ratio) * kv_dim * 4 ([P1] 关键参数调优, item 2). */
int srh_pinned_required_bytes(const srh_config* cfg, unsigned long long* out);

/*
 * The attention work split of a configuration, computed on the host without
 * a GPU (no counterpart on the pages: a check of lsa_attend's static plan).
 *   cfg       a configuration, validated as srh_create does
 *   sm_count  SMs to plan for (> 0)
 *   layer     -1: the plan of lsa_attend(layer = -1); else that layer's plan
 *   info      [6] out: CTAs, segments, split pairs, the largest CTA's rows in
 *             KiB (window rows 2 KiB, staged rows 1 KiB, at max_select rows
 *             per pair), 1 if each pair is cut into chunks of equal bytes (one
 *             wave) or 0 for stream-K tile ranges, 1 if the plan keeps its
 *             invariants (at most one CTA per SM, every pair covered once in
 *             row order, merge limits) -- srh_create fails otherwise.
 * Returns SRH_OK, SRH_ERR_INVALID or SRH_ERR_NOMEM.
 */
int srh_attend_plan_info(const srh_config* cfg, int sm_count, int layer, long long* info);

/* Host pointer to the pinned pool of (layer, seq): [cap][kv_dim] fp32, owned by
 * the context, valid until srh_destroy(). The caller writes chunks here and then
 * calls srh_mark_stored(). NULL on a bad argument. */
float* srh_pool_host_ptr(srh_ctx* ctx, int layer, int seq);

/* Store flow ([P1] KV_SWAP 实现细节, Store): mark chunks [c0, c0+n) of (layer, seq)
 * as present in the host pool (host_ready = 1). Synchronous. Swap-disabled
 * layers re-copy those chunks into their staging rows on the next kvswap_stage. */
int srh_mark_stored(srh_ctx* ctx, int layer, int seq, long long c0, long long n);

/*
 * Store flow on the device ([P1] KV_SWAP 实现细节, Store: the compressor made a
 * new chunk; D2H it to h_compressed_kv[logical], set host_ready[logical], and a
 * chunk that is in a GPU staging slot stays there).
 *   layer, seq  the (layer, sequence) the chunks belong to
 *   c0, n       chunks [c0, c0+n) of that layer, 0 <= c0, c0 + n <= cap
 *   d_rows      [n][kv_dim] fp32 device rows, read by the call's kernel
 * One kernel copies each row into the pinned host pool (zero-copy writes),
 * sets host_ready, and keeps the staging consistent: a chunk that currently
 * holds a staging slot keeps it and its staged row gets the new content; on a
 * layer that does not swap, staging row c gets it. Nothing is evicted.
 * Asynchronous on `stream`: issue it before the kvswap_stage that may select
 * these chunks, on the same stream. Counts n * kv_dim * 4 bytes in d2h_bytes.
 * Errors: SRH_ERR_INVALID (range, pointers), SRH_ERR_CUDA.
 */
int kvswap_store(srh_ctx* ctx, int layer, int seq, long long c0, int n, const float* d_rows,
                 srh_stream_t stream);

/* Layer facts: chunk capacity and whether the layer swaps (cap > gpu_chunks,
 * [P1] 故障排查, the swap auto-disable note). */
int srh_layer_info(srh_ctx* ctx, int layer, long long* cap, int* swap_enabled);

/* Row stride S of selection-shaped arrays. */
int srh_max_select(srh_ctx* ctx);

/*
 * a1+a2: indexer scoring + ensemble ([P1] 架构概览, scoring box steps 1-3; [P2] LSA,
 * Memory Indexer 放哪里).
 *   d_keys   [batch][n][128] bf16, the frozen compressed indexer keys of one
 *            shared source layer (n <= the ratio-src_ratio capacity)
 *   d_q      [batch][3][8][128] bf16, the memory-indexer query sets
 *   scale    logit scale applied to the per-indexer max over heads
 *   bias3    host [3], per-indexer logit bias b_i
 *   ensemble SRH_ENSEMBLE_MAX or SRH_ENSEMBLE_MEAN
 *   d_scores [batch][n] fp32 output: s(c), where
 *            s_i(c) = scale * max_h <Q[i,h], K[c]> + b_i and s = max_i or mean_i.
 * Also fills a per-sequence score histogram inside the context that fm_select
 * uses when it is called on the same d_scores. After a threshold selection
 * (fm_select with SRH_SELECT_THRESH) the next fm_score instead appends every
 * chunk above that threshold to a candidate list inside the context; the next
 * threshold selection with the same tau on the same d_scores selects from that
 * list and skips its own pass over the scores. Either way the outputs are
 * those of the definitions above; only the work fm_select does changes.
 */
int fm_score(srh_ctx* ctx, const uint16_t* d_keys, int n, const uint16_t* d_q, float scale,
             const float* bias3, int ensemble, float* d_scores, srh_stream_t stream);

/*
 * fm_score with one key set per memory indexer ([P1] 限制与未来工作,
 * "Multi-layer compressed_k": each FlashMemory scorer reads the indexer keys of
 * its own layer, l10/l12/l20, instead of one shared source layer).
 *   d_keys3  [3][batch][n][128] bf16: key set i is scored by indexer i
 * Everything else as fm_score, with s_i(c) = scale * max_h <Q[i,h], K_i[c]> + b_i;
 * the key stream is three times that of fm_score.
 */
int fm_score_multi(srh_ctx* ctx, const uint16_t* d_keys3, int n, const uint16_t* d_q, float scale,
                   const float* bias3, int ensemble, float* d_scores, srh_stream_t stream);

/*
 * fp8 indexer keys ([P1] 限制与未来工作: quantize the indexer keys to fp8 to cut
 * the scoring pass's key stream; the scorer kernel reads them directly).
 *
 * fm_quantize_keys: d_keys [batch][n][128] bf16 -> d_codes [batch][n][128] e4m3
 * codes (uint8) and d_kscale [batch][n] fp32, per chunk
 *     kscale_c = amax_c / 448,  code = e4m3(K / kscale_c)
 * in IEEE fp32 division, rounded to nearest (ties to even), saturated; an
 * all-zero chunk gets kscale 0 and zero codes. Run once for frozen keys.
 *
 * fm_score_fp8: as fm_score on those codes,
 *     s_i(c) = scale * kscale_c * max_h <Q[i,h], e4m3(K8[c])> + b_i,
 * reading 132 bytes per chunk instead of 256. Fills the same histogram for
 * fm_select. Errors as fm_score.
 */
int fm_quantize_keys(srh_ctx* ctx, const uint16_t* d_keys, int n, uint8_t* d_codes, float* d_kscale,
                     srh_stream_t stream);
int fm_score_fp8(srh_ctx* ctx, const uint8_t* d_codes, const float* d_kscale, int n, const uint16_t* d_q,
                 float scale, const float* bias3, int ensemble, float* d_scores, srh_stream_t stream);

/*
 * a3: selection ([P1] 架构概览 step 3: global top-k; [P2] LSA: sigmoid threshold).
 *   d_scores [batch][n] fp32
 *   mode     SRH_SELECT_TOPK: the min(k, n) best chunks;
 *            SRH_SELECT_THRESH: chunks with s > ln(tau/(1-tau)), at most clamp
 *            of them (the best ones) -- clamp must be <= gpu_chunks;
 *   d_sel    [batch][S] int32 output: chunk ids in (score desc, index asc) order;
 *            entries past the count are left unspecified
 *   d_count  [batch] int32 output: how many ids each sequence selected
 * Requires k <= S (TOPK) and clamp <= S.
 */
int fm_select(srh_ctx* ctx, const float* d_scores, int n, int mode, int k, float tau, int clamp,
              int32_t* d_sel, int32_t* d_count, srh_stream_t stream);

/*
 * fm_select without a context and without any device allocation. The pages
 * have no counterpart: this is a library entry point for callers that may not
 * allocate GPU memory themselves -- an engine that has already reserved the
 * whole device for its own pool (a stray cudaMalloc would fail or fragment it),
 * or code on a latency-critical path where cudaMalloc/cudaFree would stall
 * other streams by synchronizing the device. Creating an srh_ctx allocates, so
 * such a caller uses this instead of fm_select.
 *
 * It computes exactly what fm_select computes (the same histogram and
 * selection kernels, the same results). It skips fm_select's candidate pass
 * for n above 16384, so each sequence's selection scans all n scores in one
 * CTA: calls with n far above 16384 are much slower than fm_select's.
 * The caller owns every input and output buffer; the only scratch is the
 * per-sequence first-digit histogram, held in a fixed array compiled into the
 * library: SRH_NOALLOC_MAX_BATCH x 4096 uint32 (1 MiB). Every GPU that loads
 * the library keeps that array until the process exits.
 *
 *   d_scores   [batch][n] fp32 (device)
 *   batch      1 .. SRH_NOALLOC_MAX_BATCH; larger values are rejected with
 *              SRH_ERR_INVALID before any GPU work
 *   n          1 .. SRH_NOALLOC_MAX_N
 *   mode, k, tau, clamp   as for fm_select; k and clamp must be <= max_select
 *   max_select row stride of d_sel, 1 .. 4096
 *   d_sel      [batch][max_select] int32 output, d_count [batch] int32 output
 *   err, err_len  optional (may be NULL/0): receives a NUL-terminated message
 *              when the call fails
 * Returns SRH_OK, SRH_ERR_INVALID or SRH_ERR_CUDA.
 *
 * The first call on each device looks up the device address of the scratch
 * array on the current device; make that first call before any stream capture
 * begins. Every call on a device shares the one array, and the array keeps the
 * last call's histogram (each call clears it first on its stream). Calls whose
 * GPU work overlaps -- on different streams, or from threads that do not order
 * them -- race on the array and may return wrong selections: order them on
 * one stream. The scratch address found by the first call is kept for the
 * life of the process: calls after cudaDeviceReset() on that device are not
 * supported.
 */
#define SRH_NOALLOC_MAX_BATCH 64
#define SRH_NOALLOC_MAX_N (1 << 30)
int fm_select_noalloc(const float* d_scores, int batch, int n, int mode, int k, float tau, int clamp,
                      int max_select, int32_t* d_sel, int32_t* d_count, srh_stream_t stream, char* err,
                      size_t err_len);

/*
 * a4+a5: KV_SWAP staging ([P1] KV_SWAP 实现细节, Swap-in flow).
 *   layer      one sparse layer, or -1 for all layers
 *   d_sel, d_count  the fm_select outputs ([batch][S], [batch])
 *   d_staging  [L][batch][G][kv_dim] fp16 (IEEE binary16 bits), 32-byte
 *              aligned: the GPU staging slots. A staged row is the pool's fp32
 *              row rounded to nearest fp16: lsa_attend rounds every row to fp16
 *              for its tensor-core products, so its results are the same as
 *              from fp32 slots, from half the bytes (a departure from the page's
 *              fp32 slot layout). A pool value beyond +-65504 sets
 *              SRH_ERR_RANGE at the next srh_check_error. This buffer is part
 *              of the cache state: pass the same buffer to every call on a
 *              context (a different one is rejected with SRH_ERR_INVALID).
 *              Swap-disabled layers keep their chunk c in row c.
 *   d_phys     [L][batch][S] int32 output: physical row of each selected chunk of
 *              the layer, window + slot (window + c when the layer does not swap)
 *   d_count_l  [L][batch] int32 output: chunks of the layer's list. A layer of
 *              ratio r uses the list c -> floor(c * src_ratio / r), first
 *              occurrence kept, in selection order.
 *   main       stream of the LRU resolve; side: stream of the miss gathers (may
 *              equal main). On return, work queued later on main sees the
 *              staged rows.
 * The LRU is the sequential list of the Swap-in flow: the selected ids are
 * taken in order; a hit moves its slot to the front, a miss pops the back slot
 * (all slots start free, slot 0 first) and copies h_compressed_kv[c] into it.
 * Overlap: a call may run on another stream while an lsa_attend still reads
 * the rows the previous call staged (the lookahead schedule), provided it
 * writes other d_phys/d_count_l buffers and every swapped layer has at least
 * as many slots in use as the two selections' list lengths together: the
 * previous list's slots are then the most recently used and none is evicted.
 */
int kvswap_stage(srh_ctx* ctx, int layer, const int32_t* d_sel, const int32_t* d_count,
                 uint16_t* d_staging, int32_t* d_phys, int32_t* d_count_l, srh_stream_t main,
                 srh_stream_t side);

/*
 * a6: sparse attention ([P1] 架构概览, per-layer box step 3; Memory Layout).
 *   layer      one sparse layer, or -1 for all layers
 *   d_q        [L][batch][n_heads][kv_dim] bf16 queries (16-byte aligned)
 *   n_heads    16, 32 or 64
 *   d_window   [L][batch][128][kv_dim] fp32 window rows (32-byte aligned)
 *   d_staging, d_phys, d_count_l  as written by kvswap_stage
 *   d_out      [L][batch][n_heads][kv_dim] fp32 output (16-byte aligned):
 *              o_h = sum_j softmax_j(<q_h, e_j> / sqrt(kv_dim)) e_j over the 128
 *              window rows and the layer's staged rows (K = V = the latent row).
 * Precision: the products run on the tensor cores with fp16 operands (11
 * significant bits) and fp32 accumulation; a pair split over several CTAs is
 * combined from fp16 partial outputs (each a softmax-weighted mean of rows).
 * Query and latent values must lie within +-65504 (else SRH_ERR_RANGE at the
 * next srh_check_error; a staged value that is not finite fp16 counts too);
 * values below 2^-14 (about 6.1e-5) in magnitude keep an absolute precision of
 * 2^-25 instead of 11 significant bits.
 * Calls on one context must not overlap in time: they share the context's
 * partial buffers and arrival counters. Asynchronous; returns SRH_OK,
 * SRH_ERR_INVALID or SRH_ERR_CUDA.
 */
int lsa_attend(srh_ctx* ctx, int layer, const uint16_t* d_q, int n_heads, const float* d_window,
               const uint16_t* d_staging, const int32_t* d_phys, const int32_t* d_count_l,
               float* d_out, srh_stream_t stream);

/*
 * Chained launches (no counterpart on the pages: a launch-latency option).
 * With on != 0, the calls that follow on this context may start their kernels
 * before the previous kernel on the stream has finished (programmatic
 * dependent launch): each kernel waits for the previous one before it reads
 * anything an earlier kernel wrote, and reads only the call's own inputs
 * (queries, window rows) before that. Turn it on only around calls issued back
 * to back on one stream -- fm_score, fm_select, kvswap_stage, lsa_attend --
 * whose inputs were written before the first of them was issued; turn it off
 * (the default) before issuing calls after other kernels of your own.
 * Returns SRH_OK or SRH_ERR_INVALID (NULL context).
 */
int srh_set_chained(srh_ctx* ctx, int on);

/*
 * Adaptive staging capacity ([P1] 未来优化方向, item 4: size the staging from
 * the runtime LRU hit rate; the pages give the direction, not a rule).
 * Each swapped (layer, sequence) uses slots [0, g) of its gpu_chunks staging
 * rows; kvswap_stage resolves against those g slots only. Every `epoch` swap
 * steps of that (layer, sequence) the hit rate h = hits / selected of those
 * steps sets g for the steps that follow:
 *   hits*1000 <  lo_permille*selected  -> g = min(g_max, g + delta)
 *   hits*1000 >  hi_permille*selected  -> g = max(g_min, g - delta)
 *   otherwise g stays (so does it when nothing was selected).
 * A resize moves no row: growing adds the new slots, empty, at the
 * least-recently-used end (lowest slot first), so they fill before any held
 * slot is evicted; shrinking drops slots [g_new, g) and forgets their chunks
 * (a later selection of one is a miss). A step whose layer list is longer
 * than g keeps the first g chunks of the list (as with gpu_chunks < index_topk).
 * The decisions are taken on the device by the resolve kernel, so they also
 * run inside a captured CUDA graph.
 */
typedef struct {
    int enabled;        /* 0: every swapped layer uses all gpu_chunks slots (the default) */
    int g_min;          /* >= index_topk (>= 1 with allow_topk_reduction) */
    int g_max;          /* <= gpu_chunks */
    int g_init;         /* slots in use from the next kvswap_stage on; g_min <= g_init <= g_max */
    int epoch;          /* swap steps per decision, >= 1 */
    int lo_permille;    /* grow below this hit rate (per mille), 0..1000 */
    int hi_permille;    /* shrink above this hit rate, lo_permille..1000 */
    int delta;          /* slots added or removed per decision, >= 1 */
} srh_adaptive;

/*
 * Install (policy->enabled != 0) or remove (policy NULL or enabled == 0) the
 * adaptive capacity of every swapped (layer, sequence). Waits for the device.
 * The next kvswap_stage resizes each swapped (layer, sequence) to g_init
 * (to gpu_chunks on removal) and restarts its hit-rate window; the staged
 * rows of the kept slots stay valid. Returns SRH_OK or SRH_ERR_INVALID (bad
 * bounds, recorded in srh_last_error) or SRH_ERR_CUDA.
 */
int srh_set_adaptive(srh_ctx* ctx, const srh_adaptive* policy);

/*
 * Slots in use per (layer, sequence): out is a host array [n_layers][batch];
 * a swapped layer reports the g of its last kvswap_stage (gpu_chunks before
 * the first), a swap-disabled layer its cap (its chunks are staged at their
 * own rows). Waits for the device. Returns SRH_OK, SRH_ERR_INVALID or SRH_ERR_CUDA.
 */
int srh_get_active_slots(srh_ctx* ctx, int* out);

/* Copy the swap counters out (waits for the device). */
int srh_get_stats(srh_ctx* ctx, srh_stats* out);

/* Zero the swap counters (waits for the device). */
int srh_reset_stats(srh_ctx* ctx);

/*
 * Native host loop (no counterpart on the pages: the serving loop around the
 * four calls, in native code so that issuing a step costs a few microseconds
 * of host time). Decode steps fed from host memory and read back into it, with
 * the copies of neighbouring steps overlapping the step in flight. Two sets of
 * device step buffers alternate; each set has its own CUDA graph of one decode
 * step over all layers -- fm_score, then fm_select, kvswap_stage and
 * lsa_attend chained (srh_set_chained) -- captured at creation on the loop's
 * compute stream (nothing runs then). Step i copies its indexer and attention
 * queries from host memory into set i % 2 on a copy-in stream, replays that
 * set's graph on the compute stream and copies the attention output, the
 * selection and the count back on a copy-out stream; events order each set's
 * reuse after its previous step's outputs have left the device. Steps run in
 * issue order, so the LRU state advances as with srh calls on one stream.
 *
 *   d_keys, n, d_scores                      as for fm_score / fm_select
 *   d_staging, d_phys, d_count_l, d_window   as for kvswap_stage / lsa_attend
 *   n_heads                                  16, 32 or 64
 *   scale, bias3[3], ensemble                as for fm_score
 *   mode, k, tau, clamp                      as for fm_select
 *   d_fm_q[2]   [B][3][8][128] bf16, d_q[2] [L][B][n_heads][512] bf16 (inputs)
 *   d_out[2]    [L][B][n_heads][512] fp32, d_sel[2] [B][max_select] int32,
 *   d_count[2]  [B] int32 (outputs); every set's buffers distinct
 *   stream      GPU work already issued on it precedes the loop's first step
 *   out         receives the loop (NULL on failure)
 * The loop keeps the pointers: the buffers must outlive it. The context's
 * chaining flag (srh_set_chained) is as the caller left it when the call
 * returns; inside the graphs the first kernel is never chained and the others
 * always are. Returns SRH_OK, SRH_ERR_INVALID,
 * SRH_ERR_NOMEM or SRH_ERR_CUDA (details in srh_last_error(ctx)).
 */
typedef struct srh_hostloop srh_hostloop;
int srh_hostloop_create(srh_ctx* ctx, const uint16_t* d_keys, int n, float* d_scores, uint16_t* d_staging,
                        int32_t* d_phys, int32_t* d_count_l, const float* d_window, int n_heads, float scale,
                        const float* bias3, int ensemble, int mode, int k, float tau, int clamp,
                        uint16_t* const d_fm_q[2], uint16_t* const d_q[2], float* const d_out[2],
                        int32_t* const d_sel[2], int32_t* const d_count[2], srh_stream_t stream,
                        srh_hostloop** out);

/*
 * Issues step i (i = 0, 1, 2, ...; consecutive): h_fm_q [B][3][8][128] bf16 and
 * h_q [L][B][n_heads][512] bf16 are read, h_out / h_sel [B][max_select] /
 * h_count [B] written -- host memory, page-locked for the copies to be
 * asynchronous. Asynchronous: the outputs are complete once srh_hostloop_wait
 * for step i (or srh_hostloop_sync) returns, and the host buffers must not be
 * reused before then. Returns SRH_OK, SRH_ERR_INVALID or SRH_ERR_CUDA.
 */
int srh_hostloop_step(srh_hostloop* lp, long long i, const uint16_t* h_fm_q, const uint16_t* h_q, float* h_out,
                      int32_t* h_sel, int32_t* h_count);

/* Blocks until step i's outputs are in host memory. Valid for the last two
 * steps issued (an earlier step's outputs are complete already). */
int srh_hostloop_wait(srh_hostloop* lp, long long i);

/* Blocks until every step issued so far has finished. */
int srh_hostloop_sync(srh_hostloop* lp);

/* Waits for the loop's work and frees it (its streams, events and graphs). */
void srh_hostloop_destroy(srh_hostloop* lp);

/* Wait for the device and report the sticky device error word: SRH_OK,
 * SRH_ERR_NOT_STORED, SRH_ERR_BOUNDS, SRH_ERR_TIMEOUT or SRH_ERR_RANGE (first
 * match in that order), or SRH_ERR_CUDA. The word is cleared after it is read. */
int srh_check_error(srh_ctx* ctx);

/*
 * Self-test of the device-side bounded waits (failure detection without a
 * fault; the pages have no counterpart, their errors are host-side guards,
 * [P1] 故障排查). Launches one CTA on `stream` that waits on an mbarrier phase
 * nothing completes, with a limit of `limit_us` microseconds in [1, 2000000]
 * (the kernels' own waits use 2 s); when the limit passes, the wait gives up
 * and records the timeout in the context's sticky error word, exactly as a
 * stuck wait in a step kernel would. The next srh_check_error() then returns
 * SRH_ERR_TIMEOUT and the context stays usable. Asynchronous; returns SRH_OK,
 * SRH_ERR_INVALID (NULL context, limit out of range) or SRH_ERR_CUDA.
 */
int srh_selftest_wait_timeout(srh_ctx* ctx, int limit_us, srh_stream_t stream);

/* Static text for a return code. */
const char* srh_error_string(int code);

/* Detail of the last failing call on the context (or of the last failing
 * srh_create when ctx is NULL), e.g. "required_mib=84 cap_mib=64". */
const char* srh_last_error(srh_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* SRH_H */
