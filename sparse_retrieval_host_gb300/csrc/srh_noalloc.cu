// fm_select_noalloc: the selection step for callers that may not allocate GPU
// memory (an engine that has reserved the whole device for its own pool, or a
// latency-critical path where cudaMalloc/cudaFree would synchronize the device
// and stall other streams). It needs no srh_ctx, which allocates on creation.
//
// The one piece of scratch the selection needs -- the per-sequence histogram
// of the first 12-bit digit of the composite key -- lives in a fixed array
// compiled into the library. Every GPU that loads the library keeps that array
// (SRH_NOALLOC_MAX_BATCH x 4096 uint32 = 1 MiB) until the process exits. All
// calls on a device share it, and it keeps the last call's histogram; each call
// zeroes the rows it uses on its own stream before filling them, so calls in
// stream order are independent, while calls whose GPU work overlaps race.
//
// It launches fm_select's histogram and selection kernels, with the histogram
// in the fixed array, so its results are identical to fm_select's on the same
// inputs. It does not run fm_select's candidate pass for n above 16384 (that
// pass needs a candidate buffer): each sequence's selection then scans all n
// scores in one CTA, so calls with n far above 16384 are much slower than
// fm_select's.
//
// The array's device address is looked up once per device ordinal and kept for
// the life of the process; calls after cudaDeviceReset() on that device (which
// unloads the library's device code) are not supported.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "srh_internal.cuh"

static_assert(SRH_NOALLOC_MAX_BATCH >= 1, "no-alloc batch limit");

// The histogram scratch. In host code this name is only a stand-in that the
// runtime maps to the array's copy on the current device; its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t srh_noalloc_hist[SRH_NOALLOC_MAX_BATCH * srh::kHistBins];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint32_t* g_hist_dev[kMaxDevices];   // device address of the scratch, per device ordinal

int report(char* err, size_t err_len, int code, const char* fmt, ...) {
    if (err && err_len > 0) {
        va_list ap;
        va_start(ap, fmt);
        std::vsnprintf(err, err_len, fmt, ap);
        va_end(ap);
    }
    return code;
}

// Once per device, with that device current: look up where the scratch array
// lives on it. Returns nullptr (and fills err) on failure.
uint32_t* scratch_on_current_device(char* err, size_t err_len, int* code) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *code = report(err, err_len, SRH_ERR_CUDA, "fm_select_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *code = report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: device ordinal %d above %d", dev,
                       kMaxDevices - 1);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_hist_dev[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, srh_noalloc_hist);
        if (e != cudaSuccess || !p) {
            *code = report(err, err_len, SRH_ERR_CUDA, "fm_select_noalloc: cudaGetSymbolAddress on device %d: %s",
                           dev, cudaGetErrorString(e));
            return nullptr;
        }
        e = srh::set_select_attrs();
        if (e != cudaSuccess) {
            *code = report(err, err_len, SRH_ERR_CUDA, "fm_select_noalloc: kernel attributes on device %d: %s", dev,
                           cudaGetErrorString(e));
            return nullptr;
        }
        g_hist_dev[dev] = static_cast<uint32_t*>(p);
    }
    return g_hist_dev[dev];
}

}  // namespace

extern "C" int fm_select_noalloc(const float* d_scores, int batch, int n, int mode, int k, float tau, int clamp,
                                 int max_select, int32_t* d_sel, int32_t* d_count, srh_stream_t stream,
                                 char* err, size_t err_len) {
    if (err && err_len > 0) err[0] = '\0';
    if (!d_scores || !d_sel || !d_count) return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: NULL pointer");
    if (batch < 1 || batch > SRH_NOALLOC_MAX_BATCH)
        return report(err, err_len, SRH_ERR_INVALID,
                      "fm_select_noalloc: batch=%d outside [1, %d] (the fixed scratch holds %d sequences)", batch,
                      SRH_NOALLOC_MAX_BATCH, SRH_NOALLOC_MAX_BATCH);
    if (n < 1 || n > SRH_NOALLOC_MAX_N)
        return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: n=%d outside [1, %d]", n, SRH_NOALLOC_MAX_N);
    if (max_select < 1 || max_select > srh::kMaxSelect)
        return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: max_select=%d outside [1, %d]", max_select,
                      srh::kMaxSelect);
    float thresh = 0.f;
    if (mode == SRH_SELECT_TOPK) {
        if (k < 1 || k > max_select)
            return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: k=%d outside [1, max_select=%d]", k,
                          max_select);
    } else if (mode == SRH_SELECT_THRESH) {
        if (!(tau > 0.f && tau < 1.f))
            return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: tau must be in (0, 1)");
        if (clamp < 0 || clamp > max_select)
            return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: clamp=%d outside [0, max_select=%d]",
                          clamp, max_select);
        thresh = (float)std::log((double)tau / (1.0 - (double)tau));
    } else {
        return report(err, err_len, SRH_ERR_INVALID, "fm_select_noalloc: unknown selection mode %d", mode);
    }

    int code = SRH_OK;
    uint32_t* hist = scratch_on_current_device(err, err_len, &code);
    if (!hist) return code;

    cudaStream_t st = (cudaStream_t)stream;
    uint32_t* hist_in = nullptr;
    if (mode == SRH_SELECT_TOPK || clamp > 0) {
        // launch_hist zeroes the batch rows of the scratch on `st`, then fills them.
        const cudaError_t e = srh::launch_hist(d_scores, n, batch, hist, st, true);
        if (e != cudaSuccess)
            return report(err, err_len, SRH_ERR_CUDA, "fm_select_noalloc histogram: %s", cudaGetErrorString(e));
        hist_in = hist;
    }
    const cudaError_t e =
        srh::launch_select(d_scores, n, batch, mode, k, thresh, clamp, max_select, hist_in, d_sel, d_count, st);
    if (e != cudaSuccess)
        return report(err, err_len, SRH_ERR_CUDA, "fm_select_noalloc launch: %s", cudaGetErrorString(e));
    return SRH_OK;
}
