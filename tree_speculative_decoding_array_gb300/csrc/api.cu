// Library-wide entry points: error strings, version, device queries.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace tsv {

static thread_local char g_err[512] = "";

tsv_status fail(tsv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { g_err[0] = '\0'; }

tsv_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TSV_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return TSV_OK;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace tsv

extern "C" const char* tsv_last_error(void) { return tsv::g_err; }

extern "C" int tsv_version(void) { return 102; }

// ---------------------------------------------------------------------------
// tsv_selftest_bounded_wait: one CTA of the library's bounded waits on a
// barrier that nothing completes.  Every tcgen05 kernel waits the same way;
// after the limit the waiting warp raises the CTA's abort flag, the other
// warps see the flag and stop, and the CTA records TSV_DEV_TIMEOUT.
// ---------------------------------------------------------------------------
#include "tc.cuh"

namespace tsv {

__global__ void selftest_wait_kernel(int32_t* status) {
    griddep_begin();
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);  // count 1; nobody arrives
        abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    bool ok = true;
    if (warp == 0) ok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar, 0, &abort_flag));     // times out, raises abort
    else ok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&bar, 0, &abort_flag, 1024));        // leaves on the abort flag
    __syncthreads();
    if (threadIdx.x == 0 && (!ok || abort_flag)) dev_fail(status, TSV_DEV_TIMEOUT, abort_flag, warp);
}

}  // namespace tsv

extern "C" tsv_status tsv_selftest_bounded_wait(int32_t* dev_status, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (!dev_status) return fail(TSV_EINVAL, "selftest_bounded_wait: dev_status is null");
    launch_pdl(selftest_wait_kernel, 1, 64, 0, stream, dev_status);
    return check_launch("selftest_bounded_wait");
}
